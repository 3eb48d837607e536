// Chunked-prefill segment of a ragged call on the 5th-generation tensor cores
// (tcgen05 with the accumulators in tensor memory).  Same work and result as
// prefill_tc.cuh (the mma.sync form, kept as a selectable alternative):
//
// "flashlet" README, design bullets: one ragged plan()/run() serves chunked
// prefills and decode rows together (qo_indptr lengths [512, 1, 1, ...]) with a
// causal mask over both; row i of an L-row chunk over N keys attends keys
// j <= N - L + i.
//
// One CTA per (request, kv head, 128 consecutive (row, head) pairs, key slice), the
// pairs of a kv head's G query heads packed as m = i * G + h so that each staged K/V
// tile serves the whole group.  The 128 pairs are the M = 128 rows of the products,
// one TMEM lane each.  Per 64-key tile:
//   S[128 x 64]  = Q[128 x d] . K^T   tcgen05.mma, Q and K K-major in 128B-swizzled smem
//   two threads per pair (warps w and w + 4 reach the same TMEM lanes) each load 32
//   of the row's scores (tcgen05.ld), apply the causal bound and the online softmax
//   (the row maximum is the one value they exchange, through shared memory; each keeps
//   its own partial row sum), and write their P back over S as two 16-bit terms
//   (P = P_hi + P_lo);
//   O[128 x d] += P_hi . V + P_lo . V   tcgen05.mma with A from TMEM, V MN-major; O
//   accumulates over the tiles in TMEM.  The row's running maximum moves only when the
//   row maximum exceeds it by more than 2^8 (rare after the first tiles); then the two
//   threads scale their halves of the row of O in TMEM (after P.V of the previous tile)
//   and their sums.  At the end each thread reads its d/2 columns once and normalises.
//
// Warp specialisation.  Issuing a product holds the issuing thread for about as long
// as the tensor pipe takes to run it (measured on GB300: ~23 ns per 128x64x16 product,
// ~37 ns with two CTAs per SM), so warp 8 does nothing but wait for each K/V stage,
// make the generic stores it needs (the chunk's own new rows, zeros past the slice end)
// and issue the products; warp 9 issues the TMA copies (a tile's copies took its
// issuing thread ~770 cycles); warps 0-7 do only the softmax and the output.  They hand
// over through mbarriers:
//   stage full (TMA complete_tx) and stage free (tcgen05.commit after the tile's P.V);
//   S ready (tcgen05.commit, one per S buffer) -> the softmax of tile k;
//   P ready (256 arrivals, two barriers by tile parity): P of tile k (and any scaled
//     row of O) is in TMEM -> P.V of tile k;
//   P.V done (tcgen05.commit, two by parity) -> a rescale of O, the final read of O, and
//     the reuse of the tile's S buffer.
// With three S buffers (d = 64) S runs two tiles ahead of P.V, so the threads find
// each tile's scores ready.  Every wait is bounded; a thread whose wait gives up
// reports it, stops waiting and still takes part in every barrier, so the CTA ends.
#pragma once

#include <climits>

#include "decode_tc.cuh"
#include "tcgen05.cuh"

namespace pgqa {

template <int D>
struct T5Cfg {
    static constexpr int KT = 64;                        // keys per tile
    static constexpr int MP = 128;                       // pairs per CTA (TMEM lanes, MMA M)
    static constexpr int NT = 256;                       // softmax threads (warps 0-7): two per pair
    static constexpr int NTHREADS = NT + 64;             // + the product warp and the copy warp
    static constexpr int DH = D / 2;                     // output columns per thread
    static constexpr int ST = D == 64 ? 5 : 2;           // K/V stages: two CTAs per SM either way
    static constexpr int NSB = D == 64 ? 3 : 2;          // S / P buffers in TMEM
    static constexpr int HALVES = D / 64;
    static constexpr int HALF_BYTES = KT * 128;          // 64 keys x 64 channels of K or V
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K tile, then V tile
    static constexpr int QHALF_BYTES = MP * 128;         // 128 pairs x 64 channels of Q
    static constexpr int Q_BYTES = HALVES * QHALF_BYTES;
    static constexpr int PIPE_OFF = Q_BYTES;
    static constexpr int BAR_OFF = PIPE_OFF + ST * STAGE_BYTES;
    static constexpr int NBAR = 2 * ST + NSB + 2 + 2;    // stage full [ST], stage free [ST], S, P.V done [2], P ready [2]
    static constexpr int SLOT_OFF = BAR_OFF + NBAR * 8;
    static constexpr int PAGE_OFF = (SLOT_OFF + 4 + 15) / 16 * 16;
    static constexpr int XCH_OFF = PAGE_OFF + kSlicePageCap * 4;  // [3][2][MP] floats: row max by tile parity, row sum
    static constexpr int SMEM_BYTES = XCH_OFF + 3 * 2 * MP * 4;
    // the output staging of the epilogue: per softmax warp 32 rows of 32 floats, padded
    // to 36 so that 8 lanes writing 16 bytes each hit different banks; in the stages
    static constexpr int STAGE_ROW = 36;
    static_assert((NT / 32) * 32 * STAGE_ROW * 4 <= ST * STAGE_BYTES, "the staging fits the stages");
    // TMEM: NSB S / P buffers of 64 columns, then D columns for O; 256 columns leave
    // room for two CTAs per SM.
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr int S_COL = 0, O_COL = 64 * NSB;
    static_assert(O_COL + D <= static_cast<int>(TMEM_COLS), "TMEM columns");
    static_assert(Q_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
};

// Offset of 16-byte chunk c (0 .. D/8-1) of row r in a 128B-swizzled tile whose
// 64-channel blocks are half_bytes apart.
__device__ __forceinline__ uint32_t swz_off(int r, int c, int half_bytes) {
    return (c >> 3) * half_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Two CTAs per SM: 20 warps, five on each of the SM's four sub-partitions, whose 16K
// registers then allow 96 a thread (102, rounded down to the allocation unit of 8).
template <int D, bool ROPE, typename T>
__global__ void __launch_bounds__(T5Cfg<D>::NTHREADS, 2)
    prefill_t5_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const PrefillParams p, int G) {
    using C = T5Cfg<D>;
    using M = MmaType<T>;
    constexpr int CH = D / 8;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer = warp == C::NT / 32;        // the product warp
    const bool copier = warp == C::NT / 32 + 1;    // the copy warp
    const int quarter = warp & 3;            // TMEM lanes [32 quarter, +32): this warp's pairs
    const int half = (warp >> 2) & 1;        // which 32 keys of each tile and which d/2 output columns
    const int prow = quarter * 32 + lane;    // the pair within the CTA (TMEM lane)
    uint8_t *qs = smem;
    uint8_t *pipe = smem + C::PIPE_OFF;
    const uint32_t bar0 = smem_addr(smem + C::BAR_OFF);
    const uint32_t bar_free = bar0 + 8 * C::ST, bar_s = bar_free + 8 * C::ST, bar_o = bar_s + 8 * C::NSB,
                   bar_p = bar_o + 16;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::SLOT_OFF);
    int32_t *page_buf = reinterpret_cast<int32_t *>(smem + C::PAGE_OFF);
    float *xch = reinterpret_cast<float *>(smem + C::XCH_OFF);

    if (smem_addr(smem) & 1023u) {  // the swizzled tiles assume this alignment of the window
        if (tid == 0) atomicOr(p.flags, PGQA_FLAG_SMEM_ALIGN);
        pdl_wait();
        return;
    }
    const PrefillItem it = p.items[blockIdx.x];  // written by plan_update's copy only
    const int key_begin = it.key_begin, key_end = it.key_end;
    const bool fused = p.k_new != nullptr;
    const int new_begin = it.n_keys - it.rows;  // the chunk's own keys (a fused call supplies them)
    // this thread's pair (row of every product); the product and copy warps compute one they never use
    const int pm = it.pair0 + prow;
    const int qi = pm / G, qh = pm - (pm / G) * G;
    const bool valid = warp < C::NT / 32 && qi < it.rows;
    int limit = !valid ? -1 : (p.causal ? it.n_keys - it.rows + qi : it.n_keys - 1);
    limit = min(limit, key_end - 1);  // keys of this CTA's slice only
    // key tiles up to the largest admissible key of the CTA's pairs (rows grow with m)
    const int i_last = min(it.rows - 1, (it.pair0 + C::MP - 1) / G);
    const int cta_last = min(p.causal ? it.n_keys - it.rows + i_last : it.n_keys - 1, key_end - 1);
    const int ntiles = cta_last >= key_begin ? (cta_last - key_begin) / C::KT + 1 : 0;

    // Chunk ch of the new K (rotated at its key position when the plan uses RoPE) or V
    // row of key position pos >= new_begin.
    auto new_chunk = [&](bool isv, int pos, int ch) -> uint4 {
        const T *row = static_cast<const T *>(isv ? p.v_new : p.k_new) +
                       (static_cast<size_t>(it.q_row0 + pos - new_begin) * p.num_kv_heads + it.kv_head) * D;
        if (ROPE && !isv) return rope_chunk<T, D>(row, ch, p.rope_cs + static_cast<size_t>(pos) * (D / 2));
        return __ldg(reinterpret_cast<const uint4 *>(row + ch * 8));
    };

    if (issuer && lane == 0) {
        for (int b = 0; b < C::NBAR; ++b) mbar_init(bar0 + 8 * b, b >= C::NBAR - 2 ? C::NT : 1);
        fence_barrier_init();
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    const SlicePages pages = stage_slice_pages(page_buf, p.kv_indices, it.page_base, key_begin, key_end, p.page_size);
    if (warp == 0) t5::alloc(smem_addr(tslot), C::TMEM_COLS);
    t5::fence_before();
    __syncthreads();
    t5::fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    auto t_s = [&](int kt) { return tmem + C::S_COL + 64u * static_cast<uint32_t>(kt % C::NSB); };
    const uint32_t t_o = tmem + C::O_COL;
    const uint64_t policy = l2_evict_first_policy();

    // TMA of tile kt's K and V into its stage (copy warp, lane 0)
    auto issue = [&](int kt) {
        const int s = kt % C::ST;
        const uint32_t kdst = smem_addr(pipe + s * C::STAGE_BYTES);
        const uint32_t vdst = kdst + C::TILE_BYTES;
        const uint32_t bar = bar0 + 8 * s;
        const int t0 = key_begin + kt * C::KT;
        int nvalid = 0;
        for (int r = 0; r < C::KT && t0 + r < key_end; r += p.box_rows) {
            const int64_t page = pages(t0 + r, p.page_size);
            if (page >= 0 && page < p.num_pages) ++nvalid;
        }
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nvalid * p.box_rows * D * 2 * 2));
        for (int r = 0; r < C::KT; r += p.box_rows) {
            const int tt = t0 + r;
            if (tt >= key_end) break;
            const int64_t page = pages(tt, p.page_size);
            if (page < 0 || page >= p.num_pages) {  // skipped (stale rows) and reported
                atomicOr(p.flags, PGQA_FLAG_PAGE_INDEX);
                continue;
            }
            const int row = static_cast<int>(page * p.page_size + tt % p.page_size);
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf) {
                const uint32_t off = hf * C::HALF_BYTES + r * 128;
                tma_load_3d_hint(kdst + off, &tm_k, hf * 64, it.kv_head, row, bar, policy);
                tma_load_3d_hint(vdst + off, &tm_v, hf * 64, it.kv_head, row, bar, policy);
            }
        }
    };

    const int pre = ntiles < C::ST ? ntiles : C::ST;
    if (p.prefetch_pool && copier && lane == 0)
        for (int kt = 0; kt < pre; ++kt) issue(kt);
    pdl_wait();
    pdl_launch_dependents();
    if (!p.prefetch_pool && copier && lane == 0)
        for (int kt = 0; kt < pre; ++kt) issue(kt);

    // ---- Q: the pair rows into the swizzled K-major tile (zeros for no pair).  Four
    // threads share a row, each taking chunks c and c + CH/2 (rotate-half partners) for
    // its c in [0, CH/2) with c = its lane mod 4 (+ 4 at head_dim 128), so that every
    // load instruction reads whole 32-byte sectors of 8 rows; 64 rows per pass, two passes.
    if (warp < C::NT / 32) {
        constexpr int CQ = CH / 8;  // first-half chunks per thread and row
#pragma unroll
        for (int pass = 0; pass < C::MP / 64; ++pass) {
            const int r = pass * 64 + (tid >> 2);  // the pair row within the CTA
            const int rm = it.pair0 + r;
            const int ri = rm / G, rh = rm - (rm / G) * G;
            const bool rvalid = ri < it.rows;
            const T *qrow = static_cast<const T *>(p.q) +
                            (static_cast<size_t>(it.q_row0 + (rvalid ? ri : 0)) * p.num_qo_heads + it.kv_head * G +
                             (rvalid ? rh : 0)) * D;
#pragma unroll
            for (int u = 0; u < CQ; ++u) {
                const int c = (tid & 3) + 4 * u;
                uint4 lo4 = rvalid ? __ldg(reinterpret_cast<const uint4 *>(qrow + c * 8)) : make_uint4(0u, 0u, 0u, 0u);
                uint4 hi4 = rvalid ? __ldg(reinterpret_cast<const uint4 *>(qrow + (c + CH / 2) * 8))
                                   : make_uint4(0u, 0u, 0u, 0u);
                if (ROPE && rvalid) {
                    const float2 *cs = p.rope_cs + static_cast<size_t>(new_begin + ri) * (D / 2);
                    uint32_t lo[4] = {lo4.x, lo4.y, lo4.z, lo4.w}, hi[4] = {hi4.x, hi4.y, hi4.z, hi4.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        rope_rotate2<T>(lo[j], hi[j], __ldg(reinterpret_cast<const float4 *>(cs + 8 * c + 2 * j)));
                    lo4 = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    hi4 = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                }
                *reinterpret_cast<uint4 *>(qs + swz_off(r, c, C::QHALF_BYTES)) = lo4;
                *reinterpret_cast<uint4 *>(qs + swz_off(r, c + CH / 2, C::QHALF_BYTES)) = hi4;
            }
        }
    }
    fence_proxy_async_smem();  // generic stores before the products read the tile
    __syncthreads();

    float m_run = -INFINITY, l_run = 0.f;  // running row max (scaled log2 units); this thread's partial sum

    if (issuer) {
        // ================= the issue warp =================
        constexpr uint32_t id_s = t5::idesc_f16<T>(C::MP, C::KT, false);
        constexpr uint32_t id_o = t5::idesc_f16<T>(C::MP, D, true);
        constexpr uint64_t kmaj = t5::smem_desc_bits(16, 1024);
        constexpr uint64_t vmaj = t5::smem_desc_bits(C::HALF_BYTES, 1024);
        bool live = true;                       // false once one of its waits gave up
        int s_issued = -1, pv_issued = -1;      // the last S and P.V committed
        // a bounded wait by the whole warp; the outcome is warp-uniform
        auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
            const bool got = __all_sync(0xffffffffu, live && mbar_wait_bounded(bar, parity));
            if (!got && live && lane == 0) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
            live = live && got;
            return got;
        };
        // Tile kt's stage: wait for it, make its generic stores (the chunk's own new rows;
        // zeros over V rows past the slice end, where P is 0 but 0 x NaN would not be),
        // then S = Q . K^T into S buffer kt % NSB.
        auto stage_s = [&](int kt) {
            const int s = kt % C::ST;
            if (!wait_all(bar0 + 8 * s, (kt / C::ST) & 1)) return;
            uint8_t *kp = pipe + s * C::STAGE_BYTES;
            uint8_t *vp = kp + C::TILE_BYTES;
            const int t0 = key_begin + kt * C::KT;
            const int nvalid = min(C::KT, key_end - t0);
            if (fused && max(new_begin, t0) < t0 + nvalid) {
                const int first = max(new_begin, t0) - t0;  // first new row of the tile
                const int n = (nvalid - first) * 2 * CH;
                constexpr int U = 8;  // loads in flight per lane
                for (int base = 0; base < n; base += 32 * U) {
                    uint4 v[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int idx = base + u * 32 + lane;
                        if (idx < n) {
                            const int r = first + idx / (2 * CH), rem = idx % (2 * CH);
                            v[u] = new_chunk(rem >= CH, t0 + r, rem % CH);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int idx = base + u * 32 + lane;
                        if (idx < n) {
                            const int r = first + idx / (2 * CH), rem = idx % (2 * CH);
                            *reinterpret_cast<uint4 *>((rem >= CH ? vp : kp) + swz_off(r, rem % CH, C::HALF_BYTES)) =
                                v[u];
                        }
                    }
                }
            }
            for (int idx = lane; idx < (C::KT - nvalid) * CH; idx += 32) {
                const int r = nvalid + idx / CH, ch = idx % CH;
                *reinterpret_cast<uint4 *>(vp + swz_off(r, ch, C::HALF_BYTES)) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                // descriptors as base + offset / 16: the start-address field cannot carry (shared
                // memory is below 2^18 bytes), so each product costs one add per operand
                const uint64_t qd = t5::smem_desc(smem_addr(qs), kmaj), kd = t5::smem_desc(smem_addr(kp), kmaj);
                t5::fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t kofs = (ks >> 2) * C::HALF_BYTES + (ks & 3) * 32;
                    const uint32_t qofs = (ks >> 2) * C::QHALF_BYTES + (ks & 3) * 32;
                    t5::mma_ss(t_s(kt), qd + (qofs >> 4), kd + (kofs >> 4), id_s, ks > 0);
                }
                t5::commit(bar_s + 8 * (kt % C::NSB));
            }
            s_issued = kt;
        };
        if (ntiles > 0) stage_s(0);
        if (C::NSB == 3 && ntiles > 1) stage_s(1);
        for (int kt = 0; kt < ntiles; ++kt) {
            // P of tile kt (and any scaled row of O) is in TMEM
            if (wait_all(bar_p + 8 * (kt & 1), (kt >> 1) & 1)) {
                if (lane == 0) {
                    const uint64_t vd = t5::smem_desc(smem_addr(pipe + (kt % C::ST) * C::STAGE_BYTES + C::TILE_BYTES), vmaj);
                    const uint32_t ts = t_s(kt);
                    t5::fence_after();
#pragma unroll
                    for (int kk = 0; kk < C::KT / 16; ++kk)  // O accumulates over the tiles
                        t5::mma_ts(t_o, ts + 8 * kk, vd + kk * (2048 >> 4), id_o, kt > 0 || kk > 0);
#pragma unroll
                    for (int kk = 0; kk < C::KT / 16; ++kk)
                        t5::mma_ts(t_o, ts + 32 + 8 * kk, vd + kk * (2048 >> 4), id_o, true);
                    t5::commit(bar_o + 8 * (kt & 1));
                    t5::commit(bar_free + 8 * (kt % C::ST));  // the stage is free for the copy warp
                }
                pv_issued = kt;
            }
            // S of tile kt + NSB - 1 goes in the S buffer of tile kt - 1, whose P.V (its last
            // reader) must be done
            if (kt + C::NSB - 1 < ntiles && live &&
                (kt == 0 || wait_all(bar_o + 8 * ((kt - 1) & 1), ((kt - 1) >> 1) & 1)))
                stage_s(kt + C::NSB - 1);
        }
        // drain what is still in flight (bounded; immediate when every wait succeeded): the
        // last commit on each barrier, which is the only phase a wait can still name
        if (lane == 0) {
            for (int k = max(0, pv_issued - 1); k <= pv_issued; ++k)
                mbar_wait_bounded(bar_o + 8 * (k & 1), (k >> 1) & 1);
            for (int k = max(0, pv_issued - C::ST + 1); k <= pv_issued; ++k)
                mbar_wait_bounded(bar_free + 8 * (k % C::ST), (k / C::ST) & 1);
            for (int k = max(0, s_issued - C::NSB + 1); k <= s_issued; ++k)
                mbar_wait_bounded(bar_s + 8 * (k % C::NSB), (k / C::NSB) & 1);
        }
    } else if (copier) {
        // ================= the copy warp =================
        // Tile j goes in stage j % ST once P.V of tile j - ST, the stage's last reader, is done.
        if (lane == 0) {
            int issued = pre;
            for (int j = pre; j < ntiles; ++j) {
                if (!mbar_wait_bounded(bar_free + 8 * (j % C::ST), ((j / C::ST) - 1) & 1)) {
                    atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
                    break;
                }
                issue(j);
                issued = j + 1;
            }
            // drain: the last copy into each stage (bounded; immediate when it was consumed)
            for (int j = max(0, issued - C::ST); j < issued; ++j)
                mbar_wait_bounded(bar0 + 8 * (j % C::ST), (j / C::ST) & 1);
        }
    } else {
        // ================= the softmax warps =================
        // O accumulates over the tiles in TMEM.  The running maximum m_run moves only when a
        // row's maximum exceeds it by more than 2^8 (P then stays below 256, exact enough in
        // two 16-bit terms); O and the row sum are then scaled by 2^(m_old - m_new).
        constexpr float kRescale = 8.f;
        bool live = true;  // false once one of this thread's waits gave up
        auto wait_pv = [&](int kt) {  // P.V of tile kt is done
            const bool got = live && mbar_wait_bounded(bar_o + 8 * (kt & 1), (kt >> 1) & 1);
            if (!got && live) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
            live = got;
            t5::fence_after();
        };
        for (int kt = 0; kt < ntiles; ++kt) {
            // ---- S of tile kt: mask, online softmax, P (two 16-bit terms) back over S
            const bool got = live && mbar_wait_bounded(bar_s + 8 * (kt % C::NSB), (kt / C::NSB) & 1);
            if (!got && live) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
            live = got;
            t5::fence_after();
            const int t0 = key_begin + kt * C::KT;
            const int k0 = t0 + 32 * half;  // this thread's 32 keys
            float sc[32];
            {
                uint32_t r0[32];
                t5::ld32(t_s(kt) + lane_base + 32 * half, r0);
                t5::wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) sc[j] = __uint_as_float(r0[j]);
            }
            if (k0 + 31 > limit) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (k0 + j > limit) sc[j] = -INFINITY;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) mx = fmaxf(mx, sc[j]);
            // the row max over both halves: warps w and w + 4 hold the same pairs.  The slots
            // alternate with the tile parity, so a slot is rewritten only after the partner
            // has passed the next exchange, that is after it read the slot.
            float *xc = xch + (kt & 1) * 2 * C::MP;
            xc[half * C::MP + prow] = mx;
            named_bar_sync_id(1 + quarter, 64);
            mx = fmaxf(mx, xc[(1 - half) * C::MP + prow]) * p.scale_log2;  // the scale is positive
            // both threads of a pair take the same decision
            float alpha = 1.f;
            if (mx > m_run + kRescale) {  // also the first key of the row (m_run = -inf)
                if (m_run != -INFINITY) alpha = ex2_approx(m_run - mx);
                m_run = mx;
            }
            const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;  // a row with no key yet: every P is 0
            {
                // key pairs through packed fp32x2 arithmetic (fewer issue slots, which the
                // product warp on the same sub-partition needs)
                uint32_t ph[16], pl[16];
                const uint64_t scale2 = t5::f2(p.scale_log2, p.scale_log2), negm2 = t5::f2(neg_m, neg_m);
                uint64_t lsum2 = t5::f2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 x = t5::f2_split(t5::f2_fma(t5::f2(sc[2 * j], sc[2 * j + 1]), scale2, negm2));
                    const uint64_t p01 = t5::f2(ex2_approx(x.x), ex2_approx(x.y));
                    lsum2 = t5::f2_add(lsum2, p01);
                    const float2 pv = t5::f2_split(p01);
                    ph[j] = M::pack(pv.x, pv.y);
                    const float2 f = unpack2<T>(ph[j]);
                    const float2 lo = t5::f2_split(t5::f2_sub(p01, t5::f2(f.x, f.y)));
                    pl[j] = M::pack(lo.x, lo.y);
                }
                const float2 ls = t5::f2_split(lsum2);
                l_run = l_run * alpha + (ls.x + ls.y);
                // keys [32 half, +32) are columns [16 half, +16) of P_hi ([0, 32)) and of P_lo ([32, 64))
                t5::st16(t_s(kt) + lane_base + 16 * half, ph);
                t5::st16(t_s(kt) + lane_base + 32 + 16 * half, pl);
            }
            // ---- rows whose maximum moved: O (tiles before kt) scaled once P.V of tile kt - 1 is
            // done; warp-collective, the other lanes scale by 1
            if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                wait_pv(kt - 1);
#pragma unroll
                for (int c0 = 0; c0 < C::DH; c0 += 32) {
                    uint32_t r[32];
                    t5::ld32(t_o + lane_base + C::DH * half + c0, r);
                    t5::wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                    t5::st32(t_o + lane_base + C::DH * half + c0, r);
                }
            }
            t5::wait_st();
            // ---- P of tile kt (and any scaled O) is in TMEM: the product warp may go on
            t5::fence_before();
            t5::arrive(bar_p + 8 * (kt & 1));
        }
        if (ntiles > 0) wait_pv(ntiles - 1);
        // the row sum is the sum of both threads' parts
        float *xl = xch + 2 * 2 * C::MP;
        xl[half * C::MP + prow] = l_run;
        named_bar_sync_id(1 + quarter, 64);
        l_run += xl[(1 - half) * C::MP + prow];

        // ---- normalise this thread's columns of its pair's row, read from TMEM, and store
        // them through a per-warp staging area in shared memory (the stages are free once
        // the last P.V is done), so that each store instruction writes whole 128-byte
        // lines of 4 rows (fp32) or 8 rows (16-bit) rather than one 16-byte piece of each
        // of 32 rows.  Measured on GB300 (512-row chunk, d 64): the per-thread stores took
        // ~3300 cycles of the epilogue.
        const float L = l_run;
        // L == 0 only for a row with no admissible key; NaN (a poisoned row) propagates.
        const float inv = (L == 0.f) ? 0.f : rcp_approx(L);
        const float lse2 = (L == 0.f) ? -INFINITY : m_run + lg2_approx(L);
        const bool split_keys = it.part_base >= 0;
        const size_t slot = split_keys && valid
                                ? static_cast<size_t>(it.part_base + qi * it.num_splits + it.split) * G + qh
                                : 0;
        const size_t row = static_cast<size_t>(it.q_row0 + (valid ? qi : 0)) * p.num_qo_heads + it.kv_head * G + qh;
        const bool f32 = split_keys || p.out_dtype == PGQA_FP32;
        // element offset of this lane's row (column 0) in its destination, -1 for no pair
        const long long own = valid ? static_cast<long long>((split_keys ? slot : row) * D) : -1ll;
        float *stage = reinterpret_cast<float *>(pipe) + warp * 32 * C::STAGE_ROW;  // [32 rows][STAGE_ROW]
#pragma unroll
        for (int c0 = 0; c0 < C::DH; c0 += 32) {
            uint32_t r[32];
            if (ntiles > 0) {  // CTA-uniform
                t5::ld32(t_o + lane_base + C::DH * half + c0, r);
                t5::wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = 0u;
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(stage + lane * C::STAGE_ROW + j) =
                    make_float4(__uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv,
                                __uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv);
            __syncwarp();
            const int col = C::DH * half + c0;
            if (f32) {  // 8 lanes per row: 16 bytes each
                float *base = split_keys ? p.partial_o : static_cast<float *>(p.out);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr = (lane >> 3) + 4 * k, ch = lane & 7;
                    const long long off = __shfl_sync(0xffffffffu, own, rr);
                    const float4 v = *reinterpret_cast<const float4 *>(stage + rr * C::STAGE_ROW + 4 * ch);
                    if (off >= 0) *reinterpret_cast<float4 *>(base + off + col + 4 * ch) = v;
                }
            } else {  // 4 lanes per row: 8 16-bit values each
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int rr = (lane >> 2) + 8 * k, ch = lane & 3;
                    const long long off = __shfl_sync(0xffffffffu, own, rr);
                    const float4 a = *reinterpret_cast<const float4 *>(stage + rr * C::STAGE_ROW + 8 * ch);
                    const float4 b = *reinterpret_cast<const float4 *>(stage + rr * C::STAGE_ROW + 8 * ch + 4);
                    if (off >= 0)
                        *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + off + col + 8 * ch) =
                            make_uint4(M::pack(a.x, a.y), M::pack(a.z, a.w), M::pack(b.x, b.y), M::pack(b.z, b.w));
                }
            }
            __syncwarp();  // the staging rows are read before the next chunk overwrites them
        }
        if (valid && half == 0) {
            if (split_keys)  // its log2-sum-exp, for the merge
                p.partial_lse[slot] = lse2;
            else if (p.lse != nullptr)
                p.lse[row] = lse2 * 0.6931471805599453f;
        }
    }

    // ---- fused append: the split-0 CTA holding pair (i, head 0) stores row i's new K/V
    if (fused && it.split == 0) {
        for (int idx = tid; idx < C::MP * 2 * CH; idx += C::NTHREADS) {
            const int mloc = idx / (2 * CH);
            const int m = it.pair0 + mloc;
            if (m % G != 0) continue;
            const int i = m / G;
            if (i >= it.rows) continue;
            const int rem = idx - mloc * 2 * CH;
            const bool isv = rem >= CH;
            const int ch = rem - (isv ? CH : 0);
            const int pos = new_begin + i;
            const int64_t page = p.kv_indices[it.page_base + pos / p.page_size];
            if (page < 0 || page >= p.num_pages) {
                atomicOr(p.flags, PGQA_FLAG_PAGE_INDEX);
                continue;
            }
            T *dst = static_cast<T *>(isv ? p.v_pool : p.k_pool) +
                     ((page * p.page_size + pos % p.page_size) * p.num_kv_heads + it.kv_head) * D + ch * 8;
            *reinterpret_cast<uint4 *>(dst) = new_chunk(isv, pos, ch);
        }
    }

    // ---- TMEM back once every product has completed (the issue warp's drain) and every
    // thread's reads are done
    t5::fence_before();
    __syncthreads();
    if (warp == 0) {
        t5::fence_after();
        t5::dealloc(tmem, C::TMEM_COLS);
    }

}

template <int D, bool ROPE, typename T>
cudaError_t launch_prefill_t5_r(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const PrefillParams &p,
                                int num_items, bool pdl, cudaStream_t stream) {
    using C = T5Cfg<D>;
    auto kern = prefill_t5_kernel<D, ROPE, T>;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_items);
    cfg.blockDim = dim3(C::NTHREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_k, tm_v, p, group);
}

template <int D, typename T>
cudaError_t launch_prefill_t5(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const PrefillParams &p,
                              int num_items, bool pdl, cudaStream_t stream) {
    return p.rope_cs != nullptr ? launch_prefill_t5_r<D, true, T>(group, tm_k, tm_v, p, num_items, pdl, stream)
                                : launch_prefill_t5_r<D, false, T>(group, tm_k, tm_v, p, num_items, pdl, stream);
}

}  // namespace pgqa
