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
//   each thread loads its pair's row of S from TMEM (tcgen05.ld), applies the causal
//   bound and the online softmax on its own row (no cross-lane reductions), and writes
//   P back over S as two 16-bit terms (P = P_hi + P_lo);
//   O_t[128 x d] = P_hi . V + P_lo . V   tcgen05.mma with A from TMEM, V MN-major
//   each thread folds its row of O_t into its fp32 output registers.
// One thread issues the products and the TMA loads; completion is signalled through
// mbarriers (tcgen05.commit); every wait is bounded.
#pragma once

#include <climits>

#include "decode_tc.cuh"
#include "tcgen05.cuh"

namespace pgqa {

template <int D>
struct T5Cfg {
    static constexpr int KT = 64;                        // keys per tile
    static constexpr int MP = 128;                       // pairs per CTA (TMEM lanes, MMA M)
    static constexpr int ST = D == 64 ? 4 : 2;           // K/V stages: two CTAs per SM either way
    static constexpr int HALVES = D / 64;
    static constexpr int HALF_BYTES = KT * 128;          // 64 keys x 64 channels of K or V
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K tile, then V tile
    static constexpr int QHALF_BYTES = MP * 128;         // 128 pairs x 64 channels of Q
    static constexpr int Q_BYTES = HALVES * QHALF_BYTES;
    static constexpr int PIPE_OFF = Q_BYTES;
    static constexpr int BAR_OFF = PIPE_OFF + ST * STAGE_BYTES;  // ST stage barriers, then S, O
    static constexpr int SLOT_OFF = BAR_OFF + (ST + 2) * 8;
    static constexpr int PAGE_OFF = (SLOT_OFF + 4 + 15) / 16 * 16;
    static constexpr int SMEM_BYTES = PAGE_OFF + kSlicePageCap * 4;
    static constexpr uint32_t TMEM_COLS = 256;           // S / P: columns [0, 64); O_t: [64, 64 + D)
    static constexpr int S_COL = 0, O_COL = 64;
    static_assert(O_COL + D <= static_cast<int>(TMEM_COLS), "TMEM columns");
    static_assert(Q_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
};

// Offset of 16-byte chunk c (0 .. D/8-1) of row r in a 128B-swizzled tile whose
// 64-channel blocks are half_bytes apart.
__device__ __forceinline__ uint32_t swz_off(int r, int c, int half_bytes) {
    return (c >> 3) * half_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

template <int D, bool ROPE, typename T>
__global__ void __launch_bounds__(128, 2)
    prefill_t5_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const PrefillParams p, int G) {
    using C = T5Cfg<D>;
    using M = MmaType<T>;
    constexpr int CH = D / 8;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int tid = threadIdx.x, warp = tid >> 5;
    uint8_t *qs = smem;
    uint8_t *pipe = smem + C::PIPE_OFF;
    const uint32_t bar0 = smem_addr(smem + C::BAR_OFF);
    const uint32_t bar_s = bar0 + 8 * C::ST, bar_o = bar_s + 8;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::SLOT_OFF);
    int32_t *page_buf = reinterpret_cast<int32_t *>(smem + C::PAGE_OFF);

    if (smem_addr(smem) & 1023u) {  // the swizzled tiles assume this alignment of the window
        if (tid == 0) atomicOr(p.flags, PGQA_FLAG_SMEM_ALIGN);
        pdl_wait();
        return;
    }
    const PrefillItem it = p.items[blockIdx.x];  // written by plan_update's copy only
    const int key_begin = it.key_begin, key_end = it.key_end;
    const bool fused = p.k_new != nullptr;
    const int new_begin = it.n_keys - it.rows;  // the chunk's own keys (a fused call supplies them)
    // this thread's pair (row of every product)
    const int pm = it.pair0 + tid;
    const int qi = pm / G, qh = pm - (pm / G) * G;
    const bool valid = qi < it.rows;
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

    if (tid == 0) {
        for (int s = 0; s < C::ST + 2; ++s) mbar_init(bar0 + 8 * s, 1);
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
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t t_s = tmem + C::S_COL, t_o = tmem + C::O_COL;
    const uint64_t policy = l2_evict_first_policy();

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
    if (p.prefetch_pool && tid == 0)
        for (int kt = 0; kt < pre; ++kt) issue(kt);
    pdl_wait();
    pdl_launch_dependents();
    if (!p.prefetch_pool && tid == 0)
        for (int kt = 0; kt < pre; ++kt) issue(kt);

    // ---- Q: this thread's pair row into the swizzled K-major tile (zeros for no pair)
    {
        uint4 v[CH];
        const T *qrow = static_cast<const T *>(p.q) +
                        (static_cast<size_t>(it.q_row0 + (valid ? qi : 0)) * p.num_qo_heads + it.kv_head * G +
                         (valid ? qh : 0)) * D;
#pragma unroll
        for (int c = 0; c < CH; ++c)
            v[c] = valid ? __ldg(reinterpret_cast<const uint4 *>(qrow + c * 8)) : make_uint4(0u, 0u, 0u, 0u);
        if (ROPE && valid) {
            // rotate-half pairs: chunk c of the first half with chunk c + CH/2
            const float2 *cs = p.rope_cs + static_cast<size_t>(new_begin + qi) * (D / 2);
#pragma unroll
            for (int c = 0; c < CH / 2; ++c) {
                uint32_t lo[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
                uint32_t hi[4] = {v[c + CH / 2].x, v[c + CH / 2].y, v[c + CH / 2].z, v[c + CH / 2].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    rope_rotate2<T>(lo[j], hi[j], __ldg(reinterpret_cast<const float4 *>(cs + 8 * c + 2 * j)));
                v[c] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                v[c + CH / 2] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            }
        }
#pragma unroll
        for (int c = 0; c < CH; ++c) *reinterpret_cast<uint4 *>(qs + swz_off(tid, c, C::QHALF_BYTES)) = v[c];
    }
    fence_proxy_async_smem();  // generic stores before the products read the tile
    __syncthreads();

    float o[D];
#pragma unroll
    for (int j = 0; j < D; ++j) o[j] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;  // running max (scaled log2 units) and sum of this row
    constexpr uint32_t id_s = t5::idesc_f16<T>(C::MP, C::KT, false);
    constexpr uint32_t id_o = t5::idesc_f16<T>(C::MP, D, true);
    constexpr uint64_t kmaj = t5::smem_desc_bits(16, 1024);
    constexpr uint64_t vmaj = t5::smem_desc_bits(C::HALF_BYTES, 1024);

    bool ok = true;
    int waited = 0;
    for (int kt = 0; kt < ntiles; ++kt) {
        const int s = kt % C::ST;
        if (!__syncthreads_and(mbar_wait_bounded(bar0 + 8 * s, (kt / C::ST) & 1))) {
            if (tid == 0) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
            ok = false;
            break;
        }
        waited = kt + 1;
        uint8_t *kp = pipe + s * C::STAGE_BYTES;
        uint8_t *vp = kp + C::TILE_BYTES;
        const int t0 = key_begin + kt * C::KT;
        const int nvalid = min(C::KT, key_end - t0);

        // ---- generic stores into the stage: the chunk's own new rows (fused append), and
        // zeros over V rows past the slice end (P is 0 there, but 0 x NaN would not be)
        bool wrote = false;
        if (fused && max(new_begin, t0) < t0 + nvalid) {
            for (int idx = tid; idx < nvalid * 2 * CH; idx += 128) {
                const int r = idx / (2 * CH);
                const int rem = idx - r * 2 * CH;
                const bool isv = rem >= CH;
                const int ch = rem - (isv ? CH : 0);
                const int pos = t0 + r;
                if (pos < new_begin) continue;
                *reinterpret_cast<uint4 *>((isv ? vp : kp) + swz_off(r, ch, C::HALF_BYTES)) = new_chunk(isv, pos, ch);
            }
            wrote = true;
        }
        if (nvalid < C::KT) {
            for (int idx = tid; idx < (C::KT - nvalid) * CH; idx += 128) {
                const int r = nvalid + idx / CH, ch = idx - (idx / CH) * CH;
                *reinterpret_cast<uint4 *>(vp + swz_off(r, ch, C::HALF_BYTES)) = make_uint4(0u, 0u, 0u, 0u);
            }
            wrote = true;
        }
        if (wrote) {  // CTA-uniform
            fence_proxy_async_smem();
            __syncthreads();
        }

        // ---- S = Q . K^T into TMEM
        if (tid == 0) {
            t5::fence_after();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t kofs = (ks >> 2) * C::HALF_BYTES + (ks & 3) * 32;
                const uint32_t qofs = (ks >> 2) * C::QHALF_BYTES + (ks & 3) * 32;
                t5::mma_ss(t_s, t5::smem_desc(smem_addr(qs) + qofs, kmaj), t5::smem_desc(smem_addr(kp) + kofs, kmaj),
                           id_s, ks > 0);
            }
            t5::commit(bar_s);
        }
        if (!__syncthreads_and(mbar_wait_bounded(bar_s, kt & 1))) {
            if (tid == 0) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
            ok = false;
            break;
        }
        t5::fence_after();

        // ---- this row's scores: mask, online softmax, P (two 16-bit terms) back into TMEM
        float sc[C::KT];
        {
            uint32_t r0[32], r1[32];
            t5::ld32(t_s + lane_base, r0);
            t5::ld32(t_s + lane_base + 32, r1);
            t5::wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                sc[j] = __uint_as_float(r0[j]);
                sc[32 + j] = __uint_as_float(r1[j]);
            }
        }
        if (t0 + C::KT - 1 > limit) {
#pragma unroll
            for (int j = 0; j < C::KT; ++j)
                if (t0 + j > limit) sc[j] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < C::KT; ++j) mx = fmaxf(mx, sc[j]);
        const float mn = fmaxf(m_run, mx * p.scale_log2);  // the scale is positive
        const float alpha = (mn == m_run) ? 1.f : ex2_approx(m_run - mn);
        m_run = mn;
        const float neg_m = (mn == -INFINITY) ? 0.f : -mn;  // a row with no key yet: every P is 0
        {
            uint32_t ph[32], pl[32];
            float lsum = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float p0 = ex2_approx(fmaf(sc[2 * j], p.scale_log2, neg_m));
                const float p1 = ex2_approx(fmaf(sc[2 * j + 1], p.scale_log2, neg_m));
                lsum += p0 + p1;
                ph[j] = M::pack(p0, p1);
                const float2 f = unpack2<T>(ph[j]);
                pl[j] = M::pack(p0 - f.x, p1 - f.y);
            }
            l_run = l_run * alpha + lsum;
            t5::st32(t_s + lane_base, ph);       // P_hi: columns [0, 32)
            t5::st32(t_s + lane_base + 32, pl);  // P_lo: columns [32, 64)
            t5::wait_st();
        }
        t5::fence_before();
        __syncthreads();

        // ---- O_t = P_hi . V + P_lo . V into TMEM
        if (tid == 0) {
            t5::fence_after();
#pragma unroll
            for (int kk = 0; kk < C::KT / 16; ++kk)
                t5::mma_ts(t_o, t_s + 8 * kk, t5::smem_desc(smem_addr(vp) + kk * 2048, vmaj), id_o, kk > 0);
#pragma unroll
            for (int kk = 0; kk < C::KT / 16; ++kk)
                t5::mma_ts(t_o, t_s + 32 + 8 * kk, t5::smem_desc(smem_addr(vp) + kk * 2048, vmaj), id_o, true);
            t5::commit(bar_o);
        }
        if (!__syncthreads_and(mbar_wait_bounded(bar_o, kt & 1))) {
            if (tid == 0) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
            ok = false;
            break;
        }
        t5::fence_after();
        // both products have read the stage: it can be refilled while this row folds O_t in
        if (tid == 0 && kt + C::ST < ntiles) issue(kt + C::ST);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
            t5::ld32(t_o + lane_base + c0, r);
            t5::wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[c0 + j] = fmaf(o[c0 + j], alpha, __uint_as_float(r[j]));
        }
    }
    if (!ok && tid == 0) {
        const int issued = ntiles < waited + C::ST ? ntiles : waited + C::ST;
        for (int kt = waited; kt < issued; ++kt) mbar_wait_bounded(bar0 + 8 * (kt % C::ST), (kt / C::ST) & 1);
    }

    // ---- fused append: the split-0 CTA holding pair (i, head 0) stores row i's new K/V
    if (fused && it.split == 0) {
        for (int idx = tid; idx < C::MP * 2 * CH; idx += 128) {
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

    // ---- TMEM back before the stores (every product has completed: the last wait above)
    t5::fence_before();
    __syncthreads();
    if (warp == 0) {
        t5::fence_after();
        t5::dealloc(tmem, C::TMEM_COLS);
    }

    // ---- normalise and store this thread's row
    if (!valid) return;
    const float L = l_run;
    // L == 0 only for a row with no admissible key; NaN (a poisoned row) propagates.
    const float inv = (L == 0.f) ? 0.f : rcp_approx(L);
    const float lse2 = (L == 0.f) ? -INFINITY : m_run + lg2_approx(L);
    if (it.part_base >= 0) {  // split keys: normalised partial + its log2-sum-exp
        const size_t slot = static_cast<size_t>(it.part_base + qi * it.num_splits + it.split) * G + qh;
        float4 *dst = reinterpret_cast<float4 *>(p.partial_o + slot * D);
#pragma unroll
        for (int j = 0; j < D; j += 4) dst[j / 4] = make_float4(o[j] * inv, o[j + 1] * inv, o[j + 2] * inv, o[j + 3] * inv);
        p.partial_lse[slot] = lse2;
        return;
    }
    const size_t row = static_cast<size_t>(it.q_row0 + qi) * p.num_qo_heads + it.kv_head * G + qh;
    if (p.out_dtype == PGQA_FP32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + row * D);
#pragma unroll
        for (int j = 0; j < D; j += 4) dst[j / 4] = make_float4(o[j] * inv, o[j + 1] * inv, o[j + 2] * inv, o[j + 3] * inv);
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + row * D);
#pragma unroll
        for (int j = 0; j < D; j += 8)
            dst[j / 8] = make_uint4(M::pack(o[j] * inv, o[j + 1] * inv), M::pack(o[j + 2] * inv, o[j + 3] * inv),
                                    M::pack(o[j + 4] * inv, o[j + 5] * inv), M::pack(o[j + 6] * inv, o[j + 7] * inv));
    }
    if (p.lse != nullptr) p.lse[row] = lse2 * 0.6931471805599453f;
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
    cfg.blockDim = dim3(128);
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
