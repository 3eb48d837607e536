// Split-KV paged GQA decode, tensor-core partial kernel (mma.sync m16n8k16).
//
// Same work decomposition as the CUDA-core kernel: one CTA per (query row, kv
// head, key slice), serving the G <= 16 query heads that share the kv head, so
// every K/V row of the slice is read from HBM once for the whole group
// ("A library kernel for decode", section "What changed", for the split-KV
// scheme; the "flashlet" README's NHD pool layout for the addressing).
//
// The group is a dense tile in "swap-AB" form: tokens are the M dimension (16
// per MMA), the G heads padded to 8 (one n tile) or 16 (two n tiles sharing
// every K and V A-fragment) are N, head_dim is K.
//   S^T[16 tok x 8 heads]  = K[16 tok x d]   . Q^T[d x 8 heads]     (fp32 accumulate)
//   O^T[16 d   x 8 heads] += V^T[16 d x tok] . P^T[tok x 8 heads]
// K comes from shared memory through ldmatrix, V through ldmatrix.trans; Q^T
// fragments are loaded once per CTA.  The probabilities leave the score
// accumulator as (row = token, col = head) pairs; movmatrix.trans turns them into
// the (row = token, col = head) B fragment of the second product.  P is carried
// as two 16-bit terms (P = P_hi + P_lo, each rounded to the input type), so the
// PV product keeps ~16 significant bits instead of 8 for bf16.
//
// Data movement: per-warp kDecodeStages-deep rings of shared-memory stages,
// filled by 3-D TMA boxes with 128-byte swizzle ([rows, 1 kv head, 64 channels];
// two boxes per row group when head_dim is 128), resolved through the page table
// by lane 0 and completed on per-stage mbarriers.  The swizzle makes every
// ldmatrix phase touch eight different 16-byte bank groups.
#pragma once

#include <math.h>

#include <atomic>

#include "common.cuh"

namespace pgqa {

template <typename T>
struct MmaType;
template <>
struct MmaType<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};
template <>
struct MmaType<__half> {
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// 16-bit value of the packed pair -> fp32 (bf16: upper bits of an fp32).
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t v) { return widen2<T>(v); }

template <int D, int STAGES, int WARPS = kDecodeWarps>
struct TcCfg {
    static constexpr int TW = decode_warp_tile(D);      // tokens per warp tile (32 for d64, 16 for d128)
    static constexpr int MT = TW / 16;                   // token m-tiles per warp tile
    static constexpr int HALVES = D / 64;                // 128-byte (64-channel) column blocks per row
    static constexpr int NW = WARPS;
    static constexpr int ST = STAGES;
    static constexpr int HALF_BYTES = TW * 128;          // one 64-channel block of a tile
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K tile, then V tile
    static constexpr int PIPE_BYTES = NW * ST * STAGE_BYTES;
    static constexpr int BAR_BYTES = NW * ST * 8;
    static constexpr int DT = D / 16;                    // d m-tiles of the PV product
    static constexpr int KS = D / 16;                    // k-steps of the QK product
    static constexpr int OS = D + 4;                     // padded row stride (floats) of a warp's O
    static constexpr int ROPE_BYTES = D * 4;             // one rotary table row: D/2 (cos, sin)
    static constexpr int SMEM_BYTES = PIPE_BYTES + BAR_BYTES + kSlicePageCap * 4 + ROPE_BYTES;
    static_assert(HALF_BYTES % 1024 == 0, "128B-swizzled blocks start on 1024-byte boundaries");
};

// Byte offset of 16-byte chunk `c` (0..D/8-1) of tile row `r` inside a stage's
// K or V tile, as the 128B-swizzled TMA boxes lay it out.
template <int D>
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
    return (c >> 3) * (decode_warp_tile(D) * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

template <int D, int STAGES, int NH, bool ROPE, typename T, int NW = kDecodeWarps>
__global__ void __launch_bounds__(NW * 32, (STAGES == 2 && NH == 1 && NW == kDecodeWarps) ? 3 : 2)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const DecodeParams p, int G) {
    // NH tiles of 8 query heads: G <= 8 * NH (NH = 2 serves groups of 9..16 heads).
    // ROPE: q and the new K rows turn by the plan's rotary table (p.rope_cs).
    // NW warps with STAGES stages each: kDecodeWarps x 2 or 3 stages streams slices of
    // any length; kDecodeWideWarps x 1 stage gives every warp of a short slice its own
    // single tile, so the whole slice is in flight at once and the longest chain of
    // dependent tile steps in the CTA is one tile long.
    using C = TcCfg<D, STAGES, NW>;
    constexpr int HP = 8 * NH;  // heads padded to whole n tiles
    using M = MmaType<T>;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    extern __shared__ __align__(1024) uint8_t smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g8 = lane >> 2;  // fragment row group
    const int c4 = lane & 3;   // fragment column pair

    uint8_t *pipe = smem;
    const uint32_t bar0 = smem_addr(smem + C::PIPE_BYTES) + warp * C::ST * 8;
    int32_t *page_buf = reinterpret_cast<int32_t *>(smem + C::PIPE_BYTES + C::BAR_BYTES);
    float2 *rope_row = reinterpret_cast<float2 *>(smem + C::PIPE_BYTES + C::BAR_BYTES + kSlicePageCap * 4);

    if (smem_addr(smem) & 1023u) {  // the stage layout assumes this alignment of the window
        if (threadIdx.x == 0) atomicOr(p.flags, PGQA_FLAG_SMEM_ALIGN);
        pdl_wait();
        return;
    }
    // The work list and kv_indices are final once plan_update is enqueued (its
    // copy sits between any earlier writer and this kernel), so they are read
    // before the grid-dependency wait; q and the new rows only after it.
    const WorkItem it = load_work_item(p.items + blockIdx.x);
    // The query row's rotary table row goes to shared memory.  The table is fixed since
    // plan creation, so it is read before the dependency wait, in flight together with
    // the page-table staging; the CTA barrier below publishes it.
    float4 rope_part = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ROPE && threadIdx.x < D / 4)
        rope_part = __ldg(reinterpret_cast<const float4 *>(p.rope_cs + static_cast<size_t>(it.q_pos) * (D / 2)) +
                          threadIdx.x);
    const int ntiles = (it.tok_end - it.tok_begin + C::TW - 1) / C::TW;
    const int my_tiles = ntiles > warp ? (ntiles - warp + C::NW - 1) / C::NW : 0;
    const bool fused = p.k_new != nullptr;

    if (lane == 0) {
        for (int s = 0; s < C::ST; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_barrier_init();
        if (warp == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
    }
    const SlicePages pages =
        stage_slice_pages(page_buf, p.kv_indices, it.page_base, it.tok_begin, it.tok_end, p.page_size);
    if (ROPE && threadIdx.x < D / 4) reinterpret_cast<float4 *>(rope_row)[threadIdx.x] = rope_part;
    __syncthreads();
    const uint64_t policy = l2_evict_first_policy();

    auto issue = [&](int k) {
        const int tile = warp + k * C::NW;
        const int t0 = it.tok_begin + tile * C::TW;
        const int s = k % C::ST;
        const uint32_t kdst = smem_addr(pipe + (warp * C::ST + s) * C::STAGE_BYTES);
        const uint32_t vdst = kdst + C::TILE_BYTES;
        const uint32_t bar = bar0 + 8 * s;
        constexpr int MAXC = C::TW / 16;
        int rows[MAXC];
        int nvalid = 0;
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
            rows[c] = -1;
            const int tt = t0 + c * p.box_rows;
            if (c * p.box_rows < C::TW && tt < it.tok_end) {
                const int64_t page = pages(tt, p.page_size);
                if (page < 0 || page >= p.num_pages) {
                    atomicOr(p.flags, PGQA_FLAG_PAGE_INDEX);
                } else {
                    rows[c] = static_cast<int>(page * p.page_size + tt % p.page_size);
                    ++nvalid;
                }
            }
        }
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nvalid * p.box_rows * D * 2 * 2));
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
            if (rows[c] >= 0) {
#pragma unroll
                for (int hf = 0; hf < C::HALVES; ++hf) {
                    const uint32_t off = hf * C::HALF_BYTES + c * p.box_rows * 128;
                    tma_load_3d_hint(kdst + off, &tm_k, hf * 64, it.kv_head, rows[c], bar, policy);
                    tma_load_3d_hint(vdst + off, &tm_v, hf * 64, it.kv_head, rows[c], bar, policy);
                }
            }
        }
    };

    // Lane 0: the boxes of warp tile k requested into L2 only (no shared memory, no
    // barrier), a hint that is safe before the dependency wait whatever the grid before
    // writes: its stores land in L2 as well, and the copies after the wait read them there.
    auto prefetch_l2 = [&](int k) {
        const int tile = warp + k * C::NW;
        const int t0 = it.tok_begin + tile * C::TW;
        constexpr int MAXC = C::TW / 16;
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
            const int tt = t0 + c * p.box_rows;
            if (c * p.box_rows < C::TW && tt < it.tok_end) {
                const int64_t page = pages(tt, p.page_size);
                if (page >= 0 && page < p.num_pages) {
                    const int row = static_cast<int>(page * p.page_size + tt % p.page_size);
#pragma unroll
                    for (int hf = 0; hf < C::HALVES; ++hf) {
                        tma_prefetch_3d(&tm_k, hf * 64, it.kv_head, row);
                        tma_prefetch_3d(&tm_v, hf * 64, it.kv_head, row);
                    }
                }
            }
        }
    };

    // Test hook (stall_wait_us != 0): warp 0 never issues its first tile, so nothing
    // ever arrives on that stage's barrier and its first wait can only give up -- the
    // path by which a CTA reports a stuck pipeline instead of hanging.  Nothing is in
    // flight into that stage, and the other stages' copies are drained as usual.
    const bool stall = p.stall_wait_us != 0 && warp == 0;
    // The group's q rows are requested into L2 before the dependency wait.  It is only a
    // hint: should the grid before this one write q, its stores land in L2 as well, and
    // the loads after the wait read them there.  (Timed on GB300: 32 mixed rows 13.97 ->
    // 13.73 us per call, 1 x 32k 10.89 -> 10.79; the 128 x 301 step unchanged.)
    if (threadIdx.x == 0) {
        const T *qg = static_cast<const T *>(p.q) + (static_cast<size_t>(it.q_row) * p.num_qo_heads + it.kv_head * G) * D;
        prefetch_l2_bulk(qg, static_cast<uint32_t>(G * D * sizeof(T)));
    }
    // K/V loads start before the grid-dependency wait when the caller has stated
    // that nothing still in flight writes the pool rows this call reads.
    const int pre = my_tiles < C::ST ? my_tiles : C::ST;
    if (p.defer_wait) {
        // Our predecessor is the prefill grid of the same call, which writes nothing
        // we read and started only after everything older completed.
        if (lane == 0)
            for (int k = stall ? 1 : 0; k < pre; ++k) issue(k);
    } else {
        // With the pool declared stable the first stages' copies start now; otherwise the
        // same boxes are requested into L2, so that the copies after the wait find them
        // there (timed on GB300, per plain run() call: 128 x 301 6.23 -> 5.43 us, 4 x 32k
        // 26.2 -> 24.0, 1 x 32k 10.8 -> 10.4, 32 mixed rows 13.7 -> 13.3; the whole slice
        // instead of the first stages helped less).
        if (p.prefetch_pool && lane == 0)
            for (int k = stall ? 1 : 0; k < pre; ++k) issue(k);
        if (!p.prefetch_pool && lane == 0)
            for (int k = 0; k < pre; ++k) prefetch_l2(k);
        pdl_wait();
        // Our predecessors are complete from here on, so a grid launched early after
        // this trigger never overlaps a kernel older than this one.
        pdl_launch_dependents();
        if (!p.prefetch_pool && lane == 0)
            for (int k = stall ? 1 : 0; k < pre; ++k) issue(k);
    }

    // Q^T fragments (B operand): b0 = q[head g8][16ks + 2c4, +1], b1 = same + 8.
    // Heads >= G are zero columns.
    uint32_t qf[C::KS][NH][2];
#pragma unroll
    for (int nh = 0; nh < NH; ++nh) {
        const int hq = g8 + 8 * nh;
        const bool real = hq < G;
        const T *qp = static_cast<const T *>(p.q) +
                      (static_cast<size_t>(it.q_row) * p.num_qo_heads + it.kv_head * G + (real ? hq : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
            const uint32_t *w = reinterpret_cast<const uint32_t *>(qp + ks * 16 + 2 * c4);
            qf[ks][nh][0] = real ? __ldg(w) : 0u;
            qf[ks][nh][1] = real ? __ldg(w + 4) : 0u;
        }
    }

    // Fused append.  A decode item of this kernel holds at most one of the call's new
    // rows -- its row's own key, the last of the request (requests with several query
    // rows run as prefill tiles) -- so the warp whose tile holds it fetches it now into
    // registers (lanes [0, CH) carry K chunks, lanes [CH, 2CH) V chunks), patches it
    // into that tile and stores it into the pool; nothing else of the append sits in
    // the tile loop.
    int pf_pos = -1;
    uint4 pf = make_uint4(0u, 0u, 0u, 0u);
    const bool row_lane = lane < 2 * CH;
    const int rch = lane % CH;
    const bool rv = lane >= CH;
    auto new_row = [&](int pos) -> const T * {
        return static_cast<const T *>(rv ? p.v_new : p.k_new) +
               (static_cast<size_t>(pos + it.new_row_base) * p.num_kv_heads + it.kv_head) * D;
    };
    auto new_row_chunk = [&](int pos) -> uint4 {
        return __ldg(reinterpret_cast<const uint4 *>(new_row(pos) + rch * 8));
    };
    // With RoPE the prefetched chunk stays raw until first used, so the owning warp does
    // not wait on it here.  Rotating it is warp-collective: the partner half of a K
    // chunk comes from lane ^ CH/2 and the table entries from shared memory (the new
    // row is the query row's own key, so its position is the query row's).
    bool pf_rot = !ROPE;
    auto rotate_pf = [&]() {
        if (pf_rot) return;
        pf_rot = true;
        uint4 y;
        y.x = __shfl_xor_sync(0xffffffffu, pf.x, CH / 2);
        y.y = __shfl_xor_sync(0xffffffffu, pf.y, CH / 2);
        y.z = __shfl_xor_sync(0xffffffffu, pf.z, CH / 2);
        y.w = __shfl_xor_sync(0xffffffffu, pf.w, CH / 2);
        if (rv) return;  // V chunks (and idle lanes) keep theirs
        const bool second = rch >= CH / 2;
        const int first = second ? rch - CH / 2 : rch;
        uint32_t lo[4] = {pf.x, pf.y, pf.z, pf.w}, hi[4] = {y.x, y.y, y.z, y.w};
        if (second) {
            lo[0] = y.x; lo[1] = y.y; lo[2] = y.z; lo[3] = y.w;
            hi[0] = pf.x; hi[1] = pf.y; hi[2] = pf.z; hi[3] = pf.w;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) rope_rotate2<T>(lo[j], hi[j], lds128_pinned(rope_row + first * 8 + 2 * j));
        pf = second ? make_uint4(hi[0], hi[1], hi[2], hi[3]) : make_uint4(lo[0], lo[1], lo[2], lo[3]);
    };
    if (fused) {
        const int nb = max(it.new_begin, it.tok_begin);
        if (nb < it.tok_end && ((nb - it.tok_begin) / C::TW) % C::NW == warp) {
            pf_pos = nb;
            if (row_lane) pf = new_row_chunk(nb);
            // The plan only builds items whose new row is the query row's own key.
            if (ROPE && nb != it.q_pos && lane == 0) atomicOr(p.flags, PGQA_FLAG_ROPE_POSITION);
        }
    }

    if (ROPE) {
        // Rotary embedding of q at its row's position: channels 16 ks + 2 c4 (+1, +8, +9)
        // of the first half sit in k-step ks, their partners (+ D/2) in k-step ks + KS/2
        // of the same thread.
#pragma unroll
        for (int ks = 0; ks < C::KS / 2; ++ks) {
            const float4 c0 = lds128_pinned(rope_row + ks * 16 + 2 * c4);
            const float4 c1 = lds128_pinned(rope_row + ks * 16 + 2 * c4 + 8);
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) {
                rope_rotate2<T>(qf[ks][nh][0], qf[ks + C::KS / 2][nh][0], c0);
                rope_rotate2<T>(qf[ks][nh][1], qf[ks + C::KS / 2][nh][1], c1);
            }
        }
    }

    // Running state for this thread's head columns 8 nh + 2 c4, + 1.
    float m_run[NH][2], l_run[NH][2];
    float o[C::DT][NH][4];
#pragma unroll
    for (int nh = 0; nh < NH; ++nh) {
        m_run[nh][0] = m_run[nh][1] = -INFINITY;
        l_run[nh][0] = l_run[nh][1] = 0.f;
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt) o[dt][nh][0] = o[dt][nh][1] = o[dt][nh][2] = o[dt][nh][3] = 0.f;
    }

    // ldmatrix lane roles: which 8x8 matrix this lane addresses and which row of it.
    const int lm = lane >> 3, lr = lane & 7;

    int waited = 0;
    bool ok = true;
    for (int k = 0; k < my_tiles; ++k) {
        const int s = k % C::ST;
        // every lane observes the phase (TMA data visibility); the outcome is made warp-uniform
        const bool landed = (stall && k == 0)
                                ? mbar_wait_limit(bar0 + 8 * s, 0, uint64_t(p.stall_wait_us) * 1000u)
                                : mbar_wait_bounded(bar0 + 8 * s, (k / C::ST) & 1);
        if (!__all_sync(0xffffffffu, landed)) {
            if (lane == 0) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
            ok = false;
            break;
        }
        waited = k + 1;
        const int tile = warp + k * C::NW;
        const int tb = it.tok_begin + tile * C::TW;
        const int nvalid = min(C::TW, it.tok_end - tb);
        uint8_t *kp = pipe + (warp * C::ST + s) * C::STAGE_BYTES;
        const uint32_t kb = smem_addr(kp);
        const uint32_t vb = kb + C::TILE_BYTES;

        // ---- fused append: the call's new row replaces what the pool held at its position
        bool patched = false;
        if (pf_pos >= tb && pf_pos < tb + nvalid) {  // warp-uniform
            rotate_pf();
            if (row_lane) *reinterpret_cast<uint4 *>(kp + (rv ? C::TILE_BYTES : 0) + tile_off<D>(pf_pos - tb, rch)) = pf;
            patched = true;
            __syncwarp();
        }

        // ---- S^T = K . Q^T for the tile's m-tiles (rows = tokens)
        float sc[C::MT][NH][4];
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) sc[mt][nh][0] = sc[mt][nh][1] = sc[mt][nh][2] = sc[mt][nh][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                // matrices: 0 = (tok 0-7, chunk 2ks), 1 = (tok 8-15, 2ks), 2 = (tok 0-7, 2ks+1), 3 = (tok 8-15, 2ks+1)
                const int r = mt * 16 + (lm & 1) * 8 + lr;
                const int c = 2 * ks + (lm >> 1);
                uint32_t a[4];
                ldsm_x4(a, kb + tile_off<D>(r, c));
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) M::mma(sc[mt][nh], a, qf[ks][nh][0], qf[ks][nh][1]);
            }
        }
        // ---- mask, scale to log2 units, tile max per head column
        float mx[NH][2];
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
            mx[nh][0] = mx[nh][1] = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int tok = mt * 16 + g8 + (j >> 1) * 8;
                    const float x = tok < nvalid ? sc[mt][nh][j] * p.scale_log2 : -INFINITY;
                    sc[mt][nh][j] = x;
                    mx[nh][j & 1] = fmaxf(mx[nh][j & 1], x);
                }
            }
        }
        bool rescale = false;
        float alpha[NH][2];
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float m = mx[nh][h];
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                const float mn = fmaxf(m_run[nh][h], m);
                alpha[nh][h] = (mn == m_run[nh][h]) ? 1.f : ex2_approx(m_run[nh][h] - mn);
                rescale = rescale || alpha[nh][h] != 1.f;
                m_run[nh][h] = mn;
                l_run[nh][h] *= alpha[nh][h];
            }
        }
        if (rescale) {
#pragma unroll
            for (int dt = 0; dt < C::DT; ++dt) {
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) {
                    o[dt][nh][0] *= alpha[nh][0];
                    o[dt][nh][1] *= alpha[nh][1];
                    o[dt][nh][2] *= alpha[nh][0];
                    o[dt][nh][3] *= alpha[nh][1];
                }
            }
        }
        // ---- P = exp2(S - m); P^T fragments as hi + lo 16-bit terms
        uint32_t pb_hi[C::MT][NH][2], pb_lo[C::MT][NH][2];
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) {
                float pr[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float x = sc[mt][nh][j];
                    pr[j] = (x == -INFINITY) ? 0.f : ex2_approx(x - m_run[nh][j & 1]);
                    l_run[nh][j & 1] += pr[j];
                }
                // rows g8 (j = 0, 1) and g8 + 8 (j = 2, 3); columns 2c4, 2c4 + 1
                const uint32_t h01 = M::pack(pr[0], pr[1]);
                const uint32_t h23 = M::pack(pr[2], pr[3]);
                const float2 f01 = unpack2<T>(h01), f23 = unpack2<T>(h23);
                const uint32_t l01 = M::pack(pr[0] - f01.x, pr[1] - f01.y);
                const uint32_t l23 = M::pack(pr[2] - f23.x, pr[3] - f23.y);
                pb_hi[mt][nh][0] = movm_t(h01);
                pb_hi[mt][nh][1] = movm_t(h23);
                pb_lo[mt][nh][0] = movm_t(l01);
                pb_lo[mt][nh][1] = movm_t(l23);
            }
        }
        // ---- O^T += V^T . P^T   (k = tokens of each m-tile)
        const bool partial = nvalid < C::TW;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
            // A fragment token pairs of this lane: regs 0/1 hold tokens 2c4, 2c4+1; regs 2/3 hold +8.
            uint32_t keep01 = 0xffffffffu, keep89 = 0xffffffffu;
            if (partial) {
                const int t = mt * 16 + 2 * c4;
                keep01 = (t < nvalid ? 0x0000ffffu : 0u) | (t + 1 < nvalid ? 0xffff0000u : 0u);
                keep89 = (t + 8 < nvalid ? 0x0000ffffu : 0u) | (t + 9 < nvalid ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int dt = 0; dt < C::DT; ++dt) {
                // matrices: 0 = (tok 0-7, chunk 2dt), 1 = (tok 0-7, 2dt+1), 2 = (tok 8-15, 2dt), 3 = (tok 8-15, 2dt+1)
                const int r = mt * 16 + (lm >> 1) * 8 + lr;
                const int c = 2 * dt + (lm & 1);
                uint32_t a[4];
                ldsm_x4_t(a, vb + tile_off<D>(r, c));
                if (partial) {  // rows past the slice may hold anything (NaN included): zero them
                    a[0] &= keep01;
                    a[1] &= keep01;
                    a[2] &= keep89;
                    a[3] &= keep89;
                }
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) {
                    M::mma(o[dt][nh], a, pb_hi[mt][nh][0], pb_hi[mt][nh][1]);
                    M::mma(o[dt][nh], a, pb_lo[mt][nh][0], pb_lo[mt][nh][1]);
                }
            }
        }
        if (patched) fence_proxy_async_smem();  // our stores precede the next TMA write of the stage
        __syncwarp();
        if (lane == 0 && k + C::ST < my_tiles) issue(k + C::ST);
    }

    if (!ok && lane == 0) {  // copies still in flight land before the CTA's shared memory is reused
        const int issued = my_tiles < waited + C::ST ? my_tiles : waited + C::ST;
        for (int k = waited; k < issued; ++k)
            if (!(stall && k == 0)) mbar_wait_bounded(bar0 + 8 * (k % C::ST), (k / C::ST) & 1);
    }

    // ---- fused append: the item owning a query row stores that row's new K/V into the pool
    if (fused && it.write_pos >= 0) {
        const int pos = it.write_pos;
        // the warp that prefetched this row stores it; otherwise warp 0 reads it again
        const int nb = max(it.new_begin, it.tok_begin);
        const bool held = nb < it.tok_end && nb == pos;
        const int writer = held ? ((nb - it.tok_begin) / C::TW) % C::NW : 0;
        if (warp == writer && held) rotate_pf();  // warp-collective, before the lanes split
        // (with RoPE the written row is always the held one: see the fused-append note above)
        if (warp == writer && row_lane && (held || !ROPE)) {
            const int64_t page = (pos >= it.tok_begin && pos < it.tok_end)
                                     ? pages(pos, p.page_size)
                                     : p.kv_indices[it.page_base + pos / p.page_size];
            if (page < 0 || page >= p.num_pages) {
                if (rch == 0) atomicOr(p.flags, PGQA_FLAG_PAGE_INDEX);
            } else {
                const uint4 val = held ? pf : new_row_chunk(pos);
                T *dst = static_cast<T *>(rv ? p.v_pool : p.k_pool) +
                         ((page * p.page_size + pos % p.page_size) * p.num_kv_heads + it.kv_head) * D + rch * 8;
                *reinterpret_cast<uint4 *>(dst) = val;
            }
        }
    }

    // ---- combine the warps.  Per head column: M = max_w m_w, L = sum_w l_w 2^(m_w - M),
    // O = sum_w 2^(m_w - M) O_w / L.  Each warp leaves (m, l, O) in its own stage area
    // (its TMA copies have all landed); after one CTA barrier every thread builds 8
    // output channels of one head.
#pragma unroll
    for (int nh = 0; nh < NH; ++nh) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l_run[nh][h] += __shfl_xor_sync(0xffffffffu, l_run[nh][h], 4);
            l_run[nh][h] += __shfl_xor_sync(0xffffffffu, l_run[nh][h], 8);
            l_run[nh][h] += __shfl_xor_sync(0xffffffffu, l_run[nh][h], 16);
        }
    }
    constexpr int OS = C::OS;
    static_assert((2 * HP + HP * OS) * 4 <= C::ST * C::STAGE_BYTES, "a warp's combine state fits its stages");
    auto state = [&](int w) { return reinterpret_cast<float *>(pipe + w * C::ST * C::STAGE_BYTES); };
    {
        float *st = state(warp);  // [HP] m, [HP] l, [HP][OS] O
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
            if (g8 == 0) {
                st[8 * nh + 2 * c4] = m_run[nh][0];
                st[8 * nh + 2 * c4 + 1] = m_run[nh][1];
                st[HP + 8 * nh + 2 * c4] = l_run[nh][0];
                st[HP + 8 * nh + 2 * c4 + 1] = l_run[nh][1];
            }
#pragma unroll
            for (int dt = 0; dt < C::DT; ++dt) {
                float *ow = st + 2 * HP + (8 * nh + 2 * c4) * OS + dt * 16 + g8;
                ow[0] = o[dt][nh][0];
                ow[OS] = o[dt][nh][1];
                ow[8] = o[dt][nh][2];
                ow[OS + 8] = o[dt][nh][3];
            }
        }
    }
    if (p.defer_wait) {
        // Completion order: this grid finishes only after the prefill grid before it.
        pdl_wait();
        pdl_launch_dependents();
    }
    __syncthreads();

    constexpr int CH8 = D / 8;
    for (int idx = threadIdx.x; idx < G * CH8; idx += C::NW * 32) {
        const int h = idx / CH8;
        const int c8 = (idx - h * CH8) * 8;
        float mw[C::NW], Mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NW; ++w) {
            mw[w] = state(w)[h];  // heads < G <= HP
            Mx = fmaxf(Mx, mw[w]);
        }
        float fw[C::NW], L = 0.f;
#pragma unroll
        for (int w = 0; w < C::NW; ++w) {
            fw[w] = (mw[w] == -INFINITY) ? 0.f : ex2_approx(mw[w] - Mx);
            L += state(w)[HP + h] * fw[w];
        }
        // L == 0 only when no key was admissible; a NaN (poisoned row) propagates.
        const float inv = (L == 0.f) ? 0.f : rcp_approx(L);
        float acc[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) acc[jj] = 0.f;
#pragma unroll
        for (int w = 0; w < C::NW; ++w) {
            const float4 a = *reinterpret_cast<const float4 *>(state(w) + 2 * HP + h * OS + c8);
            const float4 b = *reinterpret_cast<const float4 *>(state(w) + 2 * HP + h * OS + c8 + 4);
            const float f = fw[w] * inv;
            acc[0] += a.x * f; acc[1] += a.y * f; acc[2] += a.z * f; acc[3] += a.w * f;
            acc[4] += b.x * f; acc[5] += b.y * f; acc[6] += b.z * f; acc[7] += b.w * f;
        }
        const float lse2 = (L == 0.f) ? -INFINITY : Mx + lg2_approx(L);
        const int head = it.kv_head * G + h;
        if (it.out_slot < 0) {
            const size_t oi = (static_cast<size_t>(it.q_row) * p.num_qo_heads + head) * D + c8;
            if (p.out_dtype == PGQA_FP32) {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + oi);
                dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            } else {
                uint4 v;
                v.x = M::pack(acc[0], acc[1]);
                v.y = M::pack(acc[2], acc[3]);
                v.z = M::pack(acc[4], acc[5]);
                v.w = M::pack(acc[6], acc[7]);
                *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + oi) = v;
            }
            if (c8 == 0 && p.lse != nullptr)
                p.lse[static_cast<size_t>(it.q_row) * p.num_qo_heads + head] = lse2 * 0.6931471805599453f;
        } else {
            const size_t slot = static_cast<size_t>(it.out_slot) * G + h;
            float4 *dst = reinterpret_cast<float4 *>(p.partial_o + slot * D + c8);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            if (c8 == 0) p.partial_lse[slot] = lse2;
        }
    }
}

// Raises the kernel's dynamic shared-memory limit once per device.
template <int D, int STAGES, int NH, bool ROPE, typename T, int NW = kDecodeWarps>
cudaError_t configure_decode_tc() {
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(decode_tc_kernel<D, STAGES, NH, ROPE, T, NW>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<D, STAGES, NW>::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    return cudaSuccess;
}

template <int D, int STAGES, int NH, bool ROPE, typename T, int NW = kDecodeWarps>
cudaError_t launch_decode_tc_st(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeParams &p,
                                int num_items, bool pdl, cudaStream_t stream) {
    using C = TcCfg<D, STAGES, NW>;
    cudaError_t e = configure_decode_tc<D, STAGES, NH, ROPE, T, NW>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_items);
    cfg.blockDim = dim3(C::NW * 32);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel<D, STAGES, NH, ROPE, T, NW>, tm_k, tm_v, p, group);
}

// The rotary variant is a separate instantiation, so plans without RoPE run code
// with no trace of it (timed: the runtime branch alone cost 3 % on 128 x 301).
template <int D, int STAGES, int NH, typename T, int NW = kDecodeWarps>
cudaError_t launch_decode_tc_r(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeParams &p,
                               int num_items, bool pdl, cudaStream_t stream) {
    return p.rope_cs != nullptr
               ? launch_decode_tc_st<D, STAGES, NH, true, T, NW>(group, tm_k, tm_v, p, num_items, pdl, stream)
               : launch_decode_tc_st<D, STAGES, NH, false, T, NW>(group, tm_k, tm_v, p, num_items, pdl, stream);
}

// CTAs of one per-item kernel variant resident on an SM at once (registers and
// shared memory), the slot count of the split heuristic.
template <int D, int STAGES, int NH, typename T, int NW = kDecodeWarps>
cudaError_t decode_tc_blocks_per_sm_st(int *blocks) {
    cudaError_t e = configure_decode_tc<D, STAGES, NH, false, T, NW>();
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, decode_tc_kernel<D, STAGES, NH, false, T, NW>,
                                                         NW * 32, TcCfg<D, STAGES, NW>::SMEM_BYTES);
}

// stages 1 selects the wide form (kDecodeWideWarps warps, one tile each; groups of up to 8).
template <int D, typename T>
cudaError_t decode_tc_blocks_per_sm(int stages, int group, int *blocks) {
    if (stages == 1) return decode_tc_blocks_per_sm_st<D, 1, 1, T, kDecodeWideWarps>(blocks);
    if (group > 8)
        return stages == 3 ? decode_tc_blocks_per_sm_st<D, 3, 2, T>(blocks) : decode_tc_blocks_per_sm_st<D, 2, 2, T>(blocks);
    return stages == 3 ? decode_tc_blocks_per_sm_st<D, 3, 1, T>(blocks) : decode_tc_blocks_per_sm_st<D, 2, 1, T>(blocks);
}

template <int D, typename T>
cudaError_t launch_decode_tc(int stages, int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const DecodeParams &p, int num_items, bool pdl, cudaStream_t stream) {
    if (stages == 1) {
        if (group > 8) return cudaErrorInvalidValue;  // the plan never picks the wide form for them
        return launch_decode_tc_r<D, 1, 1, T, kDecodeWideWarps>(group, tm_k, tm_v, p, num_items, pdl, stream);
    }
    if (group > 8)
        return stages == 3 ? launch_decode_tc_r<D, 3, 2, T>(group, tm_k, tm_v, p, num_items, pdl, stream)
                           : launch_decode_tc_r<D, 2, 2, T>(group, tm_k, tm_v, p, num_items, pdl, stream);
    return stages == 3 ? launch_decode_tc_r<D, 3, 1, T>(group, tm_k, tm_v, p, num_items, pdl, stream)
                       : launch_decode_tc_r<D, 2, 1, T>(group, tm_k, tm_v, p, num_items, pdl, stream);
}

}  // namespace pgqa
