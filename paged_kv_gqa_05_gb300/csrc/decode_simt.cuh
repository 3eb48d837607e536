// Split-KV paged GQA decode: the partial kernel.
//
// One CTA per work item = (query row, kv head, key slice); the CTA serves all
// G = Hq/Hkv query heads that share the kv head, so each K/V row of the slice is
// read from HBM once for the whole group.  Split-KV as in "A library kernel for
// decode", section "What changed": the slice's partial (output, log-sum-exp) is
// written for a later merge, or, when the row has a single slice, the final
// output is written directly.
//
// Data movement: every warp runs its own kDecodeStages-deep ring of shared
// memory stages.  Lane 0 resolves the page of each warp tile through the page
// table and issues 3-D TMA box loads ([rows, 1 kv head, head_dim]) of K and V
// into the stage, completing on a per-stage mbarrier.  The pool is addressed as
// the 3-D tensor [num_pages * page_size, Hkv, head_dim] (the "flashlet" README's
// NHD pool layout), so one box is at most one page of one kv head.
//
// Math (fp32, CUDA cores): a key row is split over GS = head_dim/8 lanes, each
// holding 8 channels of q for all G heads in registers.  A group of GS lanes
// takes 8 tokens at a time; lane c visits them in the order t ^ (c & 7) so that
// a 3-step butterfly reduce-scatter (shfl_xor 4, 2, 1) leaves lane c holding
// the complete scores of token (c & 7) without any select.  Online softmax
// keeps a running max per (group, head) in the log2 domain (q is pre-scaled by
// scale * log2 e, exponentials are exp2).  Probabilities go through a small
// per-warp shared buffer (stored as duplicated pairs) so that PV runs as packed
// fp32x2 FMAs over each lane's 8 channels.  At the end the groups of the CTA
// are combined with the same log-sum-exp rule the merge kernel uses.
#pragma once

#include <math.h>

#include <atomic>

#include "common.cuh"

namespace pgqa {

template <int D, int G>
struct DecodeCfg {
    static constexpr int GS = D / 8;             // lanes per key row
    static constexpr int GPW = 32 / GS;          // key rows per warp step
    static constexpr int TW = 8 * GPW;           // tokens per warp tile
    static constexpr int NW = kDecodeWarps;
    static constexpr int ST = kDecodeStages;
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int TILE_BYTES = TW * ROW_BYTES;   // K (or V) of one warp tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
    static constexpr int PIPE_BYTES = NW * ST * STAGE_BYTES;
    static constexpr int BAR_BYTES = NW * ST * 8;
    static constexpr int GPAD = (G + 1) / 2 * 2;        // heads padded to an even count
    static constexpr int PB_TOK = GPAD * 8;             // one token: GPAD duplicated pairs
    static constexpr int PB_GROUP = 8 * PB_TOK + 16;    // +16 B staggers groups across banks
    static constexpr int PB_WARP = GPW * PB_GROUP;
    static constexpr int PB_BYTES = NW * PB_WARP;
    static constexpr int NG = NW * GPW;                 // softmax groups per CTA
    static constexpr int COMBINE_BYTES = NG * G * (D + 2) * 4;
    static constexpr int SMEM_BYTES = PIPE_BYTES + BAR_BYTES + PB_BYTES + kSlicePageCap * 4;
    static_assert(COMBINE_BYTES <= PIPE_BYTES, "combine buffer reuses the pipeline stages");
    static_assert(TW % 16 == 0, "warp tile covers whole 16-row boxes");
};

template <typename T>
__device__ __forceinline__ void store_out(void *out, size_t idx, float v, int out_dtype) {
    if (out_dtype == PGQA_FP32)
        static_cast<float *>(out)[idx] = v;
    else
        static_cast<T *>(out)[idx] = narrow<T>(v);
}

template <int D, int G, typename T>
__global__ void __launch_bounds__(kDecodeWarps * 32, 2)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
    using C = DecodeCfg<D, G>;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gi = lane / C::GS;      // group within the warp
    const int cc = lane % C::GS;      // channel chunk: channels [8cc, 8cc + 8)
    const int c8 = cc & 7;            // token permutation key
    const unsigned gmask = (C::GS == 32 ? 0xffffffffu : ((1u << C::GS) - 1u) << (gi * C::GS));

    uint8_t *pipe = smem;
    uint8_t *pbuf = smem + C::PIPE_BYTES + C::BAR_BYTES + warp * C::PB_WARP + gi * C::PB_GROUP;
    const uint32_t bar0 = smem_addr(smem + C::PIPE_BYTES) + warp * C::ST * 8;

    if (smem_addr(smem) & 127u) {  // the stage layout assumes this alignment of the window
        if (threadIdx.x == 0) atomicOr(p.flags, PGQA_FLAG_SMEM_ALIGN);
        pdl_wait();  // completion order: this grid ends after the one before it
        return;
    }
    // The work list and kv_indices are final once plan_update is enqueued, so they
    // are read before the dependency wait; q and the pools only after it.
    const WorkItem it = p.items[blockIdx.x];
    const int ntiles = (it.tok_end - it.tok_begin + C::TW - 1) / C::TW;
    const int my_tiles = ntiles > warp ? (ntiles - warp + C::NW - 1) / C::NW : 0;
    int32_t *page_buf = reinterpret_cast<int32_t *>(smem + C::PIPE_BYTES + C::BAR_BYTES + C::PB_BYTES);

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
    __syncthreads();

    pdl_wait();
    // Our predecessors are complete from here on, so a grid launched early after this
    // trigger never overlaps a kernel older than this one.
    pdl_launch_dependents();

    // Lane 0: resolve the pages of warp tile k and issue its K and V boxes.
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
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nvalid * p.box_rows * C::ROW_BYTES * 2));
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
            if (rows[c] >= 0) {
                const uint32_t off = c * p.box_rows * C::ROW_BYTES;
                tma_load_3d(kdst + off, &tm_k, 0, it.kv_head, rows[c], bar);
                tma_load_3d(vdst + off, &tm_v, 0, it.kv_head, rows[c], bar);
            }
        }
    };

    if (lane == 0) {
        const int pre = my_tiles < C::ST ? my_tiles : C::ST;
        for (int k = 0; k < pre; ++k) issue(k);
    }

    // q for this lane's 8 channels of the G heads, pre-scaled into the log2 domain.
    float2 q2[G][4];
    {
        const T *qp = static_cast<const T *>(p.q) +
                      (static_cast<size_t>(it.q_row) * p.num_qo_heads + it.kv_head * G) * D + cc * 8;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(qp + h * D));
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = widen2<T>(w4[j]);
                q2[h][j] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
            }
        }
    }

    float m_run[G], l_run[G];
    float2 o2[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) o2[h][j] = make_float2(0.f, 0.f);
    }

    int waited = 0;  // tiles whose barrier this warp has passed
    bool ok = true;
    for (int k = 0; k < my_tiles; ++k) {
        const int s = k % C::ST;
        // every lane observes the phase (TMA data visibility); the outcome is made warp-uniform
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * s, (k / C::ST) & 1))) {
            if (lane == 0) atomicOr(p.flags, PGQA_FLAG_WAIT_TIMEOUT);
            ok = false;
            break;
        }
        waited = k + 1;
        const int tile = warp + k * C::NW;
        const int tb = it.tok_begin + tile * C::TW;
        const int nvalid = min(C::TW, it.tok_end - tb);
        const uint8_t *kbase = pipe + (warp * C::ST + s) * C::STAGE_BYTES;
        const uint8_t *vbase = kbase + C::TILE_BYTES;
        const int gt = gi * 8;
        const int nv_g = min(max(nvalid - gt, 0), 8);

        if (nv_g > 0) {
            // ---- scores: s[t][h] = q_h . k_{t ^ c8} over this lane's 8 channels
            float sc[8][G];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint4 kr = lds128(kbase + (gt + (t ^ c8)) * C::ROW_BYTES + cc * 16);
                const float2 k0 = widen2<T>(kr.x), k1 = widen2<T>(kr.y);
                const float2 k2 = widen2<T>(kr.z), k3 = widen2<T>(kr.w);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float2 a = __fmul2_rn(q2[h][0], k0);
                    a = __ffma2_rn(q2[h][1], k1, a);
                    a = __ffma2_rn(q2[h][2], k2, a);
                    a = __ffma2_rn(q2[h][3], k3, a);
                    sc[t][h] = a.x + a.y;
                }
            }
            // ---- butterfly reduce-scatter over the 8 channel chunks: slot i of
            // this lane and slot i + m of lane ^ m hold the same token.
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int i = 0; i < 4; ++i) sc[i][h] += __shfl_xor_sync(gmask, sc[4 + i][h], 4);
#pragma unroll
                for (int i = 0; i < 2; ++i) sc[i][h] += __shfl_xor_sync(gmask, sc[2 + i][h], 2);
                sc[0][h] += __shfl_xor_sync(gmask, sc[1][h], 1);
                if (C::GS == 16) sc[0][h] += __shfl_xor_sync(gmask, sc[0][h], 8);
            }
            // ---- online softmax (log2 domain); lane holds token gt + c8
            const bool valid = (gt + c8) < nvalid;
            float pr[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float x = valid ? sc[0][h] : -INFINITY;
                float mx = x;
                mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, 4));
                if (mx > m_run[h]) {  // uniform within the group
                    const float alpha = exp2f(m_run[h] - mx);
                    m_run[h] = mx;
                    l_run[h] *= alpha;
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int j = 0; j < 4; ++j) o2[h][j] = __fmul2_rn(o2[h][j], a2);
                }
                pr[h] = valid ? exp2f(x - m_run[h]) : 0.f;
                if (cc < 8) l_run[h] += pr[h];
            }
            if (cc < 8) {
                float2 *dst = reinterpret_cast<float2 *>(pbuf + c8 * C::PB_TOK);
#pragma unroll
                for (int h = 0; h < G; ++h) dst[h] = make_float2(pr[h], pr[h]);
            }
            __syncwarp(gmask);
            // ---- o += p_t * v_t over this lane's 8 channels
            const uint8_t *pb = pbuf;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (t < nv_g) {
                    const uint4 vr = lds128(vbase + (gt + t) * C::ROW_BYTES + cc * 16);
                    const float2 v0 = widen2<T>(vr.x), v1 = widen2<T>(vr.y);
                    const float2 v2 = widen2<T>(vr.z), v3 = widen2<T>(vr.w);
#pragma unroll
                    for (int hp = 0; hp < C::GPAD / 2; ++hp) {
                        const uint4 pp = lds128(pb + t * C::PB_TOK + hp * 16);
                        const float2 pa = make_float2(__uint_as_float(pp.x), __uint_as_float(pp.y));
                        const float2 pc = make_float2(__uint_as_float(pp.z), __uint_as_float(pp.w));
                        const int h0 = 2 * hp, h1 = 2 * hp + 1;
                        o2[h0][0] = __ffma2_rn(pa, v0, o2[h0][0]);
                        o2[h0][1] = __ffma2_rn(pa, v1, o2[h0][1]);
                        o2[h0][2] = __ffma2_rn(pa, v2, o2[h0][2]);
                        o2[h0][3] = __ffma2_rn(pa, v3, o2[h0][3]);
                        if (h1 < G) {
                            o2[h1][0] = __ffma2_rn(pc, v0, o2[h1][0]);
                            o2[h1][1] = __ffma2_rn(pc, v1, o2[h1][1]);
                            o2[h1][2] = __ffma2_rn(pc, v2, o2[h1][2]);
                            o2[h1][3] = __ffma2_rn(pc, v3, o2[h1][3]);
                        }
                    }
                }
            }
        }
        __syncwarp();  // every lane is done with this stage and with pbuf
        if (lane == 0 && k + C::ST < my_tiles) issue(k + C::ST);
    }

    if (!ok && lane == 0) {
        // Let copies already in flight land before the CTA's shared memory goes away.
        const int issued = my_tiles < waited + C::ST ? my_tiles : waited + C::ST;
        for (int k = waited; k < issued; ++k) mbar_wait_bounded(bar0 + 8 * (k % C::ST), (k / C::ST) & 1);
    }

    // ---- combine the CTA's softmax groups
    float l_tot[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float l = l_run[h];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l_tot[h] = l;
    }
    __syncthreads();  // pipeline stages are free from here on
    float *cm = reinterpret_cast<float *>(smem);  // [NG][G]
    float *cl = cm + C::NG * G;                   // [NG][G]
    float *co = cl + C::NG * G;                   // [NG][G][D]
    const int grp = warp * C::GPW + gi;
    if (cc == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            cm[grp * G + h] = m_run[h];
            cl[grp * G + h] = l_tot[h];
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float4 *dst = reinterpret_cast<float4 *>(co + (grp * G + h) * D + cc * 8);
        dst[0] = make_float4(o2[h][0].x, o2[h][0].y, o2[h][1].x, o2[h][1].y);
        dst[1] = make_float4(o2[h][2].x, o2[h][2].y, o2[h][3].x, o2[h][3].y);
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < G * D; idx += C::NW * 32) {
        const int h = idx / D;
        const int c = idx - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int g = 0; g < C::NG; ++g) M = fmaxf(M, cm[g * G + h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int g = 0; g < C::NG; ++g) {
                const float mg = cm[g * G + h];
                if (mg != -INFINITY) {
                    const float w = exp2f(mg - M);
                    L += cl[g * G + h] * w;
                    O += co[(g * G + h) * D + c] * w;
                }
            }
        }
        // L == 0 only for a slice with no admissible key; NaN (a poisoned row) propagates.
        const float o = L == 0.f ? 0.f : O / L;
        const float lse2 = L == 0.f ? -INFINITY : M + log2f(L);
        const int head = it.kv_head * G + h;
        if (it.out_slot < 0) {
            const size_t oi = (static_cast<size_t>(it.q_row) * p.num_qo_heads + head) * D + c;
            store_out<T>(p.out, oi, o, p.out_dtype);
            if (c == 0 && p.lse != nullptr)
                p.lse[static_cast<size_t>(it.q_row) * p.num_qo_heads + head] = lse2 * 0.6931471805599453f;
        } else {
            const size_t slot = static_cast<size_t>(it.out_slot) * G + h;
            p.partial_o[slot * D + c] = o;
            if (c == 0) p.partial_lse[slot] = lse2;
        }
    }
}

template <int D, int G, typename T>
cudaError_t launch_decode_g(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeParams &p,
                            int num_items, bool pdl, cudaStream_t stream) {
    using C = DecodeCfg<D, G>;
    auto kern = decode_partial_kernel<D, G, T>;
    // The shared-memory opt-in is set once per device (before any stream capture
    // that follows a first eager call).
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
    cfg.blockDim = dim3(C::NW * 32);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_k, tm_v, p);
}

template <int D, typename T>
cudaError_t launch_decode_dt(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const DecodeParams &p, int num_items, bool pdl, cudaStream_t stream) {
    if (p.rope_cs != nullptr) return cudaErrorInvalidValue;  // rotary plans use the tensor-core kernel
    switch (group) {
        case 1: return launch_decode_g<D, 1, T>(tm_k, tm_v, p, num_items, pdl, stream);
        case 2: return launch_decode_g<D, 2, T>(tm_k, tm_v, p, num_items, pdl, stream);
        case 3: return launch_decode_g<D, 3, T>(tm_k, tm_v, p, num_items, pdl, stream);
        case 4: return launch_decode_g<D, 4, T>(tm_k, tm_v, p, num_items, pdl, stream);
        case 5: return launch_decode_g<D, 5, T>(tm_k, tm_v, p, num_items, pdl, stream);
        case 6: return launch_decode_g<D, 6, T>(tm_k, tm_v, p, num_items, pdl, stream);
        case 7: return launch_decode_g<D, 7, T>(tm_k, tm_v, p, num_items, pdl, stream);
        case 8: return launch_decode_g<D, 8, T>(tm_k, tm_v, p, num_items, pdl, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pgqa
