// Log-sum-exp merge of split-KV partials.
//
// "A library kernel for decode", section "What changed": the partial results of
// a request's slices are merged.  Each slice s of (query row, head) left an
// output o_s normalised over its slice and lse_s (log2 domain); the merged
// result is
//     lse = log2 sum_s 2^lse_s,   o = sum_s 2^(lse_s - lse) o_s,
// with empty slices (lse_s = -inf) carrying no weight.
//
// Two launch shapes.  Up to 32 slices per row: one warp per (task, head), the
// slice weights one per lane.  Longer lists: a block of 256 threads per (task,
// head, 32-channel chunk) = 8 float4 columns x 32 slice groups, so a long list
// is read with many independent coalesced loads in flight.
#include <math.h>

#include <type_traits>

#include "common.cuh"

namespace pgqa {

namespace {

constexpr int kMergeThreads = 256;
constexpr int kChunk = 32;  // channels per block

__device__ __forceinline__ float block_reduce(float v, float *scratch, bool is_max) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, m);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = scratch[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) v = is_max ? fmaxf(v, scratch[w]) : v + scratch[w];
    return v;
}

template <typename OutT>
__device__ __forceinline__ void put(void *out, size_t i, float v);
template <>
__device__ __forceinline__ void put<float>(void *out, size_t i, float v) { static_cast<float *>(out)[i] = v; }
template <>
__device__ __forceinline__ void put<__nv_bfloat16>(void *out, size_t i, float v) {
    static_cast<__nv_bfloat16 *>(out)[i] = __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ void put<__half>(void *out, size_t i, float v) {
    static_cast<__half *>(out)[i] = __float2half_rn(v);
}

// V consecutive outputs of one lane (V = 2 or 4, oi a multiple of V) as one store.
template <typename OutT, int V>
__device__ __forceinline__ void put_row(void *out, size_t oi, const float (&v)[V]) {
    if constexpr (std::is_same<OutT, float>::value) {
        if constexpr (V == 4)
            *reinterpret_cast<float4 *>(static_cast<float *>(out) + oi) = make_float4(v[0], v[1], v[2], v[3]);
        else
            *reinterpret_cast<float2 *>(static_cast<float *>(out) + oi) = make_float2(v[0], v[1]);
    } else {
        uint32_t w[V / 2];
#pragma unroll
        for (int j = 0; j < V / 2; ++j) {
            OutT pair[2];
            put<OutT>(pair, 0, v[2 * j]);
            put<OutT>(pair, 1, v[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t *>(pair);
        }
        if constexpr (V == 4)
            *reinterpret_cast<uint2 *>(static_cast<OutT *>(out) + oi) = make_uint2(w[0], w[1]);
        else
            *reinterpret_cast<uint32_t *>(static_cast<OutT *>(out) + oi) = w[0];
    }
}

template <typename OutT>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
    extern __shared__ float sm[];
    float *red = sm;                         // [32 slice groups][32 channels]
    float *scratch = red + 32 * kChunk;      // [8]
    float *w = scratch + 8;                  // [num_splits]

    pdl_launch_dependents();
    const MergeTask t = p.tasks[blockIdx.x];  // written by plan_update's copy only
    const int h = blockIdx.y;
    const int c0 = blockIdx.z * kChunk;
    const int G = p.group, D = p.head_dim, ns = t.num_splits;

    pdl_wait();

    // The partial outputs do not depend on the weights: the first kPrefetch of this
    // thread's slices are requested together with the lse values, so the block waits
    // out one memory latency instead of two.
    const int c4 = threadIdx.x & 7, sg = threadIdx.x >> 3;
    const float *base = p.partial_o + (static_cast<size_t>(t.slot_base) * G + h) * D + c0 + c4 * 4;
    const size_t stride = static_cast<size_t>(G) * D;
    constexpr int kPrefetch = 8;  // slices sg + 32 i, i < kPrefetch: lists of up to 256 slices
    float4 pre[kPrefetch];
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i) {
        const int s = sg + 32 * i;
        pre[i] = s < ns ? __ldg(reinterpret_cast<const float4 *>(base + s * stride)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const float *lse_in = p.partial_lse + static_cast<size_t>(t.slot_base) * G + h;
    float mx = -INFINITY;
    for (int s = threadIdx.x; s < ns; s += kMergeThreads) {
        const float v = lse_in[static_cast<size_t>(s) * G];
        w[s] = v;
        mx = fmaxf(mx, v);
    }
    mx = block_reduce(mx, scratch, true);
    float sum = 0.f;
    for (int s = threadIdx.x; s < ns; s += kMergeThreads) {
        const float e = (w[s] == -INFINITY) ? 0.f : exp2f(w[s] - mx);  // NaN lse stays NaN
        w[s] = e;
        sum += e;
    }
    sum = block_reduce(sum, scratch, false);  // also publishes w[] to the block

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i) {
        const int s = sg + 32 * i;
        const float ws = s < ns ? w[s] : 0.f;
        if (ws != 0.f) {  // also taken for NaN weights
            acc.x += ws * pre[i].x;
            acc.y += ws * pre[i].y;
            acc.z += ws * pre[i].z;
            acc.w += ws * pre[i].w;
        }
    }
#pragma unroll 4
    for (int s = sg + 32 * kPrefetch; s < ns; s += 32) {
        const float ws = w[s];
        if (ws != 0.f) {  // also taken for NaN weights
            const float4 v = __ldg(reinterpret_cast<const float4 *>(base + s * stride));
            acc.x += ws * v.x;
            acc.y += ws * v.y;
            acc.z += ws * v.z;
            acc.w += ws * v.w;
        }
    }
    reinterpret_cast<float4 *>(red)[sg * 8 + c4] = acc;
    __syncthreads();
    if (threadIdx.x < kChunk) {
        float tot = 0.f;
#pragma unroll 8
        for (int g = 0; g < 32; ++g) tot += red[g * kChunk + threadIdx.x];
        const int head = t.kv_head * G + h;
        const size_t oi = (static_cast<size_t>(t.q_row) * p.num_qo_heads + head) * D + c0 + threadIdx.x;
        put<OutT>(p.out, oi, sum == 0.f ? 0.f : tot / sum);  // NaN propagates
        if (threadIdx.x == 0 && blockIdx.z == 0 && p.lse != nullptr)
            p.lse[static_cast<size_t>(t.q_row) * p.num_qo_heads + head] =
                sum == 0.f ? -INFINITY : (mx + log2f(sum)) * 0.6931471805599453f;
    }
}

// Short slice lists (<= 32 per row): one warp per (task, head).  Lane s holds the
// weight of slice s; each lane owns D/32 consecutive channels of every slice.  The
// partials of the first P slices are requested up front; P follows the call's longest
// list (4, 8 or 16), since registers held for slices a call does not have cost
// occupancy beside the decode grid (timed on GB300: 32 mixed-length rows of 10 slices,
// 13.27 against 13.61 us per layer with P = 16 instead of 8; the ragged call, rows of
// 2-3 slices, 38.0 us with P = 4, 38.2 with 8, 38.5 with 16).
template <typename OutT, int D, int P>
__global__ void __launch_bounds__(256) merge_warp_kernel(const MergeParams p, int units) {
    pdl_launch_dependents();
    constexpr int V = D / 32;  // channels per lane: 2 (D = 64) or 4 (D = 128)
    const int lane = threadIdx.x & 31;
    const int u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (u >= units) return;
    const int G = p.group;
    const MergeTask t = p.tasks[u / G];  // written by plan_update's copy only
    const int h = u - (u / G) * G;
    const int ns = t.num_splits;

    pdl_wait();

    // Partial outputs of the first kPrefetch slices are requested with the lse values
    // (they do not depend on the weights): one memory latency before the fold, not two.
    const float *base = p.partial_o + (static_cast<size_t>(t.slot_base) * G + h) * D + lane * V;
    const size_t stride = static_cast<size_t>(G) * D;
    constexpr int kPrefetch = P;
    float pre[kPrefetch][V];
#pragma unroll
    for (int s = 0; s < kPrefetch; ++s) {
        if (s < ns) {
            if (V == 4) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(base + s * stride));
                pre[s][0] = v.x; pre[s][1 % V] = v.y; pre[s][2 % V] = v.z; pre[s][3 % V] = v.w;
            } else {
                const float2 v = __ldg(reinterpret_cast<const float2 *>(base + s * stride));
                pre[s][0] = v.x; pre[s][1 % V] = v.y;
            }
        }
    }

    const float l = lane < ns ? p.partial_lse[static_cast<size_t>(t.slot_base + lane) * G + h] : -INFINITY;
    float mx = l;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    const float w = (l == -INFINITY) ? 0.f : exp2f(l - mx);  // NaN lse stays NaN
    float sum = w;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);

    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
#pragma unroll
    for (int s = 0; s < kPrefetch; ++s) {
        const float ws = __shfl_sync(0xffffffffu, w, s);  // lanes >= ns carry weight 0
        if (s < ns) {
#pragma unroll
            for (int j = 0; j < V; ++j) acc[j] += ws * pre[s][j];
        }
    }
#pragma unroll 8
    for (int s = kPrefetch; s < ns; ++s) {
        const float ws = __shfl_sync(0xffffffffu, w, s);
        if (V == 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(base + s * stride));
            acc[0] += ws * v.x;
            acc[1 % V] += ws * v.y;
            acc[2 % V] += ws * v.z;
            acc[3 % V] += ws * v.w;
        } else {
            const float2 v = __ldg(reinterpret_cast<const float2 *>(base + s * stride));
            acc[0] += ws * v.x;
            acc[1 % V] += ws * v.y;
        }
    }
    const int head = t.kv_head * G + h;
    const size_t oi = (static_cast<size_t>(t.q_row) * p.num_qo_heads + head) * D + lane * V;
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = sum == 0.f ? 0.f : acc[j] / sum;
    put_row<OutT, V>(p.out, oi, acc);  // one vector store per lane
    if (lane == 0 && p.lse != nullptr)
        p.lse[static_cast<size_t>(t.q_row) * p.num_qo_heads + head] =
            sum == 0.f ? -INFINITY : (mx + log2f(sum)) * 0.6931471805599453f;
}

template <typename OutT>
cudaError_t launch_merge_t(const MergeParams &p, int num_tasks, int max_splits, bool pdl,
                           cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    if (max_splits <= 32) {
        const int units = num_tasks * p.group;
        cudaLaunchConfig_t cfg = {};
        // Four warps a block, or eight for long lists of units (timed on GB300: the ragged
        // call's ~8000 units 33.1 -> 32.8 us, the 512-row chunk's ~7200 15.1 -> 14.9; 32
        // mixed rows, 228 units, 13.24 -> 13.33 with eight, so they keep four).
        const int wpb = units >= 2048 ? 8 : 4;
        cfg.gridDim = dim3((units + wpb - 1) / wpb);
        cfg.blockDim = dim3(32 * wpb);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (max_splits <= 4)
            return p.head_dim == 64 ? cudaLaunchKernelEx(&cfg, merge_warp_kernel<OutT, 64, 4>, p, units)
                                    : cudaLaunchKernelEx(&cfg, merge_warp_kernel<OutT, 128, 4>, p, units);
        if (max_splits <= 8)
            return p.head_dim == 64 ? cudaLaunchKernelEx(&cfg, merge_warp_kernel<OutT, 64, 8>, p, units)
                                    : cudaLaunchKernelEx(&cfg, merge_warp_kernel<OutT, 128, 8>, p, units);
        return p.head_dim == 64 ? cudaLaunchKernelEx(&cfg, merge_warp_kernel<OutT, 64, 16>, p, units)
                                : cudaLaunchKernelEx(&cfg, merge_warp_kernel<OutT, 128, 16>, p, units);
    }
    const size_t smem = (32 * kChunk + 8 + static_cast<size_t>(max_splits)) * sizeof(float);
    auto kern = merge_kernel<OutT>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_tasks, p.group, p.head_dim / kChunk);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, int num_tasks, int max_splits, bool pdl,
                         cudaStream_t stream) {
    switch (p.out_dtype) {
        case PGQA_FP32: return launch_merge_t<float>(p, num_tasks, max_splits, pdl, stream);
        case PGQA_BF16: return launch_merge_t<__nv_bfloat16>(p, num_tasks, max_splits, pdl, stream);
        case PGQA_FP16: return launch_merge_t<__half>(p, num_tasks, max_splits, pdl, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pgqa
