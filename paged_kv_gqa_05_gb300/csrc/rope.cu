// Rotary position embedding on the append path.
//
// The "flashlet" README lists a RoPE fusion kernel among its milestones and
// "Torchlet"'s Qwen2.5-style model includes RoPE; neither writes the rotation
// out.  It is taken in the rotate-half form of the Qwen2.5 models: channel
// i < D/2 pairs with channel i + D/2 and both turn by pos * theta^(-2i/D).
//
// A plan that uses RoPE owns a table of (cos, sin) per (position, i), built once
// here in fp64 and rounded to fp32, so no kernel on the hot path evaluates a
// trigonometric function (fp64 is slow on this part; fp32 angles at positions in
// the tens of thousands would lose ~1e-3 rad).  The rotation itself is
// rope_rotate2 (common.cuh), shared by every kernel that rotates.
#include "common.cuh"

namespace pgqa {

namespace {

__global__ void __launch_bounds__(256) rope_table_kernel(float2 *cs, int64_t n, int half, int head_dim,
                                                         double log2_theta) {
    for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n;
         k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t pos = k / half;
        const int i = static_cast<int>(k - pos * half);
        const double inv_freq = exp2(-2.0 * i / head_dim * log2_theta);  // theta^(-2i/d)
        double s, c;
        sincos(static_cast<double>(pos) * inv_freq, &s, &c);
        cs[k] = make_float2(static_cast<float>(c), static_cast<float>(s));
    }
}

// One thread per 16-byte chunk of a (token, kv head) row: K rotated at the token's
// position, V copied.  A skipped row (negative slot, slot or position out of range)
// is skipped for both K and V.
template <typename T, int D>
__global__ void __launch_bounds__(256)
    kv_append_rope_kernel(T *__restrict__ k_pool, T *__restrict__ v_pool, const T *__restrict__ k,
                          const T *__restrict__ v, const int64_t *__restrict__ slots,
                          const int32_t *__restrict__ positions, int64_t num_tokens, int64_t num_slots,
                          int num_kv_heads, const float2 *__restrict__ cs, int max_position,
                          unsigned int *flags) {
    pdl_launch_dependents();  // the next grid waits for our completion before reading the pool
    pdl_wait();
    constexpr int CH = D / 8;
    const int64_t n = num_tokens * num_kv_heads * CH;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = idx / CH;  // token * num_kv_heads + head
        const int ch = static_cast<int>(idx - row * CH);
        const int64_t t = row / num_kv_heads;
        const int64_t s = __ldg(slots + t);
        if (s < 0) continue;  // padding row
        if (s >= num_slots) {
            if (ch == 0) atomicOr(flags, PGQA_FLAG_SLOT_RANGE);
            continue;
        }
        const int32_t pos = __ldg(positions + t);
        if (pos < 0 || pos >= max_position) {
            if (ch == 0) atomicOr(flags, PGQA_FLAG_ROPE_POSITION);
            continue;
        }
        const int64_t head = row - t * num_kv_heads;
        const size_t dst = (static_cast<size_t>(s) * num_kv_heads + head) * D + ch * 8;
        *reinterpret_cast<uint4 *>(k_pool + dst) =
            rope_chunk<T, D>(k + static_cast<size_t>(row) * D, ch, cs + static_cast<size_t>(pos) * (D / 2));
        *reinterpret_cast<uint4 *>(v_pool + dst) =
            __ldg(reinterpret_cast<const uint4 *>(v + static_cast<size_t>(row) * D + ch * 8));
    }
}

template <typename T, int D>
cudaError_t launch_append_rope_t(void *k_pool, void *v_pool, const void *k, const void *v, const int64_t *slots,
                                 const int32_t *positions, int64_t num_tokens, int64_t num_slots,
                                 int num_kv_heads, const float2 *cs, int max_position, unsigned int *flags,
                                 bool pdl, cudaStream_t stream) {
    const int64_t n = num_tokens * num_kv_heads * (D / 8);
    const int threads = 256;
    int64_t blocks = (n + threads - 1) / threads;
    if (blocks > 65535) blocks = 65535;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kv_append_rope_kernel<T, D>, static_cast<T *>(k_pool), static_cast<T *>(v_pool),
                              static_cast<const T *>(k), static_cast<const T *>(v), slots, positions, num_tokens,
                              num_slots, num_kv_heads, cs, max_position, flags);
}

}  // namespace

cudaError_t launch_rope_table(float2 *cs, int max_position, int head_dim, double theta, cudaStream_t stream) {
    const int half = head_dim / 2;
    const int64_t n = static_cast<int64_t>(max_position) * half;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    rope_table_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(cs, n, half, head_dim, log2(theta));
    return cudaGetLastError();
}

cudaError_t launch_kv_append_rope(void *k_pool, void *v_pool, const void *k, const void *v,
                                  const int64_t *slot_mapping, const int32_t *positions, int64_t num_tokens,
                                  int64_t num_slots, int num_kv_heads, int head_dim, pgqa_dtype dtype,
                                  const float2 *cs, int max_position, unsigned int *flags, bool pdl,
                                  cudaStream_t stream) {
    auto f = dtype == PGQA_BF16 ? (head_dim == 64 ? launch_append_rope_t<__nv_bfloat16, 64>
                                                  : launch_append_rope_t<__nv_bfloat16, 128>)
                                : (head_dim == 64 ? launch_append_rope_t<__half, 64> : launch_append_rope_t<__half, 128>);
    return f(k_pool, v_pool, k, v, slot_mapping, positions, num_tokens, num_slots, num_kv_heads, cs, max_position,
             flags, pdl, stream);
}

}  // namespace pgqa
