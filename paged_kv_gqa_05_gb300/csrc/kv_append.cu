// Paged KV append.
//
// "flashlet" README, design bullets: with the pool laid out [pages, page_size,
// kv_heads, head_dim], writing new tokens is one index copy of each token's
// [kv_heads, head_dim] row into its flat slot (page * page_size + offset).
// Each thread moves one 16-byte vector of K and the matching one of V, so a
// warp writes contiguous 512-byte runs of a row; the copy is bit-exact.
#include "common.cuh"

namespace pgqa {

namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(uint4 *__restrict__ k_pool,
                                                        uint4 *__restrict__ v_pool,
                                                        const uint4 *__restrict__ k,
                                                        const uint4 *__restrict__ v,
                                                        const int64_t *__restrict__ slots,
                                                        int64_t num_tokens, int64_t num_slots,
                                                        int row_vecs, unsigned int *flags) {
    pdl_launch_dependents();  // the next grid waits for our completion before reading the pool
    pdl_wait();
    const int64_t n = num_tokens * row_vecs;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / row_vecs;
        const int64_t vec = i - t * row_vecs;
        const int64_t s = __ldg(slots + t);
        if (s < 0) continue;  // padding row
        if (s >= num_slots) {
            if (vec == 0) atomicOr(flags, PGQA_FLAG_SLOT_RANGE);
            continue;
        }
        k_pool[s * row_vecs + vec] = __ldg(k + t * row_vecs + vec);
        v_pool[s * row_vecs + vec] = __ldg(v + t * row_vecs + vec);
    }
}

}  // namespace

cudaError_t launch_kv_append(void *k_pool, void *v_pool, const void *k, const void *v,
                             const int64_t *slot_mapping, int64_t num_tokens, int64_t num_slots,
                             int row_bytes, unsigned int *flags, bool pdl, cudaStream_t stream) {
    const int row_vecs = row_bytes / 16;
    const int64_t n = num_tokens * row_vecs;
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
    return cudaLaunchKernelEx(&cfg, kv_append_kernel, static_cast<uint4 *>(k_pool),
                              static_cast<uint4 *>(v_pool), static_cast<const uint4 *>(k),
                              static_cast<const uint4 *>(v), slot_mapping, num_tokens, num_slots,
                              row_vecs, flags);
}

}  // namespace pgqa
