// Split-KV decode partial kernels instantiated for bf16, head_dim 128: the
// tensor-core kernel (any group width up to 16; one CTA per work item: 2- or
// 3-stage rings, or the wide form), the CUDA-core kernel (groups 1..8) and
// the prefill-segment kernels (tcgen05, and the mma.sync form).
#include "decode_simt.cuh"
#include "decode_tc.cuh"
#include "prefill_t5.cuh"
#include "prefill_tc.cuh"

namespace pgqa {
cudaError_t launch_decode_bf16_d128(int kind, int stages, int group, const CUtensorMap &tm_k,
                                      const CUtensorMap &tm_v, const DecodeParams &p, int num_items,
                                      bool pdl, cudaStream_t stream) {
    if (kind == PGQA_DECODE_CUDA_CORE)
        return launch_decode_dt<128, __nv_bfloat16>(group, tm_k, tm_v, p, num_items, pdl, stream);
    return launch_decode_tc<128, __nv_bfloat16>(stages, group, tm_k, tm_v, p, num_items, pdl, stream);
}

cudaError_t decode_blocks_per_sm_bf16_d128(int stages, int group, int *blocks) {
    return decode_tc_blocks_per_sm<128, __nv_bfloat16>(stages, group, blocks);
}

cudaError_t launch_prefill_bf16_d128(int kind, int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                      const PrefillParams &p, int num_items, bool pdl, cudaStream_t stream) {
    if (kind == PGQA_PREFILL_MMA_SYNC) return launch_prefill_tc<128, __nv_bfloat16>(group, tm_k, tm_v, p, num_items, pdl, stream);
    return launch_prefill_t5<128, __nv_bfloat16>(group, tm_k, tm_v, p, num_items, pdl, stream);
}
}  // namespace pgqa
