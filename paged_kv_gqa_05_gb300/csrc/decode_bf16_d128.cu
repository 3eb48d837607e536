// Split-KV decode partial kernel instantiated for bf16, head_dim 128, groups 1..8.
#include "decode.cuh"

namespace pgqa {
cudaError_t launch_decode_bf16_d128(int group, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                      const DecodeParams &p, int num_items, bool pdl,
                                      cudaStream_t stream) {
    return launch_decode_dt<128, __nv_bfloat16>(group, tm_k, tm_v, p, num_items, pdl, stream);
}
}  // namespace pgqa
