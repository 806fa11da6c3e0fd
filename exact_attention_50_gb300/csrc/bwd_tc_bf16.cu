// bwd_tc_bf16.cu -- bf16 instantiations of the tcgen05 backward (bwd_tc.cuh).
#include "bwd_tc.cuh"

namespace attn {
cudaError_t launch_bwd_tc_bf16(const BwdMaps& maps, const BwdParams& p, bool causal, cudaStream_t stream) {
  return launch_bwd_tc_dtype<__nv_bfloat16>(maps, p, causal, stream);
}
}  // namespace attn
