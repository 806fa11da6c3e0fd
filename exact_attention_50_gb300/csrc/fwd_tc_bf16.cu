// fwd_tc_bf16.cu -- bf16 instantiations of the tcgen05 forward (fwd_tc.cuh).
#include "fwd_tc.cuh"

namespace attn {
cudaError_t launch_fwd_tc_bf16(const FwdMaps& maps, const FwdParams& p, bool causal, int mode,
                               cudaStream_t stream) {
  return launch_fwd_tc_dtype<__nv_bfloat16>(maps, p, causal, mode, stream);
}
}  // namespace attn
