// fwd_tc_f16.cu -- fp16 instantiations of the tcgen05 forward (fwd_tc.cuh), and the dtype switch.
#include "fwd_tc.cuh"

namespace attn {
cudaError_t launch_fwd_tc_bf16(const FwdMaps& maps, const FwdParams& p, bool causal, int mode,
                               cudaStream_t stream);

cudaError_t launch_fwd_tc(const FwdMaps& maps, const FwdParams& p, attn_dtype_t dtype, bool causal, int mode,
                          cudaStream_t stream) {
  if (dtype == ATTN_BF16) return launch_fwd_tc_bf16(maps, p, causal, mode, stream);
  return launch_fwd_tc_dtype<__half>(maps, p, causal, mode, stream);
}
}  // namespace attn
