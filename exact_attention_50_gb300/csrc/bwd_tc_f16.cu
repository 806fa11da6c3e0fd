// bwd_tc_f16.cu -- fp16 instantiations of the tcgen05 backward (bwd_tc.cuh), and the dtype switch.
#include "bwd_tc.cuh"

namespace attn {
cudaError_t launch_bwd_tc_bf16(const BwdMaps& maps, const BwdParams& p, bool causal, cudaStream_t stream);

cudaError_t launch_bwd_tc(const BwdMaps& maps, const BwdParams& p, attn_dtype_t dtype, bool causal,
                          cudaStream_t stream) {
  if (dtype == ATTN_BF16) return launch_bwd_tc_bf16(maps, p, causal, stream);
  return launch_bwd_tc_dtype<__half>(maps, p, causal, stream);
}
}  // namespace attn
