// fwd_short.cu -- instantiations of the short-sequence forward (fwd_short.cuh).
#include "fwd_short.cuh"

namespace attn {

template <typename T>
cudaError_t launch_fwd_short_dtype(const FwdMaps& maps, const ShortParams& p, bool causal, cudaStream_t stream) {
  if (p.d <= 64)
    return causal ? launch_fwd_short_t<T, 64, true>(maps, p, stream) : launch_fwd_short_t<T, 64, false>(maps, p, stream);
  return causal ? launch_fwd_short_t<T, 128, true>(maps, p, stream) : launch_fwd_short_t<T, 128, false>(maps, p, stream);
}

cudaError_t launch_fwd_short(const FwdMaps& maps, const ShortParams& p, attn_dtype_t dtype, bool causal,
                             cudaStream_t stream) {
  return dtype == ATTN_BF16 ? launch_fwd_short_dtype<__nv_bfloat16>(maps, p, causal, stream)
                            : launch_fwd_short_dtype<__half>(maps, p, causal, stream);
}

}  // namespace attn
