// kv_combine.cu -- merges the split-KV partial results of the KV-cache / cross-attention forward.
//
// Range s of a row's keys produced O_s (normalised over the range's keys) and LSE_s (natural
// log of the range's softmax denominator, -inf when the row sees none of them).  The softmax
// over the union of the ranges is the LSE-weighted mix of the parts:
//   LSE = log sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s,
// evaluated with the largest LSE_s subtracted first.  A row with no visible key at all gets
// O = 0 and LSE = -inf.  (The blocked KV-cache computation at inference of the FlashAttention-T
// review, FAQ 4; the merge is the same online-softmax rescaling as across key tiles, its best
// practice 4.)
//
// One warp per output row; lane l owns columns 4l .. 4l+3 (d <= 128), and the loads of eight
// ranges are issued before any is used (the ranges' parts sit far apart).  Which ranges hold data
// follows from the forward's work split (kv_needed_keys): a range past the block's last
// visible key was never computed and is not read.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

template <typename T>
__device__ __forceinline__ void store4(T* dst, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float a, float b, float c, float d) {
  const __nv_bfloat162 x = __floats2bfloat162_rn(a, b), y = __floats2bfloat162_rn(c, d);
  uint2 v;
  v.x = *reinterpret_cast<const uint32_t*>(&x);
  v.y = *reinterpret_cast<const uint32_t*>(&y);
  *reinterpret_cast<uint2*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<__half>(__half* dst, float a, float b, float c, float d) {
  const __half2 x = __floats2half2_rn(a, b), y = __floats2half2_rn(c, d);
  uint2 v;
  v.x = *reinterpret_cast<const uint32_t*>(&x);
  v.y = *reinterpret_cast<const uint32_t*>(&y);
  *reinterpret_cast<uint2*>(dst) = v;
}

template <typename OutT, bool CAUSAL>
__global__ void __launch_bounds__(256) kv_combine_kernel(const FwdParams p) {
  const long rows = static_cast<long>(p.B) * p.Hkv * p.R;
  const long warps = static_cast<long>(gridDim.x) * (blockDim.x / 32);
  const int lane = threadIdx.x & 31;
  const bool col_ok = lane * 4 < p.d;
  for (long r = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; r < rows; r += warps) {
    const long bh = r / p.R;
    const int rr = static_cast<int>(r % p.R);
    const int b = static_cast<int>(bh / p.Hkv);
    int L = p.Nk;
    if (p.cache_seqlens) {
      L = p.cache_seqlens[b];
      if (L < 0 || L > p.Nk) {
        if (lane == 0 && rr == 0) raise_status(p.status, ATTN_ERR_DEVICE_INPUT);
        L = 0;
      }
    }
    const int need_tiles = (kv_needed_keys(L, p.Nq, p.R, rr / 128, CAUSAL) + 127) / 128;
    const int nv = min(p.n_splits, (need_tiles + p.tiles_per_split - 1) / p.tiles_per_split);
    // the largest range LSE: lanes over the ranges, then a warp reduction
    float mx = -INFINITY;
    for (int s = lane; s < nv; s += 32) mx = fmaxf(mx, p.lse_part[s * rows + r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // weighted sum of the range outputs, eight ranges' loads in flight at a time
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f, wsum = 0.f;
    if (mx != -INFINITY) {
      for (int s0 = 0; s0 < nv; s0 += 8) {
        float ls[8];
        float4 os[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int s = s0 + u;
          ls[u] = s < nv ? p.lse_part[s * rows + r] : -INFINITY;
          os[u] = (s < nv && col_ok) ? *reinterpret_cast<const float4*>(p.o_part + (s * rows + r) * p.d + lane * 4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float w = expf(ls[u] - mx);  // 0 for ranges past nv and for rows empty in a range
          wsum += w;
          a0 = fmaf(w, os[u].x, a0);
          a1 = fmaf(w, os[u].y, a1);
          a2 = fmaf(w, os[u].z, a2);
          a3 = fmaf(w, os[u].w, a3);
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (col_ok) store4<OutT>(static_cast<OutT*>(p.o) + r * p.d + lane * 4, a0 * inv, a1 * inv, a2 * inv, a3 * inv);
    if (lane == 0 && p.lse) p.lse[r] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
  }
}

template <typename OutT>
cudaError_t run(const FwdParams& p, bool causal, cudaStream_t stream) {
  const long rows = static_cast<long>(p.B) * p.Hkv * p.R;
  long blocks = (rows + 7) / 8;
  if (blocks > 152L * 16) blocks = 152L * 16;
  if (blocks < 1) blocks = 1;
  if (causal)
    kv_combine_kernel<OutT, true><<<static_cast<int>(blocks), 256, 0, stream>>>(p);
  else
    kv_combine_kernel<OutT, false><<<static_cast<int>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_combine(const FwdParams& p, attn_dtype_t dtype, bool causal, cudaStream_t stream) {
  if (dtype == ATTN_F32 || p.out_f32) return run<float>(p, causal, stream);
  if (dtype == ATTN_F16) return run<__half>(p, causal, stream);
  return run<__nv_bfloat16>(p, causal, stream);
}

}  // namespace attn
