// bwd_aux.cu -- the two bandwidth-bound steps around the backward's main kernel.
//
// preprocess:  D_i = sum_c dO[i,c] * O[i,c] in fp32 (equal to sum_j P_ij dP_ij, the row term
//              of dS_ij = P_ij (dP_ij - D_i)), and, for the tensor-core path, zero the fp32 dQ
//              accumulator that the main kernel reduces into.
// postprocess: dQ = scale * dQacc, rounded to the output dtype (or kept fp32 on request).
// One warp per row with 16-byte loads; both are HBM-bound streams.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "kernels.h"

namespace attn {
namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T>
__global__ void __launch_bounds__(256) preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                         float* __restrict__ delta, float* __restrict__ dq_acc,
                                                         long rows, int d) {
  constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
  const long warps = static_cast<long>(gridDim.x) * (blockDim.x / 32);
  const int lane = threadIdx.x & 31;
  for (long r = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; r < rows; r += warps) {
    const T* orow = o + r * d;
    const T* grow = dout + r * d;
    float acc = 0.f;
    for (int c = lane * kVec; c < d; c += 32 * kVec) {
      const uint4 a = *reinterpret_cast<const uint4*>(orow + c);
      const uint4 b = *reinterpret_cast<const uint4*>(grow + c);
      const T* av = reinterpret_cast<const T*>(&a);
      const T* bv = reinterpret_cast<const T*>(&b);
#pragma unroll
      for (int i = 0; i < kVec; ++i) acc = fmaf(to_f(av[i]), to_f(bv[i]), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) delta[r] = acc;
    if (dq_acc) {
      float4* z = reinterpret_cast<float4*>(dq_acc + r * d);
      for (int c = lane; c < d / 4; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

template <typename T, typename OutT>
__global__ void __launch_bounds__(256) postprocess_kernel(const float* __restrict__ acc, OutT* __restrict__ out,
                                                          long n4, float scale) {
  const long stride = static_cast<long>(gridDim.x) * blockDim.x;
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[i];
    OutT* dst = out + 4 * i;
    dst[0] = from_f<OutT>(a.x * scale);
    dst[1] = from_f<OutT>(a.y * scale);
    dst[2] = from_f<OutT>(a.z * scale);
    dst[3] = from_f<OutT>(a.w * scale);
  }
}

int grid_for(long work, int per_block) {
  long g = (work + per_block - 1) / per_block;
  const long cap = 152L * 16;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdParams& p, attn_dtype_t dtype, bool zero_acc, cudaStream_t stream) {
  const long rows = static_cast<long>(p.B) * p.Hq * p.N;
  const int grid = grid_for(rows, 8);
  float* acc = zero_acc ? p.dq_acc : nullptr;
  switch (dtype) {
    case ATTN_F32:
      preprocess_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(p.o),
                                                         static_cast<const float*>(p.dout), p.delta, acc, rows, p.d);
      break;
    case ATTN_F16:
      preprocess_kernel<__half><<<grid, 256, 0, stream>>>(static_cast<const __half*>(p.o),
                                                          static_cast<const __half*>(p.dout), p.delta, acc, rows, p.d);
      break;
    default:
      preprocess_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(p.o),
                                                                 static_cast<const __nv_bfloat16*>(p.dout), p.delta,
                                                                 acc, rows, p.d);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_postprocess(const BwdParams& p, attn_dtype_t dtype, cudaStream_t stream) {
  const long n4 = static_cast<long>(p.B) * p.Hq * p.N * p.d / 4;
  const int grid = grid_for(n4, 256);
  if (p.out_f32)
    postprocess_kernel<float, float><<<grid, 256, 0, stream>>>(p.dq_acc, static_cast<float*>(p.dq), n4, p.scale);
  else if (dtype == ATTN_F16)
    postprocess_kernel<__half, __half><<<grid, 256, 0, stream>>>(p.dq_acc, static_cast<__half*>(p.dq), n4, p.scale);
  else
    postprocess_kernel<__nv_bfloat16, __nv_bfloat16>
        <<<grid, 256, 0, stream>>>(p.dq_acc, static_cast<__nv_bfloat16*>(p.dq), n4, p.scale);
  return cudaGetLastError();
}

}  // namespace attn
