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

// Rows are walked in the order of the fp32 statistics (head-major: r = head * N + n); the O and
// dO row of (head, n) is at head * lay.head + n * lay.row.
template <typename T, bool CONTIG>
__global__ void __launch_bounds__(256) preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                         float* __restrict__ delta, float* __restrict__ dq_acc,
                                                         long rows, int N, BwdParams::Rows lay, int d) {
  constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
  const long warps = static_cast<long>(gridDim.x) * (blockDim.x / 32);
  const int lane = threadIdx.x & 31;
  for (long r = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; r < rows; r += warps) {
    const long long ofs = CONTIG ? r * d : (r / N) * lay.head + (r % N) * lay.row;
    const T* orow = o + ofs;
    const T* grow = dout + ofs;
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

// The accumulator is in statistics order ([heads * N, d]); row (head, n) of dQ is at
// head * lay.head + n * lay.row.
template <typename OutT, bool CONTIG>
__global__ void __launch_bounds__(256) postprocess_kernel(const float* __restrict__ acc, OutT* __restrict__ out,
                                                          long n4, int N, BwdParams::Rows lay, int d, float scale) {
  const long stride = static_cast<long>(gridDim.x) * blockDim.x;
  const int d4 = d / 4;
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[i];
    OutT* dst;
    if constexpr (CONTIG) {
      dst = out + 4 * i;
    } else {
      const long r = i / d4;
      dst = out + (r / N) * lay.head + (r % N) * lay.row + 4 * (i % d4);
    }
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

namespace {
bool contiguous(const BwdParams::Rows& lay, const BwdParams& p) {
  return lay.row == p.d && lay.head == static_cast<long long>(p.N) * p.d;
}

template <typename T>
void preprocess_t(const BwdParams& p, float* acc, long rows, int grid, cudaStream_t stream) {
  const T* o = static_cast<const T*>(p.o);
  const T* g = static_cast<const T*>(p.dout);
  if (contiguous(p.lay_o, p))
    preprocess_kernel<T, true><<<grid, 256, 0, stream>>>(o, g, p.delta, acc, rows, p.N, p.lay_o, p.d);
  else
    preprocess_kernel<T, false><<<grid, 256, 0, stream>>>(o, g, p.delta, acc, rows, p.N, p.lay_o, p.d);
}

template <typename OutT>
void postprocess_t(const BwdParams& p, long n4, int grid, cudaStream_t stream) {
  OutT* out = static_cast<OutT*>(p.dq);
  if (contiguous(p.lay_dq, p))
    postprocess_kernel<OutT, true><<<grid, 256, 0, stream>>>(p.dq_acc, out, n4, p.N, p.lay_dq, p.d, p.scale);
  else
    postprocess_kernel<OutT, false><<<grid, 256, 0, stream>>>(p.dq_acc, out, n4, p.N, p.lay_dq, p.d, p.scale);
}
}  // namespace

cudaError_t launch_bwd_preprocess(const BwdParams& p, attn_dtype_t dtype, bool zero_acc, cudaStream_t stream) {
  const long rows = static_cast<long>(p.B) * p.Hq * p.N;
  const int grid = grid_for(rows, 8);
  float* acc = zero_acc ? p.dq_acc : nullptr;
  switch (dtype) {
    case ATTN_F32: preprocess_t<float>(p, acc, rows, grid, stream); break;
    case ATTN_F16: preprocess_t<__half>(p, acc, rows, grid, stream); break;
    default: preprocess_t<__nv_bfloat16>(p, acc, rows, grid, stream); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_postprocess(const BwdParams& p, attn_dtype_t dtype, cudaStream_t stream) {
  const long n4 = static_cast<long>(p.B) * p.Hq * p.N * p.d / 4;
  const int grid = grid_for(n4, 256);
  if (p.out_f32)
    postprocess_t<float>(p, n4, grid, stream);
  else if (dtype == ATTN_F16)
    postprocess_t<__half>(p, n4, grid, stream);
  else
    postprocess_t<__nv_bfloat16>(p, n4, grid, stream);
  return cudaGetLastError();
}

}  // namespace attn
