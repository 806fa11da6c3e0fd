// bwd_aux.cu -- the two bandwidth-bound steps around the backward's main kernel.
//
// preprocess:  D_i = sum_c dO[i,c] * O[i,c] in fp32 (equal to sum_j P_ij dP_ij, the row term
//              of dS_ij = P_ij (dP_ij - D_i)), and, for the tensor-core path, zero the fp32 dQ
//              accumulator that the main kernel reduces into and its per-tile turn counters.
// postprocess: dQ = scale * dQacc, rounded to the output dtype (or kept fp32 on request).
// Both are HBM-bound streams with 16-byte accesses.
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

// Rows are walked in the order of the fp32 statistics (head-major: r = head * N + n); the O and
// dO row of (head, n) is at head * lay.head + n * lay.row.  A row is read by a group of GS lanes
// (16 bytes each; GS the power of two >= d / kVec), a warp covers 32 / GS rows per step and
// each thread issues the loads of kUnroll steps before it reduces any of them, so enough
// bytes are in flight to keep HBM busy.
template <typename T, bool CONTIG, int GS>
__global__ void __launch_bounds__(256) preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                         float* __restrict__ delta, float* __restrict__ dq_acc,
                                                         int* __restrict__ turn, long rows, int N, BwdParams::Rows lay,
                                                         int d) {
  constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
  constexpr int kRowsPerStep = 32 / GS;
  constexpr int kUnroll = 4;
  const int lane = threadIdx.x & 31;
  const int sub = lane / GS, g = lane % GS;  // row within the step, 16-byte vector within the row
  const bool col_ok = g * kVec < d;
  const long warp = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  const long warps = static_cast<long>(gridDim.x) * (blockDim.x / 32);
  constexpr long kRowsPerIter = static_cast<long>(kRowsPerStep) * kUnroll;
  for (long r0 = warp * kRowsPerIter; r0 < rows; r0 += warps * kRowsPerIter) {
    uint4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long r = r0 + u * kRowsPerStep + sub;
      a[u] = make_uint4(0u, 0u, 0u, 0u);
      b[u] = a[u];
      if (r < rows && col_ok) {
        const long long ofs = (CONTIG ? r * d : (r / N) * lay.head + (r % N) * lay.row) + g * kVec;
        a[u] = *reinterpret_cast<const uint4*>(o + ofs);
        b[u] = *reinterpret_cast<const uint4*>(dout + ofs);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const T* av = reinterpret_cast<const T*>(&a[u]);
      const T* bv = reinterpret_cast<const T*>(&b[u]);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kVec; ++i) acc = fmaf(to_f(av[i]), to_f(bv[i]), acc);
#pragma unroll
      for (int off = GS / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const long r = r0 + u * kRowsPerStep + sub;
      if (r < rows) {
        if (g == 0) delta[r] = acc;
        if (dq_acc) {
          if (g == 0) turn[r] = 0;
          float4* z = reinterpret_cast<float4*>(dq_acc + r * d);
          for (int c = g; c < d / 4; c += GS) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
}

template <typename T>
__device__ __forceinline__ void store8(T* dst, const float4& x, const float4& y, float scale);
template <>
__device__ __forceinline__ void store8<float>(float* dst, const float4& x, const float4& y, float scale) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(x.x * scale, x.y * scale, x.z * scale, x.w * scale);
  reinterpret_cast<float4*>(dst)[1] = make_float4(y.x * scale, y.y * scale, y.z * scale, y.w * scale);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const float4& x, const float4& y, float scale) {
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(x.x * scale, x.y * scale);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(x.z * scale, x.w * scale);
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(y.x * scale, y.y * scale);
  const __nv_bfloat162 h3 = __floats2bfloat162_rn(y.z * scale, y.w * scale);
  uint4 v;
  v.x = *reinterpret_cast<const uint32_t*>(&h0);
  v.y = *reinterpret_cast<const uint32_t*>(&h1);
  v.z = *reinterpret_cast<const uint32_t*>(&h2);
  v.w = *reinterpret_cast<const uint32_t*>(&h3);
  *reinterpret_cast<uint4*>(dst) = v;
}
template <>
__device__ __forceinline__ void store8<__half>(__half* dst, const float4& x, const float4& y, float scale) {
  const __half2 h0 = __floats2half2_rn(x.x * scale, x.y * scale);
  const __half2 h1 = __floats2half2_rn(x.z * scale, x.w * scale);
  const __half2 h2 = __floats2half2_rn(y.x * scale, y.y * scale);
  const __half2 h3 = __floats2half2_rn(y.z * scale, y.w * scale);
  uint4 v;
  v.x = *reinterpret_cast<const uint32_t*>(&h0);
  v.y = *reinterpret_cast<const uint32_t*>(&h1);
  v.z = *reinterpret_cast<const uint32_t*>(&h2);
  v.w = *reinterpret_cast<const uint32_t*>(&h3);
  *reinterpret_cast<uint4*>(dst) = v;
}

// The accumulator is in statistics order ([heads * N, d]); row (head, n) of dQ is at
// head * lay.head + n * lay.row.  Each thread converts groups of 8 consecutive values (d is a
// multiple of 16, so a group never straddles rows) with 16-byte stores, kUnroll groups at a
// time.  Every entry point requires dq to be 16-byte aligned, and its row and head strides are
// multiples of d, so every group starts on a 16-byte boundary.
template <typename OutT, bool CONTIG>
__global__ void __launch_bounds__(256) postprocess_vec_kernel(const float* __restrict__ acc, OutT* __restrict__ out,
                                                              long n8, int N, BwdParams::Rows lay, int d, float scale) {
  constexpr int kUnroll = 4;
  const long threads = static_cast<long>(gridDim.x) * blockDim.x;
  const int d8 = d / 8;
  for (long i0 = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n8; i0 += threads * kUnroll) {
    float4 x[kUnroll], y[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long i = i0 + u * threads;
      if (i < n8) {
        x[u] = reinterpret_cast<const float4*>(acc)[2 * i];
        y[u] = reinterpret_cast<const float4*>(acc)[2 * i + 1];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long i = i0 + u * threads;
      if (i < n8) {
        OutT* dst;
        if constexpr (CONTIG) {
          dst = out + 8 * i;
        } else {
          const long r = i / d8;
          dst = out + (r / N) * lay.head + (r % N) * lay.row + 8 * (i % d8);
        }
        store8<OutT>(dst, x[u], y[u], scale);
      }
    }
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

template <typename T, bool CONTIG>
void preprocess_g(const BwdParams& p, float* acc, long rows, int grid, cudaStream_t stream) {
  const T* o = static_cast<const T*>(p.o);
  const T* g = static_cast<const T*>(p.dout);
  const int lanes = p.d / (16 / static_cast<int>(sizeof(T)));  // 16-byte vectors per row: 2 .. 32
  if (lanes <= 4)
    preprocess_kernel<T, CONTIG, 4><<<grid, 256, 0, stream>>>(o, g, p.delta, acc, p.dq_turn, rows, p.N, p.lay_o, p.d);
  else if (lanes <= 8)
    preprocess_kernel<T, CONTIG, 8><<<grid, 256, 0, stream>>>(o, g, p.delta, acc, p.dq_turn, rows, p.N, p.lay_o, p.d);
  else if (sizeof(T) == 2 || lanes <= 16)  // 16-bit rows of d <= 128 take at most 16 vectors
    preprocess_kernel<T, CONTIG, 16><<<grid, 256, 0, stream>>>(o, g, p.delta, acc, p.dq_turn, rows, p.N, p.lay_o, p.d);
  else if constexpr (sizeof(T) == 4)
    preprocess_kernel<T, CONTIG, 32><<<grid, 256, 0, stream>>>(o, g, p.delta, acc, p.dq_turn, rows, p.N, p.lay_o, p.d);
}

template <typename T>
void preprocess_t(const BwdParams& p, float* acc, long rows, int grid, cudaStream_t stream) {
  if (contiguous(p.lay_o, p))
    preprocess_g<T, true>(p, acc, rows, grid, stream);
  else
    preprocess_g<T, false>(p, acc, rows, grid, stream);
}

template <typename OutT>
void postprocess_t(const BwdParams& p, long n4, cudaStream_t stream) {
  OutT* out = static_cast<OutT*>(p.dq);
  const long n8 = n4 / 2;
  const int grid = grid_for(n8, 256 * 4);
  if (contiguous(p.lay_dq, p))
    postprocess_vec_kernel<OutT, true><<<grid, 256, 0, stream>>>(p.dq_acc, out, n8, p.N, p.lay_dq, p.d, p.scale);
  else
    postprocess_vec_kernel<OutT, false><<<grid, 256, 0, stream>>>(p.dq_acc, out, n8, p.N, p.lay_dq, p.d, p.scale);
}
}  // namespace

cudaError_t launch_bwd_preprocess(const BwdParams& p, attn_dtype_t dtype, bool zero_acc, cudaStream_t stream) {
  const long rows = static_cast<long>(p.B) * p.Hq * p.N;
  const int grid = grid_for(rows, 64);
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
  if (p.out_f32)
    postprocess_t<float>(p, n4, stream);
  else if (dtype == ATTN_F16)
    postprocess_t<__half>(p, n4, stream);
  else
    postprocess_t<__nv_bfloat16>(p, n4, stream);
  return cudaGetLastError();
}

}  // namespace attn
