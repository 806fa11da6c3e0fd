// simt_f32.cu -- float32 attention on the CUDA cores (FFMA), forward and backward.
//
// Same tiled, online-softmax algorithm as the tensor-core path (attention-operator article
// section 2.2; FlashAttention-T review best practice 4), with every operand and accumulator
// in fp32 so the result stays within 1e-5 of the exact value.
//
// Forward: a CTA of 4 warps owns 32 query rows (8 per warp); K/V stream through shared memory
// in tiles of 32 keys.  Lane l of a warp computes the scores of its 8 rows against key l, the
// row max / sum are warp reductions, and lane l accumulates output columns l, l+32, ...
// Backward: two passes with no atomics.  The dQ kernel owns query rows and walks the keys; the
// dK/dV kernel owns key rows and walks the query rows of every head of the kv head's group,
// so each output element is written by exactly one thread.  P_ij = exp(S_ij - LSE_i) is
// recomputed from the forward's LSE (FlashAttention-T review FAQ 4).
#include <cmath>
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kRows = 32;     // rows per CTA
constexpr int kTile = 32;     // keys (or queries) per shared-memory tile
constexpr int kMaxD = 128;
constexpr int kColsPerLane = kMaxD / 32;
constexpr float kLog2e = 1.4426950408889634f;

// Row addressing shared by the dense [B,H,N,d] and packed varlen [T,3,H,d] layouts.
struct RowAddr {
  size_t base;     // element offset of row 0
  size_t stride;   // elements between consecutive rows
};

__device__ __forceinline__ void warp_max_sum(float& v, bool is_max) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
}

// ------------------------------------------------------------------ forward
template <bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(128) fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                                      const float* __restrict__ v, const FwdParams p) {
  extern __shared__ float smem_f[];
  const int dp1 = p.d + 1;
  float* sK = smem_f;                  // [kTile][d+1]
  float* sV = sK + kTile * dp1;        // [kTile][d]
  float* sQ = sV + kTile * p.d;        // [kRows][d]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int b = 0, h, seq_start = 0, seq_len;
  const int qt = blockIdx.y;
  if constexpr (VARLEN) {
    h = blockIdx.x;
    const int s = blockIdx.z;
    const int c0 = p.cu_seqlens[s], c1 = p.cu_seqlens[s + 1];
    const bool bad = c0 < 0 || c1 < c0 || c1 > p.total_tokens || c1 - c0 > p.max_seqlen ||
                     (s == 0 && c0 != 0) || (s == p.nseq - 1 && c1 != p.total_tokens);
    if (bad) {
      if (threadIdx.x == 0) raise_status(p.status, ATTN_ERR_DEVICE_INPUT);
      return;
    }
    seq_start = c0;
    seq_len = c1 - c0;
    if (qt * kRows >= seq_len) return;
  } else {
    b = blockIdx.x / p.Hq;
    h = blockIdx.x % p.Hq;
    seq_len = p.N;
  }
  const int d = p.d, g = h / p.G;
  RowAddr qa, ka, va;
  if constexpr (VARLEN) {
    // q, k and v already point at planes 0, 1 and 2 of the packed [T,3,H,d] tensor
    const size_t tok = 3ull * p.Hq * d;
    qa = {static_cast<size_t>(seq_start) * tok + static_cast<size_t>(h) * d, tok};
    ka = qa;
    va = qa;
  } else {
    qa = {(static_cast<size_t>(b) * p.Hq + h) * p.N * d, static_cast<size_t>(d)};
    ka = {(static_cast<size_t>(b) * p.Hkv + g) * p.N * d, static_cast<size_t>(d)};
    va = ka;
  }
  const int row0 = qt * kRows;
  for (int idx = threadIdx.x; idx < kRows * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    sQ[r * d + c] = (row0 + r < seq_len) ? q[qa.base + (row0 + r) * qa.stride + c] : 0.f;
  }
  float m[8], l[8], acc[8][kColsPerLane];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int i = 0; i < kColsPerLane; ++i) acc[r][i] = 0.f;
  }
  const float sl2 = p.scale_log2;
  const int row_hi = min(seq_len, row0 + kRows) - 1;
  const int n_keys = CAUSAL ? min(seq_len, row_hi + 1) : seq_len;
  for (int key0 = 0; key0 < n_keys; key0 += kTile) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTile * d; idx += blockDim.x) {
      const int r = idx / d, c = idx % d;
      const bool in = key0 + r < seq_len;
      sK[r * dp1 + c] = in ? k[ka.base + (key0 + r) * ka.stride + c] : 0.f;
      sV[r * d + c] = in ? v[va.base + (key0 + r) * va.stride + c] : 0.f;
    }
    __syncthreads();
    const int key = key0 + lane;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int lr = warp * 8 + r, qrow = row0 + lr;
      float s = 0.f;
      for (int c = 0; c < d; ++c) s = fmaf(sQ[lr * d + c], sK[lane * dp1 + c], s);
      const bool masked = key >= seq_len || (CAUSAL && key > qrow);
      float x = masked ? -INFINITY : s * sl2;
      float mx = x;
      warp_max_sum(mx, true);
      const float m_new = fmaxf(m[r], mx);
      const float mb = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m[r] - mb);
      const float pr = exp2f(x - mb);
      float rs = pr;
      warp_max_sum(rs, false);
      l[r] = l[r] * alpha + rs;
      m[r] = m_new;
#pragma unroll
      for (int i = 0; i < kColsPerLane; ++i) acc[r][i] *= alpha;
      for (int jj = 0; jj < kTile; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, pr, jj);
#pragma unroll
        for (int i = 0; i < kColsPerLane; ++i) {
          const int c = lane + 32 * i;
          if (c < d) acc[r][i] = fmaf(pj, sV[jj * d + c], acc[r][i]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int qrow = row0 + warp * 8 + r;
    if (qrow >= seq_len) continue;
    const float inv_l = 1.f / l[r];
    size_t out_off;
    if constexpr (VARLEN)
      out_off = (static_cast<size_t>(seq_start + qrow) * p.Hq + h) * d;
    else
      out_off = ((static_cast<size_t>(b) * p.Hq + h) * p.N + qrow) * d;
    float* o = static_cast<float*>(p.o);
#pragma unroll
    for (int i = 0; i < kColsPerLane; ++i) {
      const int c = lane + 32 * i;
      if (c < d) o[out_off + c] = acc[r][i] * inv_l;
    }
    if (lane == 0 && p.lse) {
      const float lse = (m[r] + log2f(l[r])) / kLog2e;
      if constexpr (VARLEN)
        p.lse[static_cast<size_t>(h) * p.total_tokens + seq_start + qrow] = lse;
      else
        p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.N + qrow] = lse;
    }
  }
}

// KV cache / cross-attention forward in fp32: CTA (batch * query head, 32-row query tile,
// key range).  Query i of batch b sees the cache keys j < L = cache_seqlens[b] (Nk when
// absent) and, when causal, only j <= L - Nq + i.  Range s covers the keys
// [s * tiles_per_split * 128, (s + 1) * tiles_per_split * 128); every range writes its
// normalised partial output and LSE (O = 0, LSE = -inf for a row that sees none of its keys),
// which the split combine merges.
template <bool CAUSAL>
__global__ void __launch_bounds__(128) fwd_f32_kv_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                                         const float* __restrict__ v, const FwdParams p) {
  extern __shared__ float smem_f[];
  const int dp1 = p.d + 1;
  float* sK = smem_f;                  // [kTile][d+1]
  float* sV = sK + kTile * dp1;        // [kTile][d]
  float* sQ = sV + kTile * p.d;        // [kRows][d]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x / p.Hq, h = blockIdx.x % p.Hq, g = h / p.G;
  const int qt = blockIdx.y, split = blockIdx.z;
  const int d = p.d, Nq = p.Nq;
  int L = p.Nk;
  if (p.cache_seqlens) {
    L = p.cache_seqlens[b];
    if (L < 0 || L > p.Nk) {
      if (threadIdx.x == 0 && h == 0 && qt == 0 && split == 0) raise_status(p.status, ATTN_ERR_DEVICE_INPUT);
      L = 0;
    }
  }
  const size_t qbase = (static_cast<size_t>(b) * p.Hq + h) * Nq * d;
  const size_t kbase = (static_cast<size_t>(b) * p.Hkv + g) * p.Nk * d;
  const int row0 = qt * kRows;
  for (int idx = threadIdx.x; idx < kRows * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    sQ[r * d + c] = (row0 + r < Nq) ? q[qbase + static_cast<size_t>(row0 + r) * d + c] : 0.f;
  }
  float m[8], l[8], acc[8][kColsPerLane];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int i = 0; i < kColsPerLane; ++i) acc[r][i] = 0.f;
  }
  const float sl2 = p.scale_log2;
  const long span = static_cast<long>(p.tiles_per_split) * 128;
  const int k_begin = static_cast<int>(min(static_cast<long>(L), split * span));
  const int k_end = static_cast<int>(min(static_cast<long>(L), (split + 1) * span));
  for (int key0 = k_begin; key0 < k_end; key0 += kTile) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTile * d; idx += blockDim.x) {
      const int r = idx / d, c = idx % d;
      const bool in = key0 + r < k_end;
      sK[r * dp1 + c] = in ? k[kbase + static_cast<size_t>(key0 + r) * d + c] : 0.f;
      sV[r * d + c] = in ? v[kbase + static_cast<size_t>(key0 + r) * d + c] : 0.f;
    }
    __syncthreads();
    const int key = key0 + lane;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int lr = warp * 8 + r, qrow = row0 + lr;
      float s = 0.f;
      for (int c = 0; c < d; ++c) s = fmaf(sQ[lr * d + c], sK[lane * dp1 + c], s);
      const bool masked = key >= k_end || (CAUSAL && key > L - Nq + qrow);
      float x = masked ? -INFINITY : s * sl2;
      float mx = x;
      warp_max_sum(mx, true);
      const float m_new = fmaxf(m[r], mx);
      const float mb = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m[r] - mb);
      const float pr = exp2f(x - mb);
      float rs = pr;
      warp_max_sum(rs, false);
      l[r] = l[r] * alpha + rs;
      m[r] = m_new;
#pragma unroll
      for (int i = 0; i < kColsPerLane; ++i) acc[r][i] *= alpha;
      for (int jj = 0; jj < kTile; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, pr, jj);
#pragma unroll
        for (int i = 0; i < kColsPerLane; ++i) {
          const int c = lane + 32 * i;
          if (c < d) acc[r][i] = fmaf(pj, sV[jj * d + c], acc[r][i]);
        }
      }
    }
  }
  const size_t rows = static_cast<size_t>(p.B) * p.Hq * Nq;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int qrow = row0 + warp * 8 + r;
    if (qrow >= Nq) continue;
    const size_t orow = static_cast<size_t>(split) * rows + (static_cast<size_t>(b) * p.Hq + h) * Nq + qrow;
    const float inv_l = l[r] > 0.f ? 1.f / l[r] : 0.f;
#pragma unroll
    for (int i = 0; i < kColsPerLane; ++i) {
      const int c = lane + 32 * i;
      if (c < d) p.o_part[orow * d + c] = acc[r][i] * inv_l;
    }
    if (lane == 0) p.lse_part[orow] = l[r] > 0.f ? (m[r] + log2f(l[r])) / kLog2e : -INFINITY;
  }
}

// Which (kv head, sequence) block x of the backward grid covers: dense x = batch * kv head
// (the whole sequence), varlen x = sequence * head (a diagonal block of a B = 1 problem).
struct BwdBlock {
  int hq0, hkv, seq_start, L, Lk;  // first query head, kv head, sequence start, query and key counts
  bool ok;
};
__device__ __forceinline__ BwdBlock bwd_block(const BwdParams& p, int x) {
  BwdBlock r{0, 0, 0, p.N, p.Nk, true};
  if (p.cu_seqlens) {
    const int s = x / p.Hkv, hh = x % p.Hkv;
    const int c0 = p.cu_seqlens[s], c1 = p.cu_seqlens[s + 1];
    if (c0 < 0 || c1 < c0 || c1 > p.N || c1 - c0 > p.max_seqlen || (s == 0 && c0 != 0) ||
        (s == p.nseq - 1 && c1 != p.N)) {
      if (threadIdx.x == 0 && blockIdx.y == 0 && hh == 0) raise_status(p.status, ATTN_ERR_DEVICE_INPUT);
      r.ok = false;
      return r;
    }
    r.seq_start = c0;
    r.L = c1 - c0;
    r.Lk = r.L;
    r.hkv = hh;
    r.hq0 = hh * p.G;
  } else {
    const int b = x / p.Hkv, g = x % p.Hkv;
    r.hkv = b * p.Hkv + g;
    r.hq0 = b * p.Hq + g * p.G;
  }
  return r;
}

// ------------------------------------------------------------------ backward: dQ
template <bool CAUSAL>
__global__ void __launch_bounds__(128) bwd_dq_f32_kernel(const BwdParams p) {
  extern __shared__ float smem_f[];
  const int dp1 = p.d + 1;
  float* sK = smem_f;                  // [kTile][d+1]
  float* sV = sK + kTile * dp1;        // [kTile][d+1]
  float* sQ = sV + kTile * dp1;        // [kRows][d]
  float* sdO = sQ + kRows * p.d;       // [kRows][d]
  const float* q = static_cast<const float*>(p.q);
  const float* k = static_cast<const float*>(p.k);
  const float* v = static_cast<const float*>(p.v);
  const float* dout = static_cast<const float*>(p.dout);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // blockIdx.x = (kv block) * G + query head within the group
  const BwdBlock bb = bwd_block(p, blockIdx.x / p.G);
  if (!bb.ok) return;
  // query i sees key j iff j <= i + off under the causal mask (off = Nk - N: the queries are
  // aligned with the last keys; 0 for self-attention)
  const int hq = bb.hq0 + blockIdx.x % p.G, d = p.d, N = bb.L, Nk = bb.Lk, off = Nk - N, s0 = bb.seq_start;
  const int row0 = blockIdx.y * kRows;
  if (row0 >= N) return;  // past this sequence's end (varlen)
  const size_t qbase = static_cast<size_t>(hq) * p.N + s0;  // row statistics of this head
  const float* qh = q + hq * p.lay_q.head + s0 * p.lay_q.row;
  const float* doh = dout + hq * p.lay_o.head + s0 * p.lay_o.row;
  const float* kh = k + bb.hkv * p.lay_kv.head + s0 * p.lay_kv.row;
  const float* vh = v + bb.hkv * p.lay_kv.head + s0 * p.lay_kv.row;
  for (int idx = threadIdx.x; idx < kRows * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    const bool in = row0 + r < N;
    sQ[r * d + c] = in ? qh[(row0 + r) * p.lay_q.row + c] : 0.f;
    sdO[r * d + c] = in ? doh[(row0 + r) * p.lay_o.row + c] : 0.f;
  }
  float lse2[8], Dr[8], acc[8][kColsPerLane];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int qrow = row0 + warp * 8 + r;
    lse2[r] = qrow < N ? p.lse[qbase + qrow] * kLog2e : 0.f;
    Dr[r] = qrow < N ? p.delta[qbase + qrow] : 0.f;
#pragma unroll
    for (int i = 0; i < kColsPerLane; ++i) acc[r][i] = 0.f;
  }
  const int n_keys = CAUSAL ? max(0, min(Nk, row0 + kRows + off)) : Nk;
  for (int key0 = 0; key0 < n_keys; key0 += kTile) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTile * d; idx += blockDim.x) {
      const int r = idx / d, c = idx % d;
      const bool in = key0 + r < Nk;
      sK[r * dp1 + c] = in ? kh[(key0 + r) * p.lay_kv.row + c] : 0.f;
      sV[r * dp1 + c] = in ? vh[(key0 + r) * p.lay_kv.row + c] : 0.f;
    }
    __syncthreads();
    const int key = key0 + lane;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int lr = warp * 8 + r, qrow = row0 + lr;
      float s = 0.f, dp = 0.f;
      for (int c = 0; c < d; ++c) {
        s = fmaf(sQ[lr * d + c], sK[lane * dp1 + c], s);
        dp = fmaf(sdO[lr * d + c], sV[lane * dp1 + c], dp);
      }
      const bool masked = qrow >= N || key >= Nk || (CAUSAL && key > qrow + off);
      const float pr = masked ? 0.f : exp2f(s * p.scale_log2 - lse2[r]);
      const float ds = pr * (dp - Dr[r]);
      for (int jj = 0; jj < kTile; ++jj) {
        const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
        for (int i = 0; i < kColsPerLane; ++i) {
          const int c = lane + 32 * i;
          if (c < d) acc[r][i] = fmaf(dsj, sK[jj * dp1 + c], acc[r][i]);
        }
      }
    }
  }
  float* dq = static_cast<float*>(p.dq) + hq * p.lay_dq.head + s0 * p.lay_dq.row;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int qrow = row0 + warp * 8 + r;
    if (qrow >= N) continue;
#pragma unroll
    for (int i = 0; i < kColsPerLane; ++i) {
      const int c = lane + 32 * i;
      if (c < d) dq[qrow * p.lay_dq.row + c] = acc[r][i] * p.scale;
    }
  }
}

// ------------------------------------------------------------------ backward: dK, dV
template <bool CAUSAL>
__global__ void __launch_bounds__(128) bwd_dkdv_f32_kernel(const BwdParams p) {
  extern __shared__ float smem_f[];
  const int dp1 = p.d + 1;
  float* sQ = smem_f;                  // [kTile][d+1]
  float* sdO = sQ + kTile * dp1;       // [kTile][d+1]
  float* sK = sdO + kTile * dp1;       // [kRows][d]
  float* sV = sK + kRows * p.d;        // [kRows][d]
  float* sLse = sV + kRows * p.d;      // [kTile]
  float* sD = sLse + kTile;            // [kTile]
  const float* q = static_cast<const float*>(p.q);
  const float* k = static_cast<const float*>(p.k);
  const float* v = static_cast<const float*>(p.v);
  const float* dout = static_cast<const float*>(p.dout);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BwdBlock bb = bwd_block(p, blockIdx.x);
  if (!bb.ok) return;
  const int d = p.d, N = bb.L, Nk = bb.Lk, off = Nk - N, s0 = bb.seq_start;
  const int key0 = blockIdx.y * kRows;
  if (key0 >= Nk) return;  // past this sequence's end (varlen)
  const float* kh = k + bb.hkv * p.lay_kv.head + s0 * p.lay_kv.row;
  const float* vh = v + bb.hkv * p.lay_kv.head + s0 * p.lay_kv.row;
  for (int idx = threadIdx.x; idx < kRows * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    const bool in = key0 + r < Nk;
    sK[r * d + c] = in ? kh[(key0 + r) * p.lay_kv.row + c] : 0.f;
    sV[r * d + c] = in ? vh[(key0 + r) * p.lay_kv.row + c] : 0.f;
  }
  float dk[8][kColsPerLane], dv[8][kColsPerLane];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int i = 0; i < kColsPerLane; ++i) dk[r][i] = dv[r][i] = 0.f;
  for (int hh = 0; hh < p.G; ++hh) {
    const int hq = bb.hq0 + hh;
    const size_t qbase = static_cast<size_t>(hq) * p.N + s0;  // row statistics of this head
    const float* qh = q + hq * p.lay_q.head + s0 * p.lay_q.row;
    const float* doh = dout + hq * p.lay_o.head + s0 * p.lay_o.row;
    // causal: the first query that sees key key0 is key0 - off
    for (int qrow0 = CAUSAL ? (max(0, key0 - off) / kTile) * kTile : 0; qrow0 < N; qrow0 += kTile) {
      __syncthreads();
      for (int idx = threadIdx.x; idx < kTile * d; idx += blockDim.x) {
        const int r = idx / d, c = idx % d;
        const bool in = qrow0 + r < N;
        sQ[r * dp1 + c] = in ? qh[(qrow0 + r) * p.lay_q.row + c] : 0.f;
        sdO[r * dp1 + c] = in ? doh[(qrow0 + r) * p.lay_o.row + c] : 0.f;
      }
      if (threadIdx.x < kTile) {
        const bool in = qrow0 + threadIdx.x < N;
        sLse[threadIdx.x] = in ? p.lse[qbase + qrow0 + threadIdx.x] * kLog2e : 0.f;
        sD[threadIdx.x] = in ? p.delta[qbase + qrow0 + threadIdx.x] : 0.f;
      }
      __syncthreads();
      const int qrow = qrow0 + lane;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int lr = warp * 8 + r, key = key0 + lr;
        float s = 0.f, dp = 0.f;
        for (int c = 0; c < d; ++c) {
          s = fmaf(sQ[lane * dp1 + c], sK[lr * d + c], s);
          dp = fmaf(sdO[lane * dp1 + c], sV[lr * d + c], dp);
        }
        const bool masked = qrow >= N || key >= Nk || (CAUSAL && key > qrow + off);
        const float pr = masked ? 0.f : exp2f(s * p.scale_log2 - sLse[lane]);
        const float ds = pr * (dp - sD[lane]);
        for (int ii = 0; ii < kTile; ++ii) {
          const float pi = __shfl_sync(0xffffffffu, pr, ii);
          const float dsi = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
          for (int i = 0; i < kColsPerLane; ++i) {
            const int c = lane + 32 * i;
            if (c < d) {
              dv[r][i] = fmaf(pi, sdO[ii * dp1 + c], dv[r][i]);
              dk[r][i] = fmaf(dsi, sQ[ii * dp1 + c], dk[r][i]);
            }
          }
        }
      }
    }
  }
  float* dkp = static_cast<float*>(p.dk) + bb.hkv * p.lay_dkv.head + s0 * p.lay_dkv.row;
  float* dvp = static_cast<float*>(p.dv) + bb.hkv * p.lay_dkv.head + s0 * p.lay_dkv.row;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int key = key0 + warp * 8 + r;
    if (key >= Nk) continue;
#pragma unroll
    for (int i = 0; i < kColsPerLane; ++i) {
      const int c = lane + 32 * i;
      if (c < d) {
        dkp[key * p.lay_dkv.row + c] = dk[r][i] * p.scale;
        dvp[key * p.lay_dkv.row + c] = dv[r][i];
      }
    }
  }
}

}  // namespace

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

cudaError_t launch_fwd_f32(const void* q, const void* k, const void* v, const FwdParams& p, bool causal,
                           int mode, cudaStream_t stream) {
  const size_t smem = sizeof(float) * (kTile * (p.d + 1) + kTile * p.d + kRows * p.d);
  const float* qf = static_cast<const float*>(q);
  const float* kf = static_cast<const float*>(k);
  const float* vf = static_cast<const float*>(v);
  auto run = [&](auto kern, dim3 grid) -> cudaError_t {
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 128, smem, stream>>>(qf, kf, vf, p);
    return cudaGetLastError();
  };
  if (mode == kModeKv) {
    const dim3 grid(p.B * p.Hq, (p.Nq + kRows - 1) / kRows, p.n_splits);
    return causal ? run(fwd_f32_kv_kernel<true>, grid) : run(fwd_f32_kv_kernel<false>, grid);
  }
  if (mode == kModeVarlen) {
    const dim3 grid(p.Hq, (p.max_seqlen + kRows - 1) / kRows, p.nseq);
    return causal ? run(fwd_f32_kernel<true, true>, grid) : run(fwd_f32_kernel<false, true>, grid);
  }
  const dim3 grid(p.B * p.Hq, (p.N + kRows - 1) / kRows, 1);
  return causal ? run(fwd_f32_kernel<true, false>, grid) : run(fwd_f32_kernel<false, false>, grid);
}

cudaError_t launch_bwd_f32(const BwdParams& p, bool causal, cudaStream_t stream) {
  // dense: x = batch * heads; varlen: x = sequence * heads, y over the longest sequence
  const int xs = p.cu_seqlens ? p.nseq : p.B;
  const int nyq = ((p.cu_seqlens ? p.max_seqlen : p.N) + kRows - 1) / kRows;
  const int nyk = ((p.cu_seqlens ? p.max_seqlen : p.Nk) + kRows - 1) / kRows;
  const dim3 gq(xs * p.Hq, nyq);
  const dim3 gk(xs * p.Hkv, nyk);
  const size_t smem_q = sizeof(float) * (2 * kTile * (p.d + 1) + 2 * kRows * p.d);
  const size_t smem_k = sizeof(float) * (2 * kTile * (p.d + 1) + 2 * kRows * p.d + 2 * kTile);
  auto kq = causal ? bwd_dq_f32_kernel<true> : bwd_dq_f32_kernel<false>;
  auto kk = causal ? bwd_dkdv_f32_kernel<true> : bwd_dkdv_f32_kernel<false>;
  cudaError_t e = set_smem(kq, smem_q);
  if (e == cudaSuccess) e = set_smem(kk, smem_k);
  if (e != cudaSuccess) return e;
  kq<<<gq, 128, smem_q, stream>>>(p);
  kk<<<gk, 128, smem_k, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
