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
// Register-tiled FFMA forward: a CTA of 256 threads owns 64 query rows and walks the keys in
// tiles of 64.  Thread (ty, tx) = (t / 16, t % 16) owns rows 4 ty .. 4 ty + 3; for S = Q K^T it
// computes the 4 x 4 block of keys 4 tx .. 4 tx + 3 (Q and K staged transposed, so each step
// over the head dimension is one float4 of Q and one of K for 16 FMAs), and for O it owns the
// columns 4 tx .. 4 tx + 3 (and 64 + 4 tx .. when d > 64).  A row's max and sum are reduced
// over the 16 threads of its half-warp with shuffles; P goes through shared memory (over the
// K^T area, free once S is computed) to the P V product.  Online softmax in base 2 with
// log2(e) folded into the scale.  About 101 KB of shared memory at d = 128: two CTAs per SM.
constexpr int kBM32 = 64, kBN32 = 64, kPad32 = 4;

template <int DMAX>
struct F32Layout {
  static constexpr int kQt = 0;                                   // [DMAX][kBM32 + pad]: Q^T
  static constexpr int kKt = kQt + DMAX * (kBM32 + kPad32);       // [DMAX][kBN32 + pad]: K^T
  static constexpr int kP = kKt;  // [kBM32][kBN32 + pad]: P over K^T, once S is computed
  static constexpr int kV = kKt + DMAX * (kBN32 + kPad32);        // [kBN32][DMAX + pad]
  static constexpr int kFloats = kV + kBN32 * (DMAX + kPad32);
  static_assert(DMAX * (kBN32 + kPad32) >= kBM32 * (kBN32 + kPad32), "P must fit in the K^T area");
};

template <bool CAUSAL, bool VARLEN, int DMAX>
__global__ void __launch_bounds__(256) fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                                      const float* __restrict__ v, const FwdParams p) {
  using L = F32Layout<DMAX>;
  constexpr int SQ = kBM32 + kPad32, SK = kBN32 + kPad32, SV = DMAX + kPad32, SP = kBN32 + kPad32;
  constexpr int NC = DMAX / 64;  // float4 column groups of O per thread
  extern __shared__ float4 smem_f4[];
  float* smem = reinterpret_cast<float*>(smem_f4);
  float* sQt = smem + L::kQt;
  float* sKt = smem + L::kKt;
  float* sV = smem + L::kV;
  float* sP = smem + L::kP;
  const int t = threadIdx.x, tx = t & 15, ty = t >> 4;
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
    if (qt * kBM32 >= seq_len) return;
  } else {
    b = blockIdx.x / p.Hq;
    h = blockIdx.x % p.Hq;
    seq_len = p.N;
  }
  const int d = p.d, g = h / p.G, d4 = d / 4;
  RowAddr qa, ka;
  if constexpr (VARLEN) {
    // q, k and v already point at planes 0, 1 and 2 of the packed [T,3,H,d] tensor
    const size_t tok = 3ull * p.Hq * d;
    qa = {static_cast<size_t>(seq_start) * tok + static_cast<size_t>(h) * d, tok};
    ka = qa;
  } else {
    qa = {(static_cast<size_t>(b) * p.Hq + h) * p.N * d, static_cast<size_t>(d)};
    ka = {(static_cast<size_t>(b) * p.Hkv + g) * p.N * d, static_cast<size_t>(d)};
  }
  const int row0 = qt * kBM32;
  // Q^T: column c of row r at sQt[c][r]; a warp stores 32 consecutive rows of one column group
  for (int idx = t; idx < kBM32 * (DMAX / 4); idx += 256) {
    const int r = idx % kBM32, c4 = idx / kBM32;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row0 + r < seq_len && c4 < d4) x = *reinterpret_cast<const float4*>(q + qa.base + (row0 + r) * qa.stride + 4 * c4);
    sQt[(4 * c4 + 0) * SQ + r] = x.x;
    sQt[(4 * c4 + 1) * SQ + r] = x.y;
    sQt[(4 * c4 + 2) * SQ + r] = x.z;
    sQt[(4 * c4 + 3) * SQ + r] = x.w;
  }
  float m[4], l[4], o[4][4 * NC];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < 4 * NC; ++c) o[i][c] = 0.f;
  }
  const float sl2 = p.scale_log2;
  const int row_hi = min(seq_len, row0 + kBM32) - 1;
  const int n_keys = CAUSAL ? min(seq_len, row_hi + 1) : seq_len;
  for (int key0 = 0; key0 < n_keys; key0 += kBN32) {
    __syncthreads();  // the previous tile's K, V and P are no longer read
    for (int idx = t; idx < kBN32 * (DMAX / 4); idx += 256) {
      const int r = idx % kBN32, c4 = idx / kBN32;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (key0 + r < seq_len && c4 < d4) x = *reinterpret_cast<const float4*>(k + ka.base + (key0 + r) * ka.stride + 4 * c4);
      sKt[(4 * c4 + 0) * SK + r] = x.x;
      sKt[(4 * c4 + 1) * SK + r] = x.y;
      sKt[(4 * c4 + 2) * SK + r] = x.z;
      sKt[(4 * c4 + 3) * SK + r] = x.w;
    }
    for (int idx = t; idx < kBN32 * (DMAX / 4); idx += 256) {
      const int r = idx / (DMAX / 4), c4 = idx % (DMAX / 4);
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (key0 + r < seq_len && c4 < d4) x = *reinterpret_cast<const float4*>(v + ka.base + (key0 + r) * ka.stride + 4 * c4);
      *reinterpret_cast<float4*>(sV + r * SV + 4 * c4) = x;
    }
    __syncthreads();
    // ---- S block: rows 4 ty + i, keys 4 tx + j
    float sblk[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) sblk[i][j] = 0.f;
#pragma unroll 4
    for (int c = 0; c < d; ++c) {
      const float4 qv = *reinterpret_cast<const float4*>(sQt + c * SQ + 4 * ty);
      const float4 kv = *reinterpret_cast<const float4*>(sKt + c * SK + 4 * tx);
      const float qq[4] = {qv.x, qv.y, qv.z, qv.w}, kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sblk[i][j] = fmaf(qq[i], kk[j], sblk[i][j]);
    }
    __syncthreads();  // every thread is done with K^T: P goes over it
    // ---- online softmax over the tile (a row lives on the 16 threads of a half-warp)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qrow = row0 + 4 * ty + i;
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = key0 + 4 * tx + j;
        const bool masked = key >= seq_len || (CAUSAL && key > qrow);
        sblk[i][j] = masked ? -INFINITY : sblk[i][j] * sl2;
        mx = fmaxf(mx, sblk[i][j]);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[i], mx);
      const float mb = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m[i] - mb);
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sblk[i][j] = exp2f(sblk[i][j] - mb);
        rs += sblk[i][j];
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
      l[i] = l[i] * alpha + rs;
      m[i] = m_new;
#pragma unroll
      for (int c = 0; c < 4 * NC; ++c) o[i][c] *= alpha;
      *reinterpret_cast<float4*>(sP + (4 * ty + i) * SP + 4 * tx) =
          make_float4(sblk[i][0], sblk[i][1], sblk[i][2], sblk[i][3]);
    }
    __syncthreads();
    // ---- O += P V: rows 4 ty + i, columns 4 tx + j (+ 64 when d > 64)
    const int kn = min(kBN32, seq_len - key0);
    for (int kb = 0; kb < kn; kb += 4) {
      float4 pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = *reinterpret_cast<const float4*>(sP + (4 * ty + i) * SP + kb);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        float vv[4 * NC];
#pragma unroll
        for (int cg = 0; cg < NC; ++cg) {
          const float4 x = *reinterpret_cast<const float4*>(sV + (kb + kk) * SV + 64 * cg + 4 * tx);
          vv[4 * cg + 0] = x.x;
          vv[4 * cg + 1] = x.y;
          vv[4 * cg + 2] = x.z;
          vv[4 * cg + 3] = x.w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float pk = kk == 0 ? pr[i].x : kk == 1 ? pr[i].y : kk == 2 ? pr[i].z : pr[i].w;
#pragma unroll
          for (int c = 0; c < 4 * NC; ++c) o[i][c] = fmaf(pk, vv[c], o[i][c]);
        }
      }
    }
  }
  // ---- epilogue: O / l, LSE
  float* out = static_cast<float*>(p.o);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int qrow = row0 + 4 * ty + i;
    if (qrow >= seq_len) continue;
    const float inv_l = 1.f / l[i];
    size_t out_off;
    if constexpr (VARLEN)
      out_off = (static_cast<size_t>(seq_start + qrow) * p.Hq + h) * d;
    else
      out_off = ((static_cast<size_t>(b) * p.Hq + h) * p.N + qrow) * d;
#pragma unroll
    for (int cg = 0; cg < NC; ++cg) {
      const int c = 64 * cg + 4 * tx;
      if (c < d)
        *reinterpret_cast<float4*>(out + out_off + c) =
            make_float4(o[i][4 * cg] * inv_l, o[i][4 * cg + 1] * inv_l, o[i][4 * cg + 2] * inv_l, o[i][4 * cg + 3] * inv_l);
    }
    if (tx == 0 && p.lse) {
      const float lse = (m[i] + log2f(l[i])) / kLog2e;
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
  // dense and varlen: the register-tiled kernel, 64 query rows per CTA
  auto run_tiled = [&](auto kern, dim3 grid, size_t bytes) -> cudaError_t {
    cudaError_t e = set_smem(kern, bytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, 256, bytes, stream>>>(qf, kf, vf, p);
    return cudaGetLastError();
  };
  const bool varlen = mode == kModeVarlen;
  const dim3 grid = varlen ? dim3(p.Hq, (p.max_seqlen + kBM32 - 1) / kBM32, p.nseq)
                           : dim3(p.B * p.Hq, (p.N + kBM32 - 1) / kBM32, 1);
  if (p.d <= 64) {
    const size_t bytes = sizeof(float) * F32Layout<64>::kFloats;
    if (varlen)
      return causal ? run_tiled(fwd_f32_kernel<true, true, 64>, grid, bytes)
                    : run_tiled(fwd_f32_kernel<false, true, 64>, grid, bytes);
    return causal ? run_tiled(fwd_f32_kernel<true, false, 64>, grid, bytes)
                  : run_tiled(fwd_f32_kernel<false, false, 64>, grid, bytes);
  }
  const size_t bytes = sizeof(float) * F32Layout<128>::kFloats;
  if (varlen)
    return causal ? run_tiled(fwd_f32_kernel<true, true, 128>, grid, bytes)
                  : run_tiled(fwd_f32_kernel<false, true, 128>, grid, bytes);
  return causal ? run_tiled(fwd_f32_kernel<true, false, 128>, grid, bytes)
                : run_tiled(fwd_f32_kernel<false, false, 128>, grid, bytes);
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
