// kernels.h -- internal launch interface between the C ABI layer (attn_api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include "attn.h"

namespace attn {

constexpr int kBM = 128;  // query rows per tile (one TMEM lane per row)
constexpr int kBN = 128;  // keys per tile

// Everything a forward launch needs besides the tensor maps.
struct FwdParams {
  void* o;                 // [B,Hq,N,d] or varlen [T,H,d]
  float* lse;              // [B,Hq,N] or varlen [H,T]; nullable
  const int32_t* cu_seqlens;  // varlen only
  unsigned* status;        // device status word
  int B, Hq, Hkv, N, d, G;
  int nseq, total_tokens, max_seqlen;
  int n_qtiles;            // query tiles per (sequence, head): grid extent
  float scale;             // softmax scale (natural units)
  float scale_log2;        // scale * log2(e)
  int out_f32;             // write o as float32
  unsigned long long wait_ns;  // limit of any single pipeline wait (0: the 4 s default)
  // KV cache / cross-attention: q [B,Hq,Nq,d] read as [B*Hkv, R = G*Nq, d] (the G query heads
  // of a kv head are consecutive), k and v [B,Hkv,Nk,d], cache_seqlens [B] (null: Nk each).
  // The key tiles of a (batch, kv head) are cut into n_splits ranges of tiles_per_split tiles;
  // each range writes its normalised fp32 partial output and LSE, combined afterwards.
  int Nq, Nk, R;
  const int32_t* cache_seqlens;
  int n_splits, tiles_per_split;
  float* o_part;           // [n_splits, B*Hkv*R, d]
  float* lse_part;         // [n_splits, B*Hkv*R] (natural log)
};

// KV cache: the number of leading keys that some row of 128-row block rb of a (batch, kv head)
// sees.  Row r of the block is query i = r % Nq; query i sees keys j < L, and when causal only
// j <= L - Nq + i (the queries are the last Nq positions of an L-token sequence).  The
// forward kernel and the split combine both derive the split ranges from it.
__host__ __device__ inline int kv_needed_keys(int L, int Nq, int R, int rb, bool causal) {
  if (!causal) return L;
  const int r0 = rb * 128;
  const int r1 = (r0 + 128 < R ? r0 + 128 : R) - 1;
  const int max_i = (r0 / Nq == r1 / Nq) ? r1 % Nq : Nq - 1;
  const int n = L - Nq + max_i + 1;
  return n < 0 ? 0 : (n > L ? L : n);
}

// Tensor maps for the tcgen05 forward: Q, K, V (dense: 3-D {d, N, B*H}; varlen: the same
// 4-D map {d, H, 3, T} three times; KV cache: Q {d, R, B*Hkv}, K and V {d, Nk, B*Hkv}).
// Boxes are {64, 128(, 1)} with 128-byte swizzle; rows past a map's extent load as zeros.
struct FwdMaps {
  CUtensorMap q, k, v;
  CUtensorMap o;  // dense 16-bit output: the epilogue's tile stores ({d, N, B*Hq}, like q)
};

// Work-item layouts of the forward kernels.
constexpr int kModeDense = 0, kModeVarlen = 1, kModeKv = 2;

cudaError_t launch_fwd_tc(const FwdMaps& maps, const FwdParams& p, attn_dtype_t dtype, bool causal, int mode,
                          cudaStream_t stream);
cudaError_t launch_fwd_f32(const void* q, const void* k, const void* v, const FwdParams& p, bool causal,
                           int mode, cudaStream_t stream);
// KV cache: merges the n_splits partial outputs of every row into o (dtype, or fp32 when
// out_f32 or dtype is fp32) and lse (nullable); a row with no visible key gets O = 0 and
// LSE = -inf.
cudaError_t launch_kv_combine(const FwdParams& p, attn_dtype_t dtype, bool causal, cudaStream_t stream);

// Short sequences (N <= 64): units of one (batch, kv head) -- R = G * N query rows against N
// keys -- packed P to a 128-row tile when R <= 128 (flat 2-D maps {d, U*R} and {d, U*N} with
// boxes of exactly P*R and P*N rows), else one unit's 128-row block per item (3-D maps
// {d, R, U} and {d, N, U}).
struct ShortParams {
  void* o;                 // [B,Hq,N,d] = flat [U*R, d]
  float* lse;              // [B,Hq,N] = flat [U*R]; nullable
  unsigned* status;
  unsigned long long wait_ns;
  int U, N, R, G, d;
  int packed, P, row_tiles, n_items;
  int box_q, box_k;        // rows of the query / output box and of the key / value box
  float scale_log2;
  int out_f32;
};

cudaError_t launch_fwd_short(const FwdMaps& maps, const ShortParams& p, attn_dtype_t dtype, bool causal,
                             cudaStream_t stream);

// Backward.
struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;   // workspace [B,Hq,N,d] fp32
  float* delta;    // workspace [B,Hq,N] fp32: D_i = dO_i . O_i
  int* dq_turn;    // workspace [B,Hq,N] int32, zeroed with dq_acc: at the first row of each
                   // 128-row dQ tile, the key tiles that have added into that tile
  int deterministic;  // add dQ tiles in key-tile order (ATTN_FLAG_DETERMINISTIC)
  unsigned* status;
  unsigned long long wait_ns;  // limit of any single pipeline wait (0: the 4 s default)
  int B, Hq, Hkv, N, d, G;
  // Keys per head (dense): N for self-attention, else the cross-attention key count, with the
  // bottom-right causal alignment: query i sees key j iff j <= i + (Nk - N).  Varlen: the
  // sequences are self-attention (Nk == N == total_tokens).
  int Nk;
  int n_ktiles;
  float scale, scale_log2;
  int out_f32;
  // Element offset of row n of head hh in a [rows, d] tensor: hh * head + n * row (a packed
  // tensor's plane is part of its pointer).  Dense [B,H,N,d]: {d, N*d} with hh = b*H + h.
  // Varlen: {token stride, d} with hh = h.
  struct Rows {
    long long row, head;
  };
  Rows lay_q, lay_kv, lay_o, lay_dq, lay_dkv;  // q; k and v; o and dout; dq; dk and dv
  // Varlen: the sequences are the diagonal blocks of a B = 1, N = total_tokens problem; the
  // fp32 row statistics (LSE, D) and the dQ accumulator are [H, T] ([H, T, d]).
  const int32_t* cu_seqlens;  // null for dense
  int nseq, max_seqlen;
};

// Tensor maps for the tcgen05 backward: 3-D {d, rows, heads} with the layout's row / head
// strides and a {64, 128, 1} box, for dense and varlen tensors alike; and the fp32 dQ
// accumulator as 2-D {d, rows} with a {32, 128} box (128-byte swizzle) for tile reductions.
struct BwdMaps {
  CUtensorMap q, k, v, dout, dq_acc;
};

cudaError_t launch_bwd_preprocess(const BwdParams& p, attn_dtype_t dtype, bool zero_acc, cudaStream_t stream);
cudaError_t launch_bwd_postprocess(const BwdParams& p, attn_dtype_t dtype, cudaStream_t stream);
cudaError_t launch_bwd_tc(const BwdMaps& maps, const BwdParams& p, attn_dtype_t dtype, bool causal,
                          cudaStream_t stream);  // varlen when p.cu_seqlens is set
cudaError_t launch_bwd_f32(const BwdParams& p, bool causal, cudaStream_t stream);

}  // namespace attn
