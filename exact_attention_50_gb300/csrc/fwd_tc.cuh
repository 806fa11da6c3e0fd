// fwd_tc.cuh -- tcgen05 forward for fp16 / bf16: TMA-fed, warp-specialised, S and O in TMEM.
//
// What it computes (per query row i of a (batch, head) or (sequence, head)):
//   S_ij = scale * Q_i . K_j, masked to -inf for j > i (causal) and for keys past the sequence;
//   online softmax over key tiles (running max m and sum l, exp2 with log2(e) folded into the
//   scale); O_i = sum_j P_ij V_j / l_i; LSE_i = m_i + ln l_i.
// The tiling follows the attention-operator article (m.xxqk.cn/news/636956) section 2.2: Q/K/V
// tiles staged on chip, the max-subtracted softmax kept in registers and only O written back.
// The online max/sum update follows the FlashAttention-T review, best practice 4; scale and
// mask are applied inside the GEMM loop as in its best practice 2.
//
// One CTA = one 128-row query tile, 6 warps:
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t); loads its S row from TMEM,
//              masks, updates m/l, writes P (16-bit, 128-byte swizzled) to shared memory,
//              rescales its O row in TMEM when the max moved, and runs the epilogue.
//   warp 4     TMA producer (lane 0) and TMEM allocator (whole warp).
//   warp 5     MMA issuer (lane 0): S_j = Q K_j^T into one of two TMEM S buffers, then
//              O += P_{j-1} V_{j-1}; each group is committed to an mbarrier.
// TMEM: S buffers at columns [0,128) and [128,256), O at [256, 256+DP).
// K and V stream through separate STAGES-deep rings; Q is loaded once.
//
// Lazy rescaling: the running max used for the exponentials is only moved when a tile's max
// exceeds it by more than kRescaleLog2 (in log2 units); the final O / l and LSE use the same
// max, so the result is exact, and P stays below 2^kRescaleLog2 (well inside fp16 range).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "kernels.h"
#include "ptx.cuh"

namespace attn {

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
  static constexpr bool kBf16 = true;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};
template <>
struct Elem<__half> {
  static constexpr bool kBf16 = false;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};

constexpr float kRescaleLog2 = 8.0f;

template <int DP>
struct FwdLayout {
  static constexpr int kStages = DP == 128 ? 2 : 3;
  static constexpr int kChunkBytes = 128 * 128;          // 128 rows x 64 elements x 2 B
  static constexpr int kTileBytes = (DP / 64) * kChunkBytes;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffP = kOffV + kStages * kTileBytes;
  static constexpr int kOffBar = kOffP + 2 * kChunkBytes;
  // barriers: q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], s_free[2],
  //           p_full, o_done, drain
  static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 3;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem base (u32), abort flag (int)
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kBytes + 1024;         // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  uint32_t s = smem_u32(p);
  return reinterpret_cast<uint8_t*>(a + ((1024u - (s & 1023u)) & 1023u));
}

template <typename T, int DP, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(192, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using L = FwdLayout<DP>;
  constexpr int S = L::kStages;
  constexpr int kChunks = DP / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  uint8_t* sP = smem + L::kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + S;
  uint64_t* v_full = k_empty + S;
  uint64_t* v_empty = v_full + S;
  uint64_t* s_full = v_empty + S;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* o_done = p_full + 1;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- which tile this CTA computes
  int b = 0, h, qt, seq_start = 0, seq_len;
  if constexpr (VARLEN) {
    h = blockIdx.x;
    const int s = blockIdx.z;
    qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.y);
    const int c0 = p.cu_seqlens[s], c1 = p.cu_seqlens[s + 1];
    const bool bad = c0 < 0 || c1 < c0 || c1 > p.total_tokens || c1 - c0 > p.max_seqlen ||
                     (s == 0 && c0 != 0) || (s == p.nseq - 1 && c1 != p.total_tokens);
    if (bad) {
      if (threadIdx.x == 0) raise_status(p.status, ATTN_ERR_DEVICE_INPUT);
      return;
    }
    seq_start = c0;
    seq_len = c1 - c0;
    if (qt * kBM >= seq_len) return;
  } else {
    b = blockIdx.x / p.Hq;
    h = blockIdx.x % p.Hq;
    qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.y);
    seq_len = p.N;
  }
  const int g = h / p.G;
  const int n_kv_all = (seq_len + kBN - 1) / kBN;
  const int n_kv = CAUSAL ? min(qt + 1, n_kv_all) : n_kv_all;

  // ---- setup
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < S; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(s_free + i, 128);
    }
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 4) tmem_alloc(tmem_slot, L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint32_t tile_bytes = L::kTileBytes;
      mbar_expect_tx(q_full, tile_bytes);
      for (int c = 0; c < kChunks; ++c) {
        if constexpr (VARLEN)
          tma_load_4d(sQ + c * L::kChunkBytes, &tmQ, q_full, c * 64, h, 0, seq_start + qt * kBM);
        else
          tma_load_3d(sQ + c * L::kChunkBytes, &tmQ, q_full, c * 64, qt * kBM, b * p.Hq + h);
      }
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % S;
        const uint32_t ph = ((j / S) - 1) & 1;
        if (j >= S && !mbar_wait(k_empty + st, ph, abort_flag, p.status)) break;
        mbar_expect_tx(k_full + st, tile_bytes);
        for (int c = 0; c < kChunks; ++c) {
          uint8_t* dst = sK + st * L::kTileBytes + c * L::kChunkBytes;
          if constexpr (VARLEN)
            tma_load_4d(dst, &tmK, k_full + st, c * 64, h, 1, seq_start + j * kBN);
          else
            tma_load_3d(dst, &tmK, k_full + st, c * 64, j * kBN, b * p.Hkv + g);
        }
        if (j >= S && !mbar_wait(v_empty + st, ph, abort_flag, p.status)) {
          issued = 2 * j + 1;
          break;
        }
        mbar_expect_tx(v_full + st, tile_bytes);
        for (int c = 0; c < kChunks; ++c) {
          uint8_t* dst = sV + st * L::kTileBytes + c * L::kChunkBytes;
          if constexpr (VARLEN)
            tma_load_4d(dst, &tmV, v_full + st, c * 64, h, 2, seq_start + j * kBN);
          else
            tma_load_3d(dst, &tmV, v_full + st, c * 64, j * kBN, b * p.Hkv + g);
        }
        issued = 2 * j + 2;
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA's shared memory goes away
        mbar_drain(q_full, 0);
        const int nk = (issued + 1) / 2, nv = issued / 2;
        for (int j = max(0, nk - S); j < nk; ++j) mbar_drain(k_full + j % S, (j / S) & 1);
        for (int j = max(0, nv - S); j < nv; ++j) mbar_drain(v_full + j % S, (j / S) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr bool kB = Elem<T>::kBf16;
      constexpr uint32_t idS = idesc_f16(kB, false, false, 128, kBN);
      constexpr uint32_t idO = idesc_f16(kB, false, true, 128, DP);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP);
      const uint32_t tO = tmem + 256;
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status);
      auto issue_pv = [&](int jj) -> bool {
        if (!mbar_wait(p_full, jj & 1, abort_flag, p.status)) return false;
        const int st = jj % S;
        if (!mbar_wait(v_full + st, (jj / S) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint64_t a = smem_desc_sw128(aP + (ks >> 2) * L::kChunkBytes + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(aV + st * L::kTileBytes + ks * 2048, L::kChunkBytes, 1024);
          mma_ss(tO, a, bd, idO, (jj > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(v_empty + st);
        return true;
      };
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % S;
        const int sb = j & 1;
        if (!mbar_wait(k_full + st, (j / S) & 1, abort_flag, p.status)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(s_free + sb, ((j >> 1) - 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < DP / 16; ++ks) {
          const uint32_t off = (ks >> 2) * L::kChunkBytes + (ks & 3) * 32;
          const uint64_t a = smem_desc_sw128(aQ + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(aK + st * L::kTileBytes + off, 16, 1024);
          mma_ss(tmem + sb * 128, a, bd, idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(s_full + sb);
        mma_commit(k_empty + st);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(n_kv - 1);
      if (!ok) {
        mma_commit(drain);  // every MMA issued so far completes before this arrives
        mbar_drain(drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ softmax warps 0-3
    const int row = threadIdx.x;  // 0..127 == TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int q_row = qt * kBM + row;  // relative to the sequence
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    uint8_t* prow = sP + row * 128;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(s_full + sb, (j >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      float s[kBN];
      {
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          tmem_ld32(tl + sb * 128 + c * 32, r);
          tmem_ld_wait();
          tmem_reg_fence(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(s_free + sb);

      const int key0 = j * kBN;
      if ((CAUSAL && key0 + kBN - 1 > q_row) || key0 + kBN > seq_len) {
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          const int key = key0 + c;
          if ((CAUSAL && key > q_row) || key >= seq_len) s[c] = -INFINITY;
        }
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kBN; ++c) mx = fmaxf(mx, s[c]);
      const float mx2 = mx * sl2;  // scale > 0: max commutes with the scaling
      float alpha = 1.f;
      bool resc = false;
      if (mx2 > m + kRescaleLog2 || (m == -INFINITY && mx2 != -INFINITY)) {
        alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - mx2);
        resc = (j > 0) && (m != -INFINITY);
        m = mx2;
      }
      const float mb = (m == -INFINITY) ? 0.f : m;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kBN; ++c) {
        s[c] = ex2_approx(fmaf(s[c], sl2, -mb));
        rs += s[c];
      }
      l = l * alpha + rs;

      if (j >= 1) {
        if (!mbar_wait(o_done, (j - 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
          const float a = resc ? alpha : 1.f;
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < DP / 32; ++c) {
            tmem_ld32(tl + 256 + c * 32, r);
            tmem_ld_wait();
            tmem_reg_fence(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * a);
            tmem_st32(tl + 256 + c * 32, r);
          }
          tmem_st_wait();
        }
      }
      // P row -> shared memory, K-major with the 128-byte swizzle (16-byte granule g of a
      // 128-byte row r lands at granule g ^ (r & 7)).
#pragma unroll
      for (int gi = 0; gi < kBN / 8; ++gi) {
        uint4 v;
        v.x = Elem<T>::pack(s[gi * 8 + 0], s[gi * 8 + 1]);
        v.y = Elem<T>::pack(s[gi * 8 + 2], s[gi * 8 + 3]);
        v.z = Elem<T>::pack(s[gi * 8 + 4], s[gi * 8 + 5]);
        v.w = Elem<T>::pack(s[gi * 8 + 6], s[gi * 8 + 7]);
        uint8_t* dst = prow + (gi >> 3) * L::kChunkBytes + ((((gi & 7) ^ (row & 7))) << 4);
        *reinterpret_cast<uint4*>(dst) = v;
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // ---- epilogue: O / l and LSE
    if (ok && n_kv > 0 && mbar_wait(o_done, (n_kv - 1) & 1, abort_flag, p.status)) {
      tc_fence_after();
      const bool valid = q_row < seq_len;
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      size_t row_off;
      if constexpr (VARLEN)
        row_off = (static_cast<size_t>(seq_start + q_row) * p.Hq + h) * p.d;
      else
        row_off = ((static_cast<size_t>(b) * p.Hq + h) * p.N + q_row) * p.d;
      uint32_t r[32];
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        tmem_ld32(tl + 256 + c * 32, r);
        tmem_ld_wait();
        tmem_reg_fence(r);
        const int col0 = c * 32;
        if (valid && col0 < p.d) {
          const int ncol = min(32, p.d - col0);  // 16 or 32 (d is a multiple of 16)
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + row_off + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (i * 4 < ncol)
                dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv_l, __uint_as_float(r[4 * i + 1]) * inv_l,
                                     __uint_as_float(r[4 * i + 2]) * inv_l, __uint_as_float(r[4 * i + 3]) * inv_l);
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.o) + row_off + col0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (i * 8 < ncol) {
                uint4 v;
                v.x = Elem<T>::pack(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l);
                v.y = Elem<T>::pack(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l);
                v.z = Elem<T>::pack(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l);
                v.w = Elem<T>::pack(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l);
                dst[i] = v;
              }
            }
          }
        }
      }
      if (valid && p.lse) {
        const float lse = (m + __log2f(l)) * 0.69314718055994531f;
        if constexpr (VARLEN)
          p.lse[static_cast<size_t>(h) * p.total_tokens + seq_start + q_row] = lse;
        else
          p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.N + q_row] = lse;
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <typename T, int DP, bool CAUSAL, bool VARLEN>
cudaError_t launch_fwd_tc_t(const FwdMaps& maps, const FwdParams& p, cudaStream_t stream) {
  using L = FwdLayout<DP>;
  auto kern = fwd_tc_kernel<T, DP, CAUSAL, VARLEN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid;
  if (VARLEN)
    grid = dim3(p.Hq, p.n_qtiles, p.nseq);
  else
    grid = dim3(p.B * p.Hq, p.n_qtiles, 1);
  kern<<<grid, 192, L::kSmemAlloc, stream>>>(maps.q, maps.k, maps.v, p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fwd_tc_dtype(const FwdMaps& maps, const FwdParams& p, bool causal, bool varlen,
                                cudaStream_t stream) {
  const bool d64 = p.d <= 64;
  if (d64) {
    if (varlen) return causal ? launch_fwd_tc_t<T, 64, true, true>(maps, p, stream)
                              : launch_fwd_tc_t<T, 64, false, true>(maps, p, stream);
    return causal ? launch_fwd_tc_t<T, 64, true, false>(maps, p, stream)
                  : launch_fwd_tc_t<T, 64, false, false>(maps, p, stream);
  }
  if (varlen) return causal ? launch_fwd_tc_t<T, 128, true, true>(maps, p, stream)
                            : launch_fwd_tc_t<T, 128, false, true>(maps, p, stream);
  return causal ? launch_fwd_tc_t<T, 128, true, false>(maps, p, stream)
                : launch_fwd_tc_t<T, 128, false, false>(maps, p, stream);
}

}  // namespace attn
