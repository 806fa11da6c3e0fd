// fwd_tc.cuh -- tcgen05 forward for fp16 / bf16: persistent, TMA-fed, warp-specialised, two
// 128-row query tiles per CTA sharing every K/V tile, S / P / O in TMEM.
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
// A CTA loops over work items (a pair of consecutive 128-row query tiles A and B of one
// (batch, head) or (sequence, head)), heaviest first under the causal mask.  320 threads:
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: thread t of a group owns query
//              row t (TMEM lane t); loads its S row, masks, updates m / l, writes P (16-bit) back
//              over columns 64-127 of its own S row, rescales its O row when the max moved,
//              and writes O / l and the LSE at the end of the item.
//   warp 8     TMA producer (lane 0) and TMEM allocator (whole warp).
//   warp 9     MMA issuer (lane 0).  Per key tile j, in order:
//                PV_A(j-1) ; S_A(j) ; PV_B(j-1) ; S_B(j)
//              so that while one group computes its softmax the tensor core works on the
//              other tile.  S_X(j) is two N=64 MMAs: the half writing columns 0-63 is queued at
//              once; the half writing columns 64-127, where P_X(j-1) lives, is issued only after
//              PV_X(j-1) has completed (its mbarrier), never just after it in program order.
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+DP), O_B [256+DP, 256+2DP).
// Shared memory: Q_A, Q_B, and STAGES-deep K and V rings.
//
// Lazy rescaling: the running max used for the exponentials is only moved when a tile's max
// exceeds it by more than kRescaleLog2 (log2 units); the final O / l and LSE use the same max,
// so the result is exact, and P stays below 2^kRescaleLog2 (well inside fp16 range).  Because
// S_X(j) is issued after PV_X(j-1) completed, a softmax group that sees S_X(j) may rescale O_X
// at once.
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
  static constexpr int kStages = DP == 128 ? 2 : 4;
  static constexpr int kChunkBytes = 128 * 128;          // 128 rows x 64 elements x 2 B
  static constexpr int kTileBytes = (DP / 64) * kChunkBytes;
  static constexpr int kOffQ = 0;                        // Q_A then Q_B
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  // q_full, q_empty, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2],
  // pv_done[2], o_free[2], drain
  static constexpr int kNumBars = 2 + 4 * kStages + 8 + 1;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem base (u32), abort flag (int)
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kBytes + 1024;         // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  // 3 warpgroups: softmax A, softmax B, and producer / MMA (+2 idle warps).  Launched at
  // kLaunchRegs registers per thread; the producer warpgroup gives registers to the softmax
  // warpgroups (kRegsLow + 2 * kRegsHigh == 3 * kLaunchRegs).
  static constexpr int kThreads = 384;
  static constexpr uint32_t kLaunchRegs = 168, kRegsLow = 104, kRegsHigh = 200;
  static_assert(kRegsLow + 2 * kRegsHigh == 3 * kLaunchRegs, "register split must match the launch");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  uint32_t s = smem_u32(p);
  return reinterpret_cast<uint8_t*>(a + ((1024u - (s & 1023u)) & 1023u));
}

// One work item: a pair of 128-row query tiles (rows [256*pair, 256*pair+256) of a sequence).
struct FwdItem {
  int b, h, pair, seq_start, seq_len, n_kv;
  bool valid;
};

template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ FwdItem fwd_item(const FwdParams& p, int idx) {
  FwdItem it;
  const int heads = VARLEN ? p.Hq : p.B * p.Hq;
  const int per_pair = VARLEN ? heads * p.nseq : heads;
  it.pair = p.n_qtiles - 1 - idx / per_pair;  // n_qtiles counts pairs here; heaviest first
  const int rem = idx % per_pair;
  it.valid = true;
  if constexpr (VARLEN) {
    const int s = rem / heads;
    it.h = rem % heads;
    it.b = 0;
    const int c0 = p.cu_seqlens[s], c1 = p.cu_seqlens[s + 1];
    const bool bad = c0 < 0 || c1 < c0 || c1 > p.total_tokens || c1 - c0 > p.max_seqlen ||
                     (s == 0 && c0 != 0) || (s == p.nseq - 1 && c1 != p.total_tokens);
    if (bad) {
      if (it.pair == 0 && it.h == 0) raise_status(p.status, ATTN_ERR_DEVICE_INPUT);
      it.valid = false;
    }
    it.seq_start = c0;
    it.seq_len = c1 - c0;
    if (it.pair * 2 * kBM >= it.seq_len) it.valid = false;
  } else {
    it.b = rem / p.Hq;
    it.h = rem % p.Hq;
    it.seq_start = 0;
    it.seq_len = p.N;
  }
  const int n_kv_all = (it.seq_len + kBN - 1) / kBN;
  it.n_kv = CAUSAL ? min(2 * it.pair + 2, n_kv_all) : n_kv_all;
  if (it.n_kv <= 0) it.valid = false;
  return it;
}

template <typename T, int DP, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(384, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p, int n_items) {
  using L = FwdLayout<DP>;
  constexpr int S = L::kStages;
  constexpr int kChunks = DP / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = k_full + S;
  uint64_t* v_full = k_empty + S;
  uint64_t* v_empty = v_full + S;
  uint64_t* s_full = v_empty + S;   // [2]: tile A, tile B
  uint64_t* p_full = s_full + 2;    // [2]
  uint64_t* pv_done = p_full + 2;   // [2]
  uint64_t* o_free = pv_done + 2;   // [2]
  uint64_t* drain = o_free + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  const uint32_t abort_flag = smem_u32(smem + L::kOffMisc + 4);  // CTA abort flag (shared)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < S; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 128);
      mbar_init(pv_done + i, 1);
      mbar_init(o_free + i, 128);
    }
    mbar_init(drain, 1);
    abort_set(abort_flag, 0);
    mbar_init_fence();
  }
  if (warp == 8) tmem_alloc(tmem_slot, L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Each register-budget change opens its own branch, which runs to the teardown.
  if (warp >= 8) {
  regs_dec<L::kRegsLow>();
  if (warp >= 10) {
    // spare warps of the producer warpgroup: nothing to do
  } else if (warp == 8) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t kv = 0;  // key tiles issued so far (ring position), across items
      uint32_t ic = 0;  // items processed
      uint32_t nk_issued = 0, nv_issued = 0;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
        const FwdItem it = fwd_item<CAUSAL, VARLEN>(p, idx);
        if (!it.valid) continue;
        if (ic > 0 && !mbar_wait(q_empty, (ic - 1) & 1, abort_flag, p.status)) { ok = false; break; }
        mbar_expect_tx(q_full, 2 * L::kTileBytes);
        for (int x = 0; x < 2; ++x) {
          const int row0 = (2 * it.pair + x) * kBM;
          for (int c = 0; c < kChunks; ++c) {
            uint8_t* dst = sQ + x * L::kTileBytes + c * L::kChunkBytes;
            if constexpr (VARLEN)
              tma_load_4d(dst, &tmQ, q_full, c * 64, it.h, 0, it.seq_start + row0);
            else
              tma_load_3d(dst, &tmQ, q_full, c * 64, row0, it.b * p.Hq + it.h);
          }
        }
        const int g = it.h / p.G;
        for (int j = 0; j < it.n_kv; ++j, ++kv) {
          const int st = kv % S;
          const uint32_t ph = ((kv / S) - 1) & 1;
          if (kv >= S && !mbar_wait(k_empty + st, ph, abort_flag, p.status)) { ok = false; break; }
          mbar_expect_tx(k_full + st, L::kTileBytes);
          for (int c = 0; c < kChunks; ++c) {
            uint8_t* dst = sK + st * L::kTileBytes + c * L::kChunkBytes;
            if constexpr (VARLEN)
              tma_load_4d(dst, &tmK, k_full + st, c * 64, it.h, 1, it.seq_start + j * kBN);
            else
              tma_load_3d(dst, &tmK, k_full + st, c * 64, j * kBN, it.b * p.Hkv + g);
          }
          nk_issued = kv + 1;
          if (kv >= S && !mbar_wait(v_empty + st, ph, abort_flag, p.status)) { ok = false; break; }
          mbar_expect_tx(v_full + st, L::kTileBytes);
          for (int c = 0; c < kChunks; ++c) {
            uint8_t* dst = sV + st * L::kTileBytes + c * L::kChunkBytes;
            if constexpr (VARLEN)
              tma_load_4d(dst, &tmV, v_full + st, c * 64, it.h, 2, it.seq_start + j * kBN);
            else
              tma_load_3d(dst, &tmV, v_full + st, c * 64, j * kBN, it.b * p.Hkv + g);
          }
          nv_issued = kv + 1;
        }
        ++ic;
      }
      if (abort_read(abort_flag)) {
        // let the copies already issued land before the CTA's shared memory goes away
        if (ic > 0) mbar_drain(q_full, (ic - 1) & 1);
        for (uint32_t j = nk_issued > (uint32_t)S ? nk_issued - S : 0; j < nk_issued; ++j)
          mbar_drain(k_full + j % S, (j / S) & 1);
        for (uint32_t j = nv_issued > (uint32_t)S ? nv_issued - S : 0; j < nv_issued; ++j)
          mbar_drain(v_full + j % S, (j / S) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr bool kB = Elem<T>::kBf16;
      constexpr uint32_t idS = idesc_f16(kB, false, false, 128, kBN / 2);
      constexpr uint32_t idO = idesc_f16(kB, false, true, 128, DP);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
      uint32_t kv = 0;  // global key-tile counter (ring position and S/P/PV phases)
      uint32_t ic = 0;
      bool ok = true;
      // Descriptors are built once; a k-step adds its byte offset >> 4 to the start-address
      // field (shared addresses stay below 256 KB, so the 14-bit field never carries).
      const uint64_t dQ = smem_desc_sw128(aQ, 16, 1024);
      const uint64_t dK = smem_desc_sw128(aK, 16, 1024);
      const uint64_t dV = smem_desc_sw128(aV, L::kChunkBytes, 1024);
      // S_x(t) in two N=64 halves: keys 0-63 -> columns 0-63 go at once (P_x(t-1) lives in
      // columns 64-127); keys 64-127 -> columns 64-127 wait until PV_x(t-1) has read P_x(t-1).
      auto issue_s = [&](int x, uint32_t t) -> bool {
        const uint64_t qx = dQ + ((x * L::kTileBytes) >> 4);
        const uint64_t kx = dK + (((t % S) * L::kTileBytes) >> 4);
        tc_fence_after();
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          if (half == 1) {
            if (t > 0 && !mbar_wait(pv_done + x, (t - 1) & 1, abort_flag, p.status)) return false;
            tc_fence_after();
          }
          const uint64_t kh = kx + ((half * 64 * 128) >> 4);  // rows 64*half.. of the K tile
#pragma unroll 1
          for (int ks = 0; ks < DP / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * L::kChunkBytes + (ks & 3) * 32) >> 4;
            mma_ss(tmem + x * 128 + half * 64, qx + off, kh + off, idS, ks > 0 ? 1u : 0u);
          }
        }
        mma_commit(s_full + x);
        return true;
      };
      auto issue_pv = [&](int x, uint32_t t, bool first, bool last_of_pair) -> bool {
        if (!mbar_wait(p_full + x, t & 1, abort_flag, p.status)) return false;
        if (first && ic > 0 && !mbar_wait(o_free + x, (ic - 1) & 1, abort_flag, p.status)) return false;
        const int st = t % S;
        if (!mbar_wait(v_full + st, (t / S) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t tO = tmem + 256 + x * DP;
        const uint64_t vx = dV + ((st * L::kTileBytes) >> 4);
#pragma unroll 1
        for (int ks = 0; ks < kBN / 16; ++ks) {
          mma_ts(tO, tmem + x * 128 + 64 + ks * 8, vx + ((ks * 2048) >> 4), idO, (!first || ks > 0) ? 1u : 0u);
        }
        mma_commit(pv_done + x);
        if (last_of_pair) mma_commit(v_empty + st);
        return true;
      };
      for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
        const FwdItem it = fwd_item<CAUSAL, VARLEN>(p, idx);
        if (!it.valid) continue;
        if (!mbar_wait(q_full, ic & 1, abort_flag, p.status)) { ok = false; break; }
        const uint32_t t0 = kv;
        // prologue: S_A(0), S_B(0)
        if (!mbar_wait(k_full + t0 % S, (t0 / S) & 1, abort_flag, p.status)) { ok = false; break; }
        if (!issue_s(0, t0) || !issue_s(1, t0)) { ok = false; break; }
        mma_commit(k_empty + t0 % S);
        if (it.n_kv == 1) mma_commit(q_empty);  // the item's last MMA reading Q_A / Q_B is issued
        for (int j = 0; j < it.n_kv; ++j) {
          const uint32_t t = t0 + j;
          const bool more = j + 1 < it.n_kv;
          if (!issue_pv(0, t, j == 0, false)) { ok = false; break; }
          if (more) {
            if (!mbar_wait(k_full + (t + 1) % S, ((t + 1) / S) & 1, abort_flag, p.status)) { ok = false; break; }
            if (!issue_s(0, t + 1)) { ok = false; break; }
          }
          if (!issue_pv(1, t, j == 0, true)) { ok = false; break; }
          if (more) {
            if (!issue_s(1, t + 1)) { ok = false; break; }
            mma_commit(k_empty + (t + 1) % S);
            if (j + 2 == it.n_kv) mma_commit(q_empty);  // last MMA reading Q_A / Q_B issued
          }
        }
        if (!ok) break;
        kv = t0 + it.n_kv;
        ++ic;
      }
      if (!ok) {
        mma_commit(drain);  // every MMA issued so far completes before this arrives
        mbar_drain(drain, 0);
      }
    }
    __syncwarp();
  }
  } else {
    regs_inc<L::kRegsHigh>();
    // ================================================================ softmax groups
    const int x = warp >> 2;                  // 0 = tile A, 1 = tile B
    const int row = threadIdx.x & 127;        // TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t tS = tl + x * 128, tO = tl + 256 + x * DP;
    const float sl2 = p.scale_log2;
    uint32_t kv = 0, ic = 0;
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
      const FwdItem it = fwd_item<CAUSAL, VARLEN>(p, idx);
      if (!it.valid) continue;
      const int q_row = (2 * it.pair + x) * kBM + row;  // relative to the sequence
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t t = kv + j;
        if (!mbar_wait(s_full + x, t & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        float s[kBN];
        {
          // all four 32-column loads in flight, one wait
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(tS + 0, r0);
          tmem_ld32(tS + 32, r1);
          tmem_ld32(tS + 64, r2);
          tmem_ld32(tS + 96, r3);
          tmem_ld_wait();
          tmem_reg_fence(r0);
          tmem_reg_fence(r1);
          tmem_reg_fence(r2);
          tmem_reg_fence(r3);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(r0[i]);
            s[32 + i] = __uint_as_float(r1[i]);
            s[64 + i] = __uint_as_float(r2[i]);
            s[96 + i] = __uint_as_float(r3[i]);
          }
        }
        // keys key0 + c with c > lim are masked (past the diagonal, or past the sequence)
        const int key0 = j * kBN;
        const int lim = CAUSAL ? min(q_row, it.seq_len - 1) - key0 : it.seq_len - 1 - key0;
        if (lim < kBN - 1) {
#pragma unroll
          for (int c = 0; c < kBN; ++c) s[c] = c > lim ? -INFINITY : s[c];
        }
        // row max with 8 independent partial maxima (short dependency chains)
        float mp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mp[k] = s[k];
#pragma unroll
        for (int c = 8; c < kBN; c += 8)
#pragma unroll
          for (int k = 0; k < 8; ++k) mp[k] = fmaxf(mp[k], s[c + k]);
        const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        const float mx2 = mx * sl2;  // scale > 0: max commutes with the scaling
        float alpha = 1.f;
        bool resc = false;
        if (mx2 > m + kRescaleLog2 || (m == -INFINITY && mx2 != -INFINITY)) {
          alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - mx2);
          resc = (j > 0) && (m != -INFINITY);
          m = mx2;
        }
        const float mb = (m == -INFINITY) ? 0.f : m;
        float sp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // 8 partial row sums
        uint32_t pk[kBN / 2];
#pragma unroll
        for (int c = 0; c < kBN; c += 2) {
          const float e0 = ex2_approx(fmaf(s[c], sl2, -mb));
          const float e1 = ex2_approx(fmaf(s[c + 1], sl2, -mb));
          sp[(c / 2) & 7] += e0 + e1;
          pk[c / 2] = Elem<T>::pack(e0, e1);
        }
        const float rs = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
        l = l * alpha + rs;
        // P row over columns 64-127 of this row's S (keys 2c, 2c+1 in column 64 + c)
#pragma unroll
        for (int c = 0; c < kBN / 64; ++c) {
          tmem_st32(tS + 64 + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + c * 32));
        }
        // O_x *= alpha (after the S row is dead, to keep registers low): PV_x(t-1) has completed
        // (S_x(t) was issued after it) and PV_x(t) waits for p_full below
        if (__any_sync(0xffffffffu, resc)) {
          const float a = resc ? alpha : 1.f;
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < DP / 32; ++c) {
            tmem_ld32(tO + c * 32, r);
            tmem_ld_wait();
            tmem_reg_fence(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * a);
            tmem_st32(tO + c * 32, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full + x);
      }
      if (!ok) break;
      kv += it.n_kv;
      // ---- epilogue: O / l and LSE, then release O_x for the next item's first PV
      if (!mbar_wait(pv_done + x, (kv - 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      const bool valid = q_row < it.seq_len;
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      size_t row_off;
      if constexpr (VARLEN)
        row_off = (static_cast<size_t>(it.seq_start + q_row) * p.Hq + it.h) * p.d;
      else
        row_off = ((static_cast<size_t>(it.b) * p.Hq + it.h) * p.N + q_row) * p.d;
      uint32_t r[32];
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        tmem_ld32(tO + c * 32, r);
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
      tc_fence_before();
      mbar_arrive(o_free + x);
      if (valid && p.lse) {
        const float lse = (m + __log2f(l)) * 0.69314718055994531f;
        if constexpr (VARLEN)
          p.lse[static_cast<size_t>(it.h) * p.total_tokens + it.seq_start + q_row] = lse;
        else
          p.lse[(static_cast<size_t>(it.b) * p.Hq + it.h) * p.N + q_row] = lse;
      }
      ++ic;
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

inline int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 148;
  }
  return n;
}

template <typename T, int DP, bool CAUSAL, bool VARLEN>
cudaError_t launch_fwd_tc_t(const FwdMaps& maps, const FwdParams& p_in, cudaStream_t stream) {
  using L = FwdLayout<DP>;
  auto kern = fwd_tc_kernel<T, DP, CAUSAL, VARLEN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
  if (e != cudaSuccess) return e;
  // The in-kernel register split assumes the launch allocation; never launch otherwise (an
  // increase beyond what the block holds would wait forever).
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != static_cast<int>(L::kLaunchRegs)) return cudaErrorInvalidConfiguration;
  FwdParams p = p_in;
  p.n_qtiles = (p_in.n_qtiles + 1) / 2;  // pairs of query tiles
  const long heads = VARLEN ? static_cast<long>(p.Hq) * p.nseq : static_cast<long>(p.B) * p.Hq;
  const long items = heads * p.n_qtiles;
  if (items > 0x7fffffffL) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < sm_count() ? items : sm_count());
  kern<<<grid, L::kThreads, L::kSmemAlloc, stream>>>(maps.q, maps.k, maps.v, p, static_cast<int>(items));
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
