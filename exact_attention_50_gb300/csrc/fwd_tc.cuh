// fwd_tc.cuh -- tcgen05 forward for fp16 / bf16: persistent, TMA-fed, warp-specialised, S / P / O
// in TMEM.
//
// What it computes (per query row i of a (batch, head) or (sequence, head)):
//   S_ij = scale * Q_i . K_j, masked to -inf for j > i (causal) and for keys past the sequence;
//   online softmax over key tiles (running max m and sum l, exp2 with log2(e) folded into the
//   scale); O_i = sum_j P_ij V_j / l_i; LSE_i = m_i + ln l_i.
// In the KV-cache mode a row is query i = row % Nq of the G query heads of a kv head, its keys
// are those of one range of the cache, masked past the cache length L and, when causal, past
// L - Nq + i; it writes fp32 partials that a combine kernel merges.
// The tiling follows the attention-operator article (m.xxqk.cn/news/636956) section 2.2: Q/K/V
// tiles staged on chip, the max-subtracted softmax kept in registers and only O written back.
// The online max/sum update follows the FlashAttention-T review, best practice 4; scale and
// mask are applied inside the GEMM loop as in its best practice 2.
//
// A CTA loops over 128-row query tiles, numbered heaviest first under the causal mask and
// dealt to the CTAs in snake order (cta_item).  512 threads:
//   warps 0-3  softmax, key columns 0-63 of each S tile; warps 4-7 softmax, key columns 64-127.
//              Thread t of either group owns query row t (TMEM lane t).  Each group keeps its
//              own running max and sum over its key columns and its own O accumulator (O_g =
//              sum of P_g V over those keys), so the two never wait for each other inside an
//              item.  Each writes its 64 P values (16-bit pairs) over the first 32 of its S
//              columns and rescales O_g when its max moved.  At the end of the item each
//              hands its (max, sum) to the epilogue warps and goes on to the next item.
//   warp 8     TMA producer (lane 0) and TMEM allocator (whole warp).
//   warp 9     MMA issuer of the S(j) stream (lane 0).
//   warps 11, 10  MMA issuers of the PV_0(j) and PV_1(j) streams (lane 0): one thread issues an
//              MMA only every ~110 cycles while busy softmax warps share its sub-partition, so
//              the two groups' PVs go in from two sub-partitions.
//   warps 12-15 epilogue: per item, once its last PV has completed, combine O_0 and O_1 with
//              the two groups' (max, sum) into O / l and LSE, staged in the item's Q slot and
//              written with TMA tile stores by warp 12 (which then frees the slot), or stored
//              per row, while the softmax warps already work on the next item.
// Registers: launched at 128 per thread, then split per warpgroup with setmaxnreg (softmax
// 168, I/O 56, epilogue 120).
// TMEM: S double buffer at columns [0,128) and [128,256), P(j) of group g over columns
// [64g, 64g+32) of S buffer j % 2, O_0 at [256, 256+DP) and O_1 after it.  S(j+2) goes into S
// buffer j % 2 once PV(j) has read P(j), so the tensor core computes S(j+1) while the softmax
// works on S(j).
//
// Lazy rescaling: the running max used for the exponentials is only moved when a tile's max
// exceeds it by more than kRescaleLog2 (log2 units); the final O / l and LSE use the same max,
// so the result is exact, and P stays below 2^kRescaleLog2 (well inside fp16 range).
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
// Which of every 8 exponential pairs run on the FMA pipe (bit k: pair k) instead of the
// special-function unit.  None: at 32 results per clock per SM the special-function unit keeps
// up with the MMAs, and the polynomial's extra instructions cost about as many issue slots as
// they save (1/8 of the pairs on the FMA pipe measured within +-1%, 1/4 and 1/2 slower).
constexpr unsigned kPolyPairs = 0x00u;

template <int DP, int MODE>
struct FwdLayout {
  // For d = 128 two Q tiles, three K and two V tiles in flight (224 KB in all): an L2 load
  // takes up to ~3000 cycles when every SM streams K and V, about two tiles of work.  The
  // second Q slot lets the next item's Q load while the current item's slot, once its last S
  // has run, stages the item's output tile for the tile stores.  (1 Q + 3 V measured the same.)
  // The KV-cache mode stores no output tiles and streams K and V from HBM: one Q slot and a
  // third V stage (more bytes in flight) serve it better.
  static constexpr bool kKv = MODE == kModeKv;
  static constexpr int kStagesQ = (DP == 128 && kKv) ? 1 : 2;
  static constexpr int kStagesK = DP == 128 ? 3 : 4;
  static constexpr int kStagesV = DP == 128 ? (kKv ? 3 : 2) : 4;
  static constexpr int kChunkBytes = 128 * 128;          // 128 rows x 64 elements x 2 B
  static constexpr int kTileBytes = (DP / 64) * kChunkBytes;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kStagesQ * kTileBytes;
  static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
  static constexpr int kOffX = kOffV + kStagesV * kTileBytes;  // item end (m, l): [2 groups][128 rows]
  static constexpr int kOffBar = kOffX + 2 * 2 * 128 * 4;
  // q_full[2], q_empty[2], k_full[SK], k_empty[SK], v_full[SV], v_empty[SV], s_full[2],
  // p_full[2 buffers][2 groups][2 halves], pv_done[2], o_free, drain,
  // o_staged[2] (per Q slot, so it cannot run two phases ahead of the tile stores: a slot takes
  // a new Q only after the tile staged in it has been written out), drain2, drain3,
  // stats_ready, stats_free
  static constexpr int kNumBars = 4 + 2 * kStagesK + 2 * kStagesV + 2 + 8 + 2 + 1 + 1 + 2 + 2 + 2;
  // tmem base (u32), abort flag (int), wait limit (u64, ns)
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kBytes;  // the dynamic shared memory starts 1024-byte aligned
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;  // O_0; O_1 at kColO + DP
  static constexpr int kThreads = 512;
  // launch 128 registers per thread; two softmax warpgroups at 168, the I/O warpgroup (producer,
  // MMA issuers, tile stores) at 56 and the epilogue warpgroup at 120: 2 * 168 + 56 + 120 = 4 * 128
  static constexpr uint32_t kLaunchRegs = 128, kRegsSmx = 168, kRegsIo = 56, kRegsEpi = 120;
  static_assert(2 * kRegsSmx + kRegsIo + kRegsEpi == 4 * kLaunchRegs, "register split must match the launch");
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  uint32_t s = smem_u32(p);
  return reinterpret_cast<uint8_t*>(a + ((1024u - (s & 1023u)) & 1023u));
}

// One work item: a 128-row query tile of one (batch, head) or (sequence, head), or for a KV
// cache a 128-row block of one (batch, kv head)'s R = G * Nq query rows against one range of
// key tiles [j0, j0 + n_kv) (h is then the kv head and seq_len the cache length).
struct FwdItem {
  int b, h, qt, seq_start, seq_len, n_kv, j0, split;
  bool valid;
};

template <bool CAUSAL, int MODE>
__device__ __forceinline__ FwdItem fwd_item(const FwdParams& p, int idx) {
  constexpr bool VARLEN = MODE == kModeVarlen;
  FwdItem it;
  it.j0 = 0;
  it.split = 0;
  if constexpr (MODE == kModeKv) {
    // later row blocks first (under the causal mask they see the most keys), then the key
    // range (first ranges first: they are full, the last ones short or empty), then (batch,
    // kv head).  A CTA takes one item per round of gridDim.x items, so it gets a mix of
    // ranges and of caches of different lengths, and the light items come last.
    const int bhs = p.B * p.Hkv;
    const int per_rb = bhs * p.n_splits;
    it.qt = p.n_qtiles - 1 - idx / per_rb;
    const int rem = idx % per_rb;
    it.split = rem / bhs;
    const int bh = rem % bhs;
    it.b = bh / p.Hkv;
    it.h = bh % p.Hkv;
    it.seq_start = 0;
    it.valid = true;
    int L = p.Nk;
    if (p.cache_seqlens) {
      L = p.cache_seqlens[it.b];
      if (L < 0 || L > p.Nk) {
        if (it.qt == 0 && it.h == 0 && it.split == 0) raise_status(p.status, ATTN_ERR_DEVICE_INPUT);
        it.valid = false;
        L = 0;
      }
    }
    it.seq_len = L;
    const int need_tiles = (kv_needed_keys(L, p.Nq, p.R, it.qt, CAUSAL) + kBN - 1) / kBN;
    it.j0 = it.split * p.tiles_per_split;
    it.n_kv = min(p.tiles_per_split, need_tiles - it.j0);
    if (it.n_kv <= 0) it.valid = false;
    return it;
  }
  const int heads = VARLEN ? p.Hq : p.B * p.Hq;
  const int per_tile = VARLEN ? heads * p.nseq : heads;
  it.qt = p.n_qtiles - 1 - idx / per_tile;  // heaviest first
  const int rem = idx % per_tile;
  it.valid = true;
  if constexpr (VARLEN) {
    const int s = rem / heads;
    it.h = rem % heads;
    it.b = 0;
    const int c0 = p.cu_seqlens[s], c1 = p.cu_seqlens[s + 1];
    const bool bad = c0 < 0 || c1 < c0 || c1 > p.total_tokens || c1 - c0 > p.max_seqlen ||
                     (s == 0 && c0 != 0) || (s == p.nseq - 1 && c1 != p.total_tokens);
    if (bad) {
      if (it.qt == 0 && it.h == 0) raise_status(p.status, ATTN_ERR_DEVICE_INPUT);
      it.valid = false;
    }
    it.seq_start = c0;
    it.seq_len = c1 - c0;
    if (it.qt * kBM >= it.seq_len) it.valid = false;
  } else {
    it.b = rem / p.Hq;
    it.h = rem % p.Hq;
    it.seq_start = 0;
    it.seq_len = p.N;
  }
  const int n_kv_all = (it.seq_len + kBN - 1) / kBN;
  it.n_kv = CAUSAL ? min(it.qt + 1, n_kv_all) : n_kv_all;
  if (it.n_kv <= 0) it.valid = false;
  return it;
}

// The CTA's k-th work item.  Items are numbered heaviest first; round k hands items
// [k G, k G + G) to the G CTAs, forwards in even rounds and backwards in odd ones (a snake), so
// a CTA that drew one of the heavier items of a round draws one of the lighter ones of the
// next and the CTAs' totals come out nearly equal (a plain stride leaves CTA 0 the heaviest
// item of every round: 94% balance against 99.6% at B = 4, H = 32, N = 2048, causal).  The
// varlen numbering has many empty items (query tiles past short sequences) in its light rounds,
// which the snake deals unevenly; it keeps the stride (89% against 85% on 16 sequences of
// U[64, 4096] tokens).  May be >= n_items in the last round: no item.
template <int MODE>
__device__ __forceinline__ int cta_item(int k) {
  const int G = gridDim.x;
  const int c = static_cast<int>(blockIdx.x);
  if (MODE == kModeVarlen) return k * G + c;
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Walks the key tiles of a CTA's work items in order (item by item, key tile by key tile).
// The producer and the MMA issuer each run such walks for their streams (Q/K, V; S, PV).
template <bool CAUSAL, int MODE>
struct TileCursor {
  int k, j;     // the CTA's work item (cta_item(k)) and key tile within it
  uint32_t t;   // key tiles passed so far: ring position and barrier phases, across items
  uint32_t ic;  // items passed so far
  FwdItem it;
  bool done;
  __device__ __forceinline__ void seek(const FwdParams& p, int n_items) {
    for (; k * static_cast<int>(gridDim.x) < n_items; ++k) {
      const int idx = cta_item<MODE>(k);
      if (idx >= n_items) continue;
      it = fwd_item<CAUSAL, MODE>(p, idx);
      if (it.valid) return;
    }
    done = true;
  }
  __device__ __forceinline__ void start(const FwdParams& p, int n_items) {
    k = 0;
    j = 0;
    t = 0;
    ic = 0;
    done = false;
    seek(p, n_items);
  }
  __device__ __forceinline__ void advance(const FwdParams& p, int n_items) {
    ++t;
    if (++j < it.n_kv) return;
    j = 0;
    ++ic;
    ++k;
    seek(p, n_items);
  }
};

template <typename T, int DP, bool CAUSAL, int MODE>
__global__ void __launch_bounds__(512, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p, int n_items) {
  constexpr bool VARLEN = MODE == kModeVarlen;
  constexpr bool KV = MODE == kModeKv;
  // 16-bit output of a dense item, or of a varlen item whose 128 rows all lie in its
  // sequence: the epilogue warps stage the item's O tile in the item's Q slot (free once its
  // last S has run) and their thread 0 writes it with tile stores, then frees the slot.
  // Otherwise (a varlen tile that ends past its sequence must not write into the next one; fp32
  // output or KV-cache partials) the epilogue warps store their rows themselves and the last S
  // frees the Q slot.  Every role decides per item with the same function.
  const bool tile_out = (MODE == kModeDense || MODE == kModeVarlen) && !p.out_f32;
  auto tile_item = [&](const FwdItem& it) -> bool {
    return tile_out && (MODE == kModeDense || (it.qt + 1) * kBM <= it.seq_len);
  };
  using L = FwdLayout<DP, MODE>;
  constexpr int SQ = L::kStagesQ, SK = L::kStagesK, SV = L::kStagesV;
  // P(j) is handed to the PV issuers in PH parts per group (d = 128: two halves of 32 keys, so
  // the first half's MMAs go in while the second half's exponentials run; d = 64, where the
  // softmax itself is the limit, in one part)
  constexpr int PH = DP == 128 ? 2 : 1;
  constexpr int kChunks = DP / 64;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The 128-byte swizzle atoms need 1024-byte aligned tiles and the layout has no slack to
  // realign: refuse to run (before any barrier or allocation) if the base is not aligned.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) raise_status(p.status, ATTN_ERR_CUDA);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  // each group's running max and sum per row at the end of an item: [group][row] (m, l)
  float2* sStats = reinterpret_cast<float2*>(smem + L::kOffX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* q_full = bars;       // [2]: item i uses Q slot i % SQ
  uint64_t* q_empty = bars + 2;  // [2]
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  // Per buffer b: s_full (S(j) ready), p_full[b * 4 + g * 2 + h] (group g has written keys
  // [32h, 32h + 32) of its half of P(j)), pv_done
  // (PV(j) of both groups done: one commit from each PV issuer), for the tiles j with
  // j % 2 == b; phase k is tile 2k + b.
  uint64_t* s_full = v_empty + SV;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 8;
  uint64_t* o_free = pv_done + 2;
  uint64_t* drain = o_free + 1;
  uint64_t* o_staged = drain + 1;  // [Q slot]: the softmax warps have staged a tile-stored item's O
  uint64_t* drain2 = o_staged + 2;  // abort paths of the PV issuers (drain: the S issuer)
  uint64_t* drain3 = drain2 + 1;
  uint64_t* stats_ready = drain3 + 1;  // the softmax warps have written an item's (m, l)
  uint64_t* stats_free = stats_ready + 1;  // the epilogue warps have read them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  const uint32_t abort_flag = smem_u32(smem + L::kOffMisc + 4);  // CTA abort flag (shared)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + i, 1);
      mbar_init(q_empty + i, 1);
    }
    for (int i = 0; i < SK; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 2);  // one commit from each PV issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      for (int h = 0; h < 4; ++h) mbar_init(p_full + 4 * i + h, 4);  // one arrival per softmax warp of the group
      mbar_init(pv_done + i, 2);
    }
    mbar_init(o_free, 4);  // one arrival per epilogue warp
    mbar_init(drain, 1);
    mbar_init(drain2, 1);
    mbar_init(drain3, 1);
    mbar_init(o_staged, 4);
    mbar_init(o_staged + 1, 4);
    mbar_init(stats_ready, 8);
    mbar_init(stats_free, 4);
    abort_set(abort_flag, 0);
    wait_limit_set(abort_flag, p.wait_ns);
    mbar_init_fence();
  }
  if (warp == 8) tmem_alloc(tmem_slot, L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8 && warp < 12) {
    regs_dec<L::kRegsIo>();
    if (warp == 8) {
      // ================================================================ TMA producer
      // Two streams over the same sequence of key tiles, polled without blocking: K (with each
      // item's Q) and V.  Neither waits behind the other, so K tiles run ahead into their
      // deeper ring while V waits for its PV to free a slot.  Every barrier tested here cannot
      // complete its next phase before this thread issues another copy, so no phase is skipped.
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        TileCursor<CAUSAL, MODE> ck, cv;
        ck.start(p, n_items);
        cv.start(p, n_items);
        uint32_t nq = 0;      // Q tiles issued (one per item, slot item % 2)
        bool q_cur = false;   // the Q of ck's item has been issued
        bool ok = true;
        unsigned long long t_idle = 0;
        while (!ck.done || !cv.done) {
          bool progress = false;
          const uint32_t qs = nq % SQ;
          if (!ck.done && !q_cur && (nq < static_cast<uint32_t>(SQ) || mbar_test(q_empty + qs, ((nq / SQ) - 1) & 1))) {
            const FwdItem& it = ck.it;
            mbar_expect_tx(q_full + qs, L::kTileBytes);
            for (int c = 0; c < kChunks; ++c) {
              uint8_t* dst = sQ + qs * L::kTileBytes + c * L::kChunkBytes;
              if constexpr (VARLEN)
                tma_load_4d(dst, &tmQ, q_full + qs, c * 64, it.h, 0, it.seq_start + it.qt * kBM);
              else if constexpr (KV)
                tma_load_3d(dst, &tmQ, q_full + qs, c * 64, it.qt * kBM, it.b * p.Hkv + it.h);
              else
                tma_load_3d(dst, &tmQ, q_full + qs, c * 64, it.qt * kBM, it.b * p.Hq + it.h);
            }
            ++nq;
            q_cur = true;
            progress = true;
          }
          if (!ck.done && q_cur) {
            const uint32_t st = ck.t % SK;
            if (ck.t < static_cast<uint32_t>(SK) || mbar_test(k_empty + st, ((ck.t / SK) - 1) & 1)) {
              const FwdItem& it = ck.it;
              mbar_expect_tx(k_full + st, L::kTileBytes);
              for (int c = 0; c < kChunks; ++c) {
                uint8_t* dst = sK + st * L::kTileBytes + c * L::kChunkBytes;
                if constexpr (VARLEN)
                  tma_load_4d(dst, &tmK, k_full + st, c * 64, it.h, 1, it.seq_start + ck.j * kBN);
                else if constexpr (KV)
                  tma_load_3d(dst, &tmK, k_full + st, c * 64, (it.j0 + ck.j) * kBN, it.b * p.Hkv + it.h);
                else
                  tma_load_3d(dst, &tmK, k_full + st, c * 64, ck.j * kBN, it.b * p.Hkv + it.h / p.G);
              }
              ck.advance(p, n_items);
              if (ck.j == 0) q_cur = false;  // the next K belongs to a new item: its Q comes first
              progress = true;
            }
          }
          if (!cv.done) {
            const uint32_t st = cv.t % SV;
            if (cv.t < static_cast<uint32_t>(SV) || mbar_test(v_empty + st, ((cv.t / SV) - 1) & 1)) {
              const FwdItem& it = cv.it;
              mbar_expect_tx(v_full + st, L::kTileBytes);
              for (int c = 0; c < kChunks; ++c) {
                uint8_t* dst = sV + st * L::kTileBytes + c * L::kChunkBytes;
                if constexpr (VARLEN)
                  tma_load_4d(dst, &tmV, v_full + st, c * 64, it.h, 2, it.seq_start + cv.j * kBN);
                else if constexpr (KV)
                  tma_load_3d(dst, &tmV, v_full + st, c * 64, (it.j0 + cv.j) * kBN, it.b * p.Hkv + it.h);
                else
                  tma_load_3d(dst, &tmV, v_full + st, c * 64, cv.j * kBN, it.b * p.Hkv + it.h / p.G);
              }
              cv.advance(p, n_items);
              progress = true;
            }
          }
          if (progress) {
            t_idle = 0;
          } else {
            const unsigned long long now = globaltimer();
            if (t_idle == 0) t_idle = now;
            if (abort_read(abort_flag)) { ok = false; break; }
            if (now - t_idle > wait_limit(abort_flag)) {
              raise_status(p.status, ATTN_ERR_TIMEOUT);
              abort_set(abort_flag, 1);
              ok = false;
              break;
            }
          }
        }
        if (!ok || abort_read(abort_flag)) {
          // let the copies already issued land before the CTA's shared memory goes away
          for (uint32_t n = nq > static_cast<uint32_t>(SQ) ? nq - SQ : 0; n < nq; ++n)
            mbar_drain(q_full + n % SQ, (n / SQ) & 1);
          for (uint32_t j = ck.t > static_cast<uint32_t>(SK) ? ck.t - SK : 0; j < ck.t; ++j)
            mbar_drain(k_full + j % SK, (j / SK) & 1);
          for (uint32_t j = cv.t > static_cast<uint32_t>(SV) ? cv.t - SV : 0; j < cv.t; ++j)
            mbar_drain(v_full + j % SV, (j / SV) & 1);
        }
      }
      __syncwarp();
    } else {
      // ================================================================ MMA issuers
      // Three threads on three sub-partitions: warp 9 issues the S stream, warps 11 and 10 the PV
      // streams of groups 0 and 1 (one thread issues a tcgen05.mma about every 64 cycles at best,
      // and at about half that rate when busy warps share its sub-partition).  The streams touch
      // disjoint TMEM (S buffers; P_0 / O_0; P_1 / O_1) and are ordered only through the
      // softmax's barriers.
      if (lane == 0) {
        constexpr bool kB = Elem<T>::kBf16;
        constexpr uint32_t idS = idesc_f16(kB, false, false, 128, kBN);
        constexpr uint32_t idO = idesc_f16(kB, false, true, 128, DP);
        const uint64_t dQ = smem_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dV = smem_desc_sw128(smem_u32(sV), L::kChunkBytes, 1024);
        const bool s_side = warp == 9;
        const int g = warp == 11 ? 0 : 1;  // the PV issuer's group
        bool ok = true;
        uint32_t kv = 0;  // global key-tile counter (ring position and S/P/PV phases)
        uint32_t ic = 0;
        for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_items; ++k) {
          const int idx = cta_item<MODE>(k);
          if (idx >= n_items) continue;
          const FwdItem it = fwd_item<CAUSAL, MODE>(p, idx);
          if (!it.valid) continue;
          const int n = it.n_kv;
          const uint32_t qs = ic % SQ;
          if (s_side) {
            if (!mbar_wait(q_full + qs, (ic / SQ) & 1, abort_flag, p.status)) { ok = false; break; }
            for (int j = 0; j < n; ++j) {
              const uint32_t t = kv + j;
              // S buffer t % 2 holds P(t-2) until PV(t-2) has read it
              if (!mbar_wait(k_full + t % SK, (t / SK) & 1, abort_flag, p.status) ||
                  (t >= 2 && !mbar_wait(pv_done + (t & 1), ((t - 2) >> 1) & 1, abort_flag, p.status))) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t qx = dQ + ((qs * L::kTileBytes) >> 4);
              const uint64_t kx = dK + (((t % SK) * L::kTileBytes) >> 4);
              const uint32_t d = tmem + (t & 1) * 128;
#pragma unroll
              for (int ks = 0; ks < DP / 16; ++ks) {
                const uint32_t off = ((ks >> 2) * L::kChunkBytes + (ks & 3) * 32) >> 4;
                mma_ss(d, qx + off, kx + off, idS, ks > 0 ? 1u : 0u);
              }
              mma_commit(s_full + (t & 1));
              mma_commit(k_empty + t % SK);
              if (j == n - 1 && !tile_item(it)) mma_commit(q_empty + qs);
            }
          } else {
            for (int j = 0; j < n; ++j) {
              const uint32_t t = kv + j;
              const uint32_t b = t & 1;
              if (!mbar_wait(v_full + t % SV, (t / SV) & 1, abort_flag, p.status) ||
                  (j == 0 && ic > 0 && !mbar_wait(o_free, (ic - 1) & 1, abort_flag, p.status))) {
                ok = false;
                break;
              }
              const uint64_t vx = dV + (((t % SV) * L::kTileBytes) >> 4);
              const uint32_t acc0 = j == 0 ? 0u : 1u;
              // PV_g(t): O_g (+)= P_g(t) V[64g, 64g + 64), P_g over the first 32 columns of group
              // g's half of S buffer b (keys 2c, 2c+1 in column c), each of its PH parts issued as
              // soon as the softmax has written it
              const uint32_t pa = tmem + b * 128 + g * 64;
              const uint64_t vg = vx + ((g * 4 * 2048) >> 4);
#pragma unroll
              for (int h = 0; h < PH; ++h) {
                if (!mbar_wait(p_full + 4 * b + 2 * g + h, (t >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int k2 = 0; k2 < 4 / PH; ++k2) {
                  const int ks = (4 / PH) * h + k2;
                  mma_ts(tmem + L::kColO + g * DP, pa + ks * 8, vg + ((ks * 2048) >> 4), idO, ks > 0 ? 1u : acc0);
                }
              }
              if (!ok) break;
              mma_commit(pv_done + b);
              mma_commit(v_empty + t % SV);
            }
          }
          kv += n;
          ++ic;
        }
        if (!ok) {
          uint64_t* dr = s_side ? drain : (g == 0 ? drain2 : drain3);
          mma_commit(dr);  // every MMA this thread issued completes before this arrives
          mbar_drain(dr, 0);
        }
      }
      __syncwarp();
  }
  } else if (warp >= 12) {
    regs_dec<L::kRegsEpi>();
    // ================================================================ epilogue warpgroup
    // Per item, thread t (row t): both groups' (max, sum) from the softmax warps, then, once the
    // item's last PV has completed, O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / l over the whole
    // row, released from TMEM as soon as it is loaded (o_free), and LSE = m + ln l.  16-bit
    // tiles are staged in the item's Q slot and written out by this warpgroup's thread 0 with
    // tile stores; otherwise rows are stored here.
    const int row = threadIdx.x - 384;  // TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool storer = row == 0 && tile_out;  // issues the tile stores of staged items
    if (storer) tma_prefetch_desc(&tmO);
    uint32_t kv = 0, ic = 0, nt[2] = {0, 0};  // nt: per Q slot, items stored by tiles (o_staged phases)
    bool ok = true;
    for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_items; ++k) {
      const int idx = cta_item<MODE>(k);
      if (idx >= n_items) continue;
      const FwdItem it = fwd_item<CAUSAL, MODE>(p, idx);
      if (!it.valid) continue;
      const int q_row = it.qt * kBM + row;
      kv += it.n_kv;
      if (!mbar_wait_warp(stats_ready, ic & 1, abort_flag, p.status)) { ok = false; break; }
      const float2 s0 = sStats[row], s1 = sStats[128 + row];
      mbar_arrive_warp(stats_free);
      const float mr = fmaxf(s0.x, s1.x);
      const float a0 = (s0.x == -INFINITY) ? 0.f : ex2_approx(s0.x - mr);
      const float a1 = (s1.x == -INFINITY) ? 0.f : ex2_approx(s1.x - mr);
      const float l_all = s0.y * a0 + s1.y * a1;
      const float inv_l = (l_all > 0.f) ? 1.f / l_all : 0.f;
      const float c0 = a0 * inv_l, c1 = a1 * inv_l;  // weights of O_0 and O_1
      const uint32_t t_last = kv - 1;
      if (!mbar_wait_warp(pv_done + (t_last & 1), (t_last >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      const bool valid = q_row < (KV ? p.R : it.seq_len);
      size_t row_off;
      // a KV cache range writes its partial output in fp32 to its slice of the split buffer
      const size_t kv_row = KV ? (static_cast<size_t>(it.split) * p.B * p.Hkv + static_cast<size_t>(it.b) * p.Hkv + it.h) * p.R + q_row : 0;
      if constexpr (VARLEN)
        row_off = (static_cast<size_t>(it.seq_start + q_row) * p.Hq + it.h) * p.d;
      else if constexpr (KV)
        row_off = kv_row * p.d;
      else
        row_off = ((static_cast<size_t>(it.b) * p.Hq + it.h) * p.N + q_row) * p.d;
      const bool o_f32 = KV || p.out_f32;
      void* const o_base = KV ? static_cast<void*>(p.o_part) : p.o;
      const bool tile = tile_item(it);
      uint8_t* srow = sQ + (ic % SQ) * L::kTileBytes + row * 128;
#pragma unroll 1
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t r0[32], r1[32];
        tmem_ld32(tl + L::kColO + c * 32, r0);
        tmem_ld32(tl + L::kColO + DP + c * 32, r1);
        tmem_ld_wait();
        tmem_reg_fence(r0);
        tmem_reg_fence(r1);
        if (c == DP / 32 - 1) {
          tc_fence_before();
          mbar_arrive_warp(o_free);  // both accumulators are in registers: the next item may overwrite them
        }
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r0[i]) * c0 + __uint_as_float(r1[i]) * c1;
        if (tile) {
          // the item's Q slot, in the 128-byte swizzled layout of the output map's {64, 128} boxes:
          // column col lands in box col / 64, 16-byte granule (col % 64) / 8; rows and columns past
          // the tensor are clipped by the store
          uint8_t* brow = srow + ((c * 32) / 64) * L::kChunkBytes;
          const int gran0 = ((c * 32) % 64) / 8;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            v.x = Elem<T>::pack(o[8 * i + 0], o[8 * i + 1]);
            v.y = Elem<T>::pack(o[8 * i + 2], o[8 * i + 3]);
            v.z = Elem<T>::pack(o[8 * i + 4], o[8 * i + 5]);
            v.w = Elem<T>::pack(o[8 * i + 6], o[8 * i + 7]);
            const int gran = gran0 + i;
            *reinterpret_cast<uint4*>(brow + ((gran ^ (row & 7)) << 4)) = v;
          }
        } else {
          const int col0 = c * 32;
          if (valid && col0 < p.d) {
            const int ncol = min(32, p.d - col0);  // 16 or 32 (d is a multiple of 16)
            if (o_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(o_base) + row_off + col0);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (i * 4 < ncol) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(o_base) + row_off + col0);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if (i * 8 < ncol) {
                  uint4 v;
                  v.x = Elem<T>::pack(o[8 * i + 0], o[8 * i + 1]);
                  v.y = Elem<T>::pack(o[8 * i + 2], o[8 * i + 3]);
                  v.z = Elem<T>::pack(o[8 * i + 4], o[8 * i + 5]);
                  v.w = Elem<T>::pack(o[8 * i + 6], o[8 * i + 7]);
                  dst[i] = v;
                }
              }
            }
          }
        }
      }
      if (tile) {
        fence_async_smem();
        mbar_arrive_warp(o_staged + ic % SQ);
        // once all four warps have staged their rows: write the tile out, then free the Q slot
        // for the Q of the item after next
        const uint32_t qs = ic % SQ;
        if (storer) {
          if (!mbar_wait(o_staged + qs, nt[qs]++ & 1, abort_flag, p.status)) {
            ok = false;
          } else {
            for (int c = 0; c < kChunks; ++c) {
              const uint8_t* src = sQ + qs * L::kTileBytes + c * L::kChunkBytes;
              if constexpr (VARLEN)  // map {d, T, H} over the [T, H, d] output
                tma_store_3d(&tmO, src, c * 64, it.seq_start + it.qt * kBM, it.h);
              else
                tma_store_3d(&tmO, src, c * 64, it.qt * kBM, it.b * p.Hq + it.h);
            }
            bulk_commit();
            bulk_wait_read<0>();
            mbar_arrive(q_empty + qs);
          }
        }
        if (warp == 12) ok = __all_sync(0xffffffffu, ok);  // the warp leaves the loop together
      }
      if (valid && (KV || p.lse)) {
        const float lse = (mr + __log2f(l_all)) * 0.69314718055994531f;
        if constexpr (KV)
          p.lse_part[kv_row] = lse;
        else if constexpr (VARLEN)
          p.lse[static_cast<size_t>(it.h) * p.total_tokens + it.seq_start + q_row] = lse;
        else
          p.lse[(static_cast<size_t>(it.b) * p.Hq + it.h) * p.N + q_row] = lse;
      }
      ++ic;
    }
    if (storer) bulk_wait_all();  // the tile stores are complete before the CTA ends
  } else {
    regs_inc<L::kRegsSmx>();
    // ================================================================ softmax groups
    const int grp = warp >> 2;                // 0: key columns 0-63, 1: key columns 64-127
    const int row = threadIdx.x & 127;        // TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t tOg = tl + L::kColO + grp * DP;  // this group's accumulator O_g
    const float sl2 = p.scale_log2;
    uint32_t kv = 0, ic = 0;
    bool ok = true;
    for (int k = 0; ok && k * static_cast<int>(gridDim.x) < n_items; ++k) {
      const int idx = cta_item<MODE>(k);
      if (idx >= n_items) continue;
      const FwdItem it = fwd_item<CAUSAL, MODE>(p, idx);
      if (!it.valid) continue;
      const int q_row = it.qt * kBM + row;  // relative to the sequence (KV cache: to the R rows)
      // the last key this row sees: the diagonal under the causal mask, the sequence's end;
      // for a KV cache row (query q_row % Nq) the same, aligned to the cache's last Nq keys
      int last_key;
      if constexpr (KV)
        last_key = CAUSAL ? min(q_row % p.Nq + it.seq_len - p.Nq, it.seq_len - 1) : it.seq_len - 1;
      else
        last_key = CAUSAL ? min(q_row, it.seq_len - 1) : it.seq_len - 1;
      float m = -INFINITY, l = 0.f;  // this group's running max (log2 units) and sum
      for (int j = 0; j < it.n_kv; ++j) {
        const uint32_t t = kv + j;
        const int b = t & 1;
        if (!mbar_wait_warp(s_full + b, (t >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tS = tl + b * 128 + grp * 64;  // this group's 64 columns of S buffer b
        float s[64];
        {
          uint32_t r0[32], r1[32];
          tmem_ld32(tS, r0);
          tmem_ld32(tS + 32, r1);
          tmem_ld_wait();
          tmem_reg_fence(r0);
          tmem_reg_fence(r1);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(r0[i]);
            s[32 + i] = __uint_as_float(r1[i]);
          }
        }
        // keys key0 + c with c > lim are masked (past the diagonal, or past the sequence)
        const int key0 = (it.j0 + j) * kBN + grp * 64;
        const int lim = last_key - key0;
        if (lim < 63) {
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = c > lim ? -INFINITY : s[c];
        }
        // row max over this group's columns (3-input max, 4 chains)
        float m0 = max3f(s[0], s[1], s[2]), m1 = max3f(s[3], s[4], s[5]);
        float m2 = max3f(s[6], s[7], s[8]), m3 = max3f(s[9], s[10], s[11]);
#pragma unroll
        for (int c = 12; c < 60; c += 8) {
          m0 = max3f(m0, s[c], s[c + 1]);
          m1 = max3f(m1, s[c + 2], s[c + 3]);
          m2 = max3f(m2, s[c + 4], s[c + 5]);
          m3 = max3f(m3, s[c + 6], s[c + 7]);
        }
        m0 = max3f(m0, s[60], s[61]);
        m1 = max3f(m1, s[62], s[63]);
        const float mx2 = max3f(m0, m1, fmaxf(m2, m3)) * sl2;  // scale > 0: max commutes with it
        float alpha = 1.f;
        bool resc = false;
        if (mx2 > m + kRescaleLog2 || (m == -INFINITY && mx2 != -INFINITY)) {
          alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - mx2);
          resc = (j > 0) && (m != -INFINITY);
          m = mx2;
        }
        const float mb = (m == -INFINITY) ? 0.f : m;
        // O_g *= alpha (only when rescaling): O_g must hold PV(t-1) first, so wait for it.  Done
        // before the first part of P(t) is handed over: ahead of the exponentials when P goes
        // in two parts, after P's store when it goes in one.
        bool resc_ok = true;
        auto rescale_o = [&]() {
          if (!__any_sync(0xffffffffu, resc)) return;
          if (t > 0 && !mbar_wait_warp(pv_done + ((t - 1) & 1), ((t - 1) >> 1) & 1, abort_flag, p.status)) {
            resc_ok = false;
            return;
          }
          tc_fence_after();
          const float a = resc ? alpha : 1.f;
          uint32_t r[32];
#pragma unroll
          for (int c = 0; c < DP / 32; ++c) {
            tmem_ld32(tOg + c * 32, r);
            tmem_ld_wait();
            tmem_reg_fence(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * a);
            tmem_st32(tOg + c * 32, r);
          }
        };
        if constexpr (PH == 2) rescale_o();
        if (!resc_ok) {
          ok = false;
          break;
        }
        // exponentials in pairs: x = s * scale * log2(e) - m with one paired FMA, 2^x, the row
        // sum in 4 paired chains, and the 16-bit pair of P.  In tiles with no masked key the
        // pairs selected by kPolyPairs run on the FMA pipe, the rest on the special-function
        // unit; masked tiles use the latter only (exact zeros).
        const uint64_t scl = f2_pack(sl2, sl2), nmb = f2_pack(-mb, -mb);
        uint64_t acc[4];
        // P over the first 32 of this group's S columns, in PH parts of 64 / PH keys: each part
        // is stored and handed to its PV issuer while the next part's exponentials run.  The S
        // buffer takes S(t+2) only after PV(t) has read P.
        constexpr int PK = 64 / PH;  // keys per part
#pragma unroll
        for (int h = 0; h < PH; ++h) {
          uint32_t pk[PK / 2];
          if (lim >= 63) {
#pragma unroll
            for (int c = PK * h; c < PK * h + PK; c += 2) {
              const uint64_t x = f2_fma(f2_pack(s[c], s[c + 1]), scl, nmb);
              uint64_t e;
              if ((kPolyPairs >> ((c >> 1) & 7)) & 1) {
                e = exp2_fma2(x);
              } else {
                const float2 xf = f2_unpack(x);
                e = f2_pack(ex2_approx(xf.x), ex2_approx(xf.y));
              }
              acc[(c >> 1) & 3] = c < 8 ? e : f2_add(acc[(c >> 1) & 3], e);
              const float2 ef = f2_unpack(e);
              pk[(c / 2) % (PK / 2)] = Elem<T>::pack(ef.x, ef.y);
            }
          } else {
#pragma unroll
            for (int c = PK * h; c < PK * h + PK; c += 2) {
              const float2 xf = f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), scl, nmb));
              const float e0 = ex2_approx(xf.x), e1 = ex2_approx(xf.y);
              const uint64_t e = f2_pack(e0, e1);
              acc[(c >> 1) & 3] = c < 8 ? e : f2_add(acc[(c >> 1) & 3], e);
              pk[(c / 2) % (PK / 2)] = Elem<T>::pack(e0, e1);
            }
          }
          if constexpr (PH == 2) {
            tmem_st16(tS + 16 * h, pk);
          } else {
            tmem_st32(tS, pk);
            rescale_o();
            if (!resc_ok) break;
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive_warp(p_full + 4 * b + 2 * grp + h);
        }
        if (!resc_ok) {
          ok = false;
          break;
        }
        const float2 rs2 = f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])));
        l = l * alpha + (rs2.x + rs2.y);
      }
      if (!ok) break;
      kv += it.n_kv;
      // ---- hand the item's (max, sum) to the epilogue warpgroup, then straight on to the next
      // item: the epilogue combines O_0 and O_1 while this item's successor is computed
      if (ic >= 1 && !mbar_wait_warp(stats_free, (ic - 1) & 1, abort_flag, p.status)) { ok = false; break; }
      sStats[grp * 128 + row] = make_float2(m, l);
      mbar_arrive_warp(stats_ready);
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

template <typename T, int DP, bool CAUSAL, int MODE>
cudaError_t launch_fwd_tc_t(const FwdMaps& maps, const FwdParams& p, cudaStream_t stream) {
  using L = FwdLayout<DP, MODE>;
  auto kern = fwd_tc_kernel<T, DP, CAUSAL, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
  if (e != cudaSuccess) return e;
  // The in-kernel register split assumes the launch allocation; never launch otherwise.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != static_cast<int>(L::kLaunchRegs)) return cudaErrorInvalidConfiguration;
  const long heads = MODE == kModeVarlen ? static_cast<long>(p.Hq) * p.nseq
                     : MODE == kModeKv   ? static_cast<long>(p.B) * p.Hkv * p.n_splits
                                         : static_cast<long>(p.B) * p.Hq;
  const long items = heads * p.n_qtiles;
  if (items > 0x7fffffffL) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < sm_count() ? items : sm_count());
  kern<<<grid, L::kThreads, L::kSmemAlloc, stream>>>(maps.q, maps.k, maps.v, maps.o, p, static_cast<int>(items));
  return cudaGetLastError();
}

template <typename T, int DP>
cudaError_t launch_fwd_tc_dp(const FwdMaps& maps, const FwdParams& p, bool causal, int mode, cudaStream_t stream) {
  switch (mode) {
    case kModeVarlen:
      return causal ? launch_fwd_tc_t<T, DP, true, kModeVarlen>(maps, p, stream)
                    : launch_fwd_tc_t<T, DP, false, kModeVarlen>(maps, p, stream);
    case kModeKv:
      return causal ? launch_fwd_tc_t<T, DP, true, kModeKv>(maps, p, stream)
                    : launch_fwd_tc_t<T, DP, false, kModeKv>(maps, p, stream);
    default:
      return causal ? launch_fwd_tc_t<T, DP, true, kModeDense>(maps, p, stream)
                    : launch_fwd_tc_t<T, DP, false, kModeDense>(maps, p, stream);
  }
}

template <typename T>
cudaError_t launch_fwd_tc_dtype(const FwdMaps& maps, const FwdParams& p, bool causal, int mode,
                                cudaStream_t stream) {
  return p.d <= 64 ? launch_fwd_tc_dp<T, 64>(maps, p, causal, mode, stream)
                   : launch_fwd_tc_dp<T, 128>(maps, p, causal, mode, stream);
}

}  // namespace attn
