// bwd_tc.cuh -- tcgen05 backward for fp16 / bf16 (dQ, dK, dV), KV-stationary.
//
// The backward recomputes the scores from Q, K and the forward's LSE instead of storing them
// (FlashAttention-T review, FAQ 4; best practice 2 on keeping the backward fused).  With
// P_ij = exp(S_ij - LSE_i), dP_ij = dO_i . V_j, D_i = dO_i . O_i and dS_ij = P_ij (dP_ij - D_i):
//   dV_j = sum_i P_ij dO_i,   dK_j = scale sum_i dS_ij Q_i,   dQ_i = scale sum_j dS_ij K_j,
// where i runs over every query row of every query head of the kv head's GQA group.
//
// One CTA owns one 128-key tile of one (batch, kv head): K and V stay in shared memory, and
// the CTA walks (query head of the group) x (query tile at or after the key tile when causal).
// Per query tile, in TMEM (128 lanes = the 128 keys, except dQ whose lanes are queries):
//   columns [0,128)     S^T = K Q^T, then P^T (hi and lo 16-bit halves, see below)
//   columns [128,256)   dP^T = V dO^T, then dQ_t = dS K
//   columns [256,256+d) dV += P^T dO   (accumulates over every iteration)
//   columns [256+d, ..) dK += dS^T Q   (accumulates over every iteration)
// P and dS are split into hi = round16(x) and lo = round16(x - hi) and both halves go through
// the MMAs, so the gradient contractions see ~16 significant bits of P and dS instead of 8
// (bf16) or 11 (fp16): rounding P or dS once to bf16 alone already moves causal GQA gradients
// by ~1e-2.  P^T hi/lo stays in TMEM (A operand of the dV MMA); dS^T hi/lo goes to shared
// memory, where it is read K-major for dK and, as dS, MN-major for dQ.
//
// 512 threads, four warpgroups with a register split:
//   WG0, WG1  elementwise (two warps per TMEM lane quadrant, each on half of the 128 query
//             columns): phase 1 turns S^T into P^T (hi/lo, back into TMEM), phase 2 turns dP^T
//             into dS^T (hi/lo, into shared memory), each in two parts of 32 columns handed
//             over separately so the dV / dK MMAs on the first part start early.  The next
//             tile's LSE and D are prefetched.
//   WG2       moves dQ_t from TMEM through shared memory into the fp32 workspace (TMA tile
//             reductions; in key-tile order when deterministic) and writes dK, dV at the end.
//   WG3       warp 12: TMA producer and TMEM allocator; warps 13 and 14: MMA issuers.
// Two MMA streams: warp 13 issues S^T, dP^T, dV (hi, lo) per query tile, warp 14 dK (hi, lo)
// then dQ (hi, lo) once dS is written.  The next tile's S^T waits only for dV to have read P^T
// and for its Q; its dP^T waits for the dQ readout.  Q and dO have separate ring slots,
// released after the last MMA that reads each (dK, dV).
#pragma once
#include "fwd_tc.cuh"

namespace attn {

template <int DP>
struct BwdLayout {
  static constexpr int kQStages = DP == 128 ? 1 : 2;
  static constexpr int kChunkBytes = 128 * 128;
  static constexpr int kTileBytes = (DP / 64) * kChunkBytes;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;                 // kQStages tiles
  static constexpr int kOffdO = kOffQ + kQStages * kTileBytes;     // kQStages tiles
  static constexpr int kOffdSh = kOffdO + kQStages * kTileBytes;   // dS^T hi [128 keys x 128 queries]
  static constexpr int kOffdSl = kOffdSh + 2 * kChunkBytes;        // dS^T lo
  // dQ staging for the tile reductions: fp32 {32 columns, 128 rows} boxes of 16 KB.  Columns
  // 0-63 have a buffer of their own; columns 64-127 (DP = 128) go through the dS lo area.
  static constexpr int kOwnStageChunks = 2;
  static constexpr int kLoStageChunks = DP / 32 - kOwnStageChunks;
  static constexpr int kOffStage = kOffdSl + 2 * kChunkBytes;
  static constexpr int kOffRow = kOffStage + kOwnStageChunks * kChunkBytes;  // LSE*log2e and D, 2 buffers each
  static constexpr int kOffBar = kOffRow + 4 * 128 * 4;
  // kv_full, q_full[QS], q_empty[QS], do_full[QS], do_empty[QS], s_full, dp_full, p_full[2],
  // dv_done, ds_full[2], dsl_free, stage_free, dq_full, dq_free, dkdv_done, rows_ready,
  // stage_full, drain, drain2
  static constexpr int kNumBars = 1 + 4 * kQStages + 16;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem base, abort flag, wait limit (u64)
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kBytes;  // the dynamic shared memory starts 1024-byte aligned
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory over the per-CTA limit");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColdP = 128, kColdV = 256, kColdK = 256 + DP;
  static constexpr uint32_t kColdQ = kColdP;
  static constexpr int kThreads = 512;
  static constexpr int kEwThreads = 256;  // warpgroups 0 and 1
  // launch 128 registers per thread; 2 * kRegsEw + kRegsDq + kRegsIo == 4 * kLaunchRegs
  static constexpr uint32_t kLaunchRegs = 128, kRegsEw = 184, kRegsDq = 88, kRegsIo = 56;
  static_assert(2 * kRegsEw + kRegsDq + kRegsIo == 4 * kLaunchRegs, "register split must match the launch");
};

// Splits x into hi = round(x) and lo = round(x - hi) in the 16-bit type T, packed in pairs.
template <typename T>
__device__ __forceinline__ void split_pack(float a, float b, uint32_t& hi, uint32_t& lo);
template <>
__device__ __forceinline__ void split_pack<__nv_bfloat16>(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const uint32_t hb = *reinterpret_cast<const uint32_t*>(&h);
  // hi back in fp32 (a bf16 is the top half of an fp32), then x - hi for both with one paired
  // FMA; the difference is exact
  const uint64_t hf = f2_pack(__uint_as_float(hb << 16), __uint_as_float(hb & 0xffff0000u));
  const float2 r = f2_unpack(f2_fma(hf, f2_pack(-1.f, -1.f), f2_pack(a, b)));
  const __nv_bfloat162 l = __floats2bfloat162_rn(r.x, r.y);
  hi = hb;
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
template <>
__device__ __forceinline__ void split_pack<__half>(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const float2 r = f2_unpack(f2_fma(f2_pack(hf.x, hf.y), f2_pack(-1.f, -1.f), f2_pack(a, b)));
  const __half2 l = __floats2half2_rn(r.x, r.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

template <typename T, int DP, bool CAUSAL>
__global__ void __launch_bounds__(512, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmAcc, const BwdParams p) {
  using L = BwdLayout<DP>;
  constexpr int QS = L::kQStages;
  constexpr int kChunks = DP / 64;
  constexpr int kEw = L::kEwThreads;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The 128-byte swizzle atoms need 1024-byte aligned tiles and the layout has no slack to
  // realign: refuse to run (before any barrier or allocation) if the base is not aligned.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) raise_status(p.status, ATTN_ERR_CUDA);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sK = smem + L::kOffK;
  uint8_t* sV = smem + L::kOffV;
  uint8_t* sQ = smem + L::kOffQ;
  uint8_t* sdO = smem + L::kOffdO;
  uint8_t* sdSh = smem + L::kOffdSh;
  uint8_t* sdSl = smem + L::kOffdSl;
  uint8_t* sStage = smem + L::kOffStage;
  float* sLse = reinterpret_cast<float*>(smem + L::kOffRow);  // [2][128]
  float* sD = sLse + 256;                                       // [2][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + QS;
  uint64_t* do_full = q_empty + QS;
  uint64_t* do_empty = do_full + QS;
  uint64_t* s_full = do_empty + QS;
  uint64_t* dp_full = s_full + 1;
  // p_full[h]: every elementwise warp has written P^T for the first (h = 0) or last (h = 1) 32 of
  // its 64 query columns, i.e. the dV k-steps {0, 1, 4, 5} or {2, 3, 6, 7}
  uint64_t* p_full = dp_full + 1;
  uint64_t* dv_done = p_full + 2;
  // ds_full[h]: every elementwise warp has written dS^T for the first (h = 0) or last (h = 1) 32
  // of its 64 query columns, i.e. the dK k-steps {0, 1, 4, 5} or {2, 3, 6, 7}
  uint64_t* ds_full = dv_done + 1;
  // the dS lo area also stages dQ columns 64-127: free once the tile's reduction has read it
  uint64_t* dsl_free = ds_full + 2;
  uint64_t* stage_free = dsl_free + 1;  // the reductions have read the own staging buffer
  uint64_t* dq_full = stage_free + 1;
  uint64_t* dq_free = dq_full + 1;
  uint64_t* dkdv_done = dq_free + 1;
  uint64_t* rows_ready = dkdv_done + 1;  // the 128 row terms (LSE, D) of the current tile are in smem
  uint64_t* stage_full = rows_ready + 1;  // the read-out warps have staged the dQ tile
  uint64_t* drain = stage_full + 1;   // abort path of issuer 13
  uint64_t* drain2 = drain + 1;        // abort path of issuer 14
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  const uint32_t abort_flag = smem_u32(smem + L::kOffMisc + 4);  // CTA abort flag (shared)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Blocks are dispatched in linear order (x fastest): every (batch, kv head) of key tile 0,
  // the heaviest under the causal mask, then key tile 1, ...; each SM that frees up takes the
  // heaviest tile left, which keeps the causal tail short.
  // Dense: x = batch * kv head.  Varlen: x = sequence * head; the sequence is the diagonal block
  // [seq_start, seq_start + seq_len) of a B = 1, N = total_tokens problem (G = 1).
  const int kt = blockIdx.y;
  // kv head (row block), its first query head; the sequence's start, its query and key counts
  int hkv, hq0, seq_start = 0, seq_len = p.N, kv_len = p.Nk;
  if (p.cu_seqlens) {
    const int s = blockIdx.x / p.Hkv, hh = blockIdx.x % p.Hkv;
    const int c0 = p.cu_seqlens[s], c1 = p.cu_seqlens[s + 1];
    const bool bad = c0 < 0 || c1 < c0 || c1 > p.N || c1 - c0 > p.max_seqlen || (s == 0 && c0 != 0) ||
                     (s == p.nseq - 1 && c1 != p.N);
    if (bad) {
      if (threadIdx.x == 0 && kt == 0 && hh == 0) raise_status(p.status, ATTN_ERR_DEVICE_INPUT);
      return;  // the whole CTA, before any barrier or allocation
    }
    seq_start = c0;
    seq_len = c1 - c0;
    kv_len = seq_len;
    hkv = hh;
    hq0 = hh * p.G;
  } else {
    const int b = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;
    hkv = b * p.Hkv + g;
    hq0 = b * p.Hq + g * p.G;
  }
  const int N = p.N;
  const int n_q = (seq_len + kBM - 1) / kBM;
  if (kt * kBN >= kv_len) return;  // a key tile past this sequence's end (varlen): the whole CTA
  // causal: query i sees key j iff j <= i + off (off = 0 for self-attention; cross-attention
  // aligns the queries with the last keys), so the first query tile that sees key tile kt is
  // the one holding query kt * 128 - off; every key tile is seen by the last query
  const int off = kv_len - seq_len;
  const int qt0 = CAUSAL ? max(0, (kt * kBN - off) >= 0 ? (kt * kBN - off) / kBM : 0) : 0;
  const int per_head = n_q - qt0;
  const int n_it = p.G * per_head;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < QS; ++i) {
      mbar_init(q_full + i, 1);
      mbar_init(q_empty + i, 1);
      mbar_init(do_full + i, 1);
      mbar_init(do_empty + i, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, kEw / 32);  // one arrival per warp
    mbar_init(p_full + 1, kEw / 32);
    mbar_init(dv_done, 1);
    mbar_init(ds_full, kEw / 32);
    mbar_init(ds_full + 1, kEw / 32);
    mbar_init(dsl_free, 1);
    mbar_init(stage_free, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);
    mbar_init(dkdv_done, 2);
    mbar_init(rows_ready, kEw / 32);
    mbar_init(stage_full, 4);
    mbar_init(drain, 1);
    mbar_init(drain2, 1);
    abort_set(abort_flag, 0);
    wait_limit_set(abort_flag, p.wait_ns);
    mbar_init_fence();
  }
  if (warp == 12) tmem_alloc(tmem_slot, L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 12) {
    regs_dec<L::kRegsIo>();
    if (warp == 12 && lane == 0) {
      // ============================================================== TMA producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_expect_tx(kv_full, 2 * L::kTileBytes);
      for (int c = 0; c < kChunks; ++c) {
        tma_load_3d(sK + c * L::kChunkBytes, &tmK, kv_full, c * 64, seq_start + kt * kBN, hkv);
        tma_load_3d(sV + c * L::kChunkBytes, &tmV, kv_full, c * 64, seq_start + kt * kBN, hkv);
      }
      int nq_issued = 0, ndo_issued = 0;
      for (int it = 0; it < n_it; ++it) {
        const int hq = hq0 + it / per_head, qt = qt0 + it % per_head;
        const int st = it % QS;
        const uint32_t ph = ((it / QS) - 1) & 1;
        // dO first: its slot frees earlier (after dV)
        if (it >= QS && !mbar_wait(do_empty + st, ph, abort_flag, p.status)) break;
        mbar_expect_tx(do_full + st, L::kTileBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_3d(sdO + st * L::kTileBytes + c * L::kChunkBytes, &tmdO, do_full + st, c * 64,
                      seq_start + qt * kBM, hq);
        ndo_issued = it + 1;
        if (it >= QS && !mbar_wait(q_empty + st, ph, abort_flag, p.status)) break;
        mbar_expect_tx(q_full + st, L::kTileBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_3d(sQ + st * L::kTileBytes + c * L::kChunkBytes, &tmQ, q_full + st, c * 64,
                      seq_start + qt * kBM, hq);
        nq_issued = it + 1;
      }
      if (abort_read(abort_flag)) {
        mbar_drain(kv_full, 0);
        for (int it = max(0, nq_issued - QS); it < nq_issued; ++it) mbar_drain(q_full + it % QS, (it / QS) & 1);
        for (int it = max(0, ndo_issued - QS); it < ndo_issued; ++it)
          mbar_drain(do_full + it % QS, (it / QS) & 1);
      }
    } else if ((warp == 13 || warp == 14) && lane == 0) {
      // ============================================================== MMA issuers
      // warp 13: S^T(t), dP^T(t), dV(t); warp 14: dK(t), then dQ(t), once dS(t) is written.  One
      // thread feeds the tensor core at most one 128 x 128 x 16 MMA per ~64 cycles, and slower
      // when busy warps share its sub-partition; with two issuers S^T(t+1) goes in as soon as
      // Q(t+1) has landed instead of behind the issue of dQ(t).
      constexpr bool kB = Elem<T>::kBf16;
      constexpr uint32_t idSS = idesc_f16(kB, false, false, 128, 128);  // S^T, dP^T
      constexpr uint32_t idKD = idesc_f16(kB, false, true, 128, DP);    // dV, dK: B MN-major
      constexpr uint32_t idQ = idesc_f16(kB, true, true, 128, DP);      // dQ: A and B MN-major
      // descriptors built once; a k-step adds its byte offset >> 4 to the start-address field
      const uint64_t dK_k = smem_desc_sw128(smem_u32(sK), 16, 1024);               // K, K-major
      const uint64_t dV_k = smem_desc_sw128(smem_u32(sV), 16, 1024);               // V, K-major
      const uint64_t dK_mn = smem_desc_sw128(smem_u32(sK), L::kChunkBytes, 1024);  // K, MN-major
      const uint64_t dQ_k = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dQ_mn = smem_desc_sw128(smem_u32(sQ), L::kChunkBytes, 1024);
      const uint64_t ddO_k = smem_desc_sw128(smem_u32(sdO), 16, 1024);
      const uint64_t ddO_mn = smem_desc_sw128(smem_u32(sdO), L::kChunkBytes, 1024);
      const uint64_t dSh_k = smem_desc_sw128(smem_u32(sdSh), 16, 1024);
      const uint64_t dSl_k = smem_desc_sw128(smem_u32(sdSl), 16, 1024);
      const uint64_t dSh_mn = smem_desc_sw128(smem_u32(sdSh), L::kChunkBytes, 1024);
      const uint64_t dSl_mn = smem_desc_sw128(smem_u32(sdSl), L::kChunkBytes, 1024);
      constexpr uint32_t kStage16 = L::kTileBytes >> 4;
      bool ok = mbar_wait(kv_full, 0, abort_flag, p.status);
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it % QS;
        const uint32_t ph = (it / QS) & 1;
        if (warp == 13) {
          // ---- S^T = K Q^T (needs Q and the S columns: dV of the previous tile has read P^T)
          if (!mbar_wait(q_full + st, ph, abort_flag, p.status)) { ok = false; break; }
          if (it >= 1 && !mbar_wait(dv_done, (it - 1) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          {
            const uint64_t a = opaque(dK_k), bq = opaque(dQ_k + st * kStage16);
#pragma unroll
            for (int ks = 0; ks < DP / 16; ++ks) {
              const uint32_t off = ((ks >> 2) * L::kChunkBytes + (ks & 3) * 32) >> 4;
              mma_ss(tmem + L::kColS, a + off, bq + off, idSS, ks > 0 ? 1u : 0u);
            }
          }
          mma_commit(s_full);
          // ---- dP^T = V dO^T (needs dO and the dP columns: dQ of the previous tile read out,
          // which also means its dK and dQ MMAs have completed)
          if (!mbar_wait(do_full + st, ph, abort_flag, p.status)) { ok = false; break; }
          if (it >= 1 && !mbar_wait(dq_free, (it - 1) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          {
            const uint64_t a = opaque(dV_k), bo = opaque(ddO_k + st * kStage16);
#pragma unroll
            for (int ks = 0; ks < DP / 16; ++ks) {
              const uint32_t off = ((ks >> 2) * L::kChunkBytes + (ks & 3) * 32) >> 4;
              mma_ss(tmem + L::kColdP, a + off, bo + off, idSS, ks > 0 ? 1u : 0u);
            }
          }
          mma_commit(dp_full);
          // ---- dV += P^T dO; P^T hi/lo in TMEM: the 16 queries of k-step ks sit in the 32-column
          // group ks/2 (hi in its first 16 columns, lo in the last 16), 8 columns per k-step
          // in two parts, each as soon as the elementwise warps have written it: k-steps
          // {0, 1, 4, 5} (the first 32 columns of each warp's half), then {2, 3, 6, 7}
          {
            const uint64_t bo = opaque(ddO_mn + st * kStage16);
            const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (!mbar_wait(p_full + h, it & 1, abort_flag, p.status)) { ok = false; break; }
              tc_fence_after();
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int ks = (j >> 1) * 4 + 2 * h + (j & 1);
                const uint32_t acol = L::kColS + (ks >> 1) * 32 + (ks & 1) * 8;
                const uint64_t bd = bo + ((ks * 2048) >> 4);
                mma_ts(tmem + L::kColdV, tmem + acol, bd, idKD, (h > 0 || j > 0) ? 1u : acc0);
                mma_ts(tmem + L::kColdV, tmem + acol + 16, bd, idKD, 1u);
              }
            }
            if (!ok) break;
          }
          mma_commit(dv_done);
          mma_commit(do_empty + st);
        } else {
          // ---- dK += dS^T Q (hi, lo)
          // in two parts, each as soon as the elementwise warps have written its 64 queries:
          // k-steps {0, 1, 4, 5} (the first 32 columns of each warp's half), then {2, 3, 6, 7}
          {
            const uint64_t ah = opaque(dSh_k), al = opaque(dSl_k), bq = opaque(dQ_mn + st * kStage16);
            const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (!mbar_wait(ds_full + h, it & 1, abort_flag, p.status)) { ok = false; break; }
              tc_fence_after();
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int ks = (j >> 1) * 4 + 2 * h + (j & 1);
                const uint32_t a_off = ((ks >> 2) * L::kChunkBytes + (ks & 3) * 32) >> 4;
                const uint64_t bd = bq + ((ks * 2048) >> 4);
                mma_ss(tmem + L::kColdK, ah + a_off, bd, idKD, (h > 0 || j > 0) ? 1u : acc0);
                mma_ss(tmem + L::kColdK, al + a_off, bd, idKD, 1u);
              }
            }
            if (!ok) break;
          }
          mma_commit(q_empty + st);
          // ---- dQ_t = dS K (hi, lo), dS read MN-major from the dS^T tiles, into the dP columns
          {
            const uint64_t ah = opaque(dSh_mn), al = opaque(dSl_mn), bk = opaque(dK_mn);
#pragma unroll
            for (int ks = 0; ks < kBN / 16; ++ks) {
              const uint32_t off = (ks * 2048) >> 4;
              mma_ss(tmem + L::kColdQ, ah + off, bk + off, idQ, ks > 0 ? 1u : 0u);
              mma_ss(tmem + L::kColdQ, al + off, bk + off, idQ, 1u);
            }
          }
          mma_commit(dq_full);
        }
      }
      uint64_t* dr = warp == 13 ? drain : drain2;
      if (ok) {
        mma_commit(dkdv_done);  // one commit from each issuer after its last MMA
      } else {
        mma_commit(dr);
        mbar_drain(dr, 0);
      }
    }
    __syncwarp();
  } else if (warp >= 8) {
    regs_dec<L::kRegsDq>();
    // ================================================================ dQ readout, dK/dV out
    const int quad = warp & 3;
    const int t = quad * 32 + lane;  // TMEM lane: query row of dQ, key row of dK / dV
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    bool ok = true;
    // dQ_t goes from TMEM through shared memory into the fp32 accumulator by tile reductions,
    // chunk c of 32 columns in the 128-byte swizzled layout of the accumulator map's {32, 128}
    // box: chunks 0 and 1 in their own staging buffer, chunks 2 and 3 (DP = 128) in the dS lo
    // area, free once the dK and dQ MMAs that read it have completed (dq_full).  The TMEM
    // columns are released as soon as they are loaded, and the dS lo chunks are reduced first,
    // so the elementwise warps may write the next dS lo as soon as they have been read.  Rows
    // of the tile past the sequence hold exact zeros (P = 0 there), so they add nothing; rows
    // past the accumulator are skipped by the map.
    for (int it = 0; it < n_it; ++it) {
      const int qt = qt0 + it % per_head;
      const int row0 = static_cast<int>(static_cast<size_t>(hq0 + it / per_head) * N + seq_start) + qt * kBM;
      if (!mbar_wait_warp(dq_full, it & 1, abort_flag, p.status)) { ok = false; break; }
      if (it >= 1 && !mbar_wait_warp(stage_free, (it - 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      // chunk c + 1 is loaded from TMEM while chunk c is written to its staging buffer, and the
      // dQ columns are released (dq_free, which the next dP^T waits for) once the last is loaded
      uint32_t ra[32], rb[32];
      tmem_ld32(tl + L::kColdQ, ra);
      tmem_ld_wait();
      tmem_reg_fence(ra);
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t(&r)[32] = (c & 1) ? rb : ra;
        uint32_t(&nx)[32] = (c & 1) ? ra : rb;
        if (c + 1 < DP / 32) {
          tmem_ld32(tl + L::kColdQ + (c + 1) * 32, nx);
        } else {
          tc_fence_before();
          mbar_arrive_warp(dq_free);  // the dQ columns may be overwritten once everything is loaded
        }
        uint8_t* row = (c < L::kOwnStageChunks ? sStage + c * 16384 : sdSl + (c - L::kOwnStageChunks) * 16384) + t * 128;
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<uint4*>(row + ((g ^ (t & 7)) << 4)) = make_uint4(r[4 * g], r[4 * g + 1], r[4 * g + 2], r[4 * g + 3]);
        if (c + 1 < DP / 32) {
          tmem_ld_wait();
          tmem_reg_fence(nx);
        }
      }
      fence_async_smem();
      mbar_arrive_warp(stage_full);
      if (warp == 8 && lane == 0) {
        if (!mbar_wait(stage_full, it & 1, abort_flag, p.status)) { ok = false; }
        // deterministic: key tile kt adds into this dQ tile after key tiles 0 .. kt-1 (the
        // tiles of the same sequence that also reach it, launched before this CTA)
        if (ok && p.deterministic) {
          if (wait_turn(p.dq_turn + row0, kt, abort_flag, p.status))
            fence_async_global();  // the reductions below come after the turn was seen
          else
            ok = false;
        }
        if (ok) {
          if (L::kLoStageChunks > 0) {
            for (int c = L::kOwnStageChunks; c < DP / 32; ++c)
              if (c * 32 < p.d) tma_reduce_add_2d(&tmAcc, sdSl + (c - L::kOwnStageChunks) * 16384, c * 32, row0);
            bulk_commit();
          }
          for (int c = 0; c < L::kOwnStageChunks; ++c)
            if (c * 32 < p.d) tma_reduce_add_2d(&tmAcc, sStage + c * 16384, c * 32, row0);
          bulk_commit();
          if (L::kLoStageChunks > 0) {
            bulk_wait_read<1>();     // every group but the last: the dS lo chunks
            mbar_arrive(dsl_free);   // the dS lo area may take the next tile's dS lo
          }
          bulk_wait_read<0>();
          mbar_arrive(stage_free);
          if (p.deterministic) {
            bulk_wait_all();       // the reductions have been performed ...
            fence_async_global();  // ... before the turn passes to key tile kt + 1
            red_release_gpu_add(p.dq_turn + row0, 1);
          }
        }
      }
      __syncwarp();
      if (!__all_sync(0xffffffffu, ok)) break;
    }
    if (warp == 8 && lane == 0) bulk_wait_all();  // the reductions complete before the CTA ends
    // ---- epilogue: dK (scaled) and dV rows of this key tile
    if (ok && mbar_wait_warp(dkdv_done, 0, abort_flag, p.status)) {
      tc_fence_after();
      const int key = kt * kBN + t;
      const long long kofs = hkv * p.lay_dkv.head + (seq_start + key) * p.lay_dkv.row;  // row start
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? L::kColdK : L::kColdV;
        const float mul = which == 0 ? p.scale : 1.f;
        void* out = which == 0 ? p.dk : p.dv;
        uint32_t r[32];
#pragma unroll 1
        for (int c = 0; c < DP / 32; ++c) {
          tmem_ld32(tl + col + c * 32, r);
          tmem_ld_wait();
          tmem_reg_fence(r);
          if (key < kv_len && c * 32 < p.d) {
            const int ncol = min(32, p.d - c * 32);
            if (p.out_f32) {
              float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(out) + kofs + c * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (i * 4 < ncol)
                  o4[i] = make_float4(__uint_as_float(r[4 * i]) * mul, __uint_as_float(r[4 * i + 1]) * mul,
                                      __uint_as_float(r[4 * i + 2]) * mul, __uint_as_float(r[4 * i + 3]) * mul);
            } else {
              uint4* o4 = reinterpret_cast<uint4*>(static_cast<T*>(out) + kofs + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (i * 8 < ncol) {
                  uint4 v;
                  v.x = Elem<T>::pack(__uint_as_float(r[8 * i + 0]) * mul, __uint_as_float(r[8 * i + 1]) * mul);
                  v.y = Elem<T>::pack(__uint_as_float(r[8 * i + 2]) * mul, __uint_as_float(r[8 * i + 3]) * mul);
                  v.z = Elem<T>::pack(__uint_as_float(r[8 * i + 4]) * mul, __uint_as_float(r[8 * i + 5]) * mul);
                  v.w = Elem<T>::pack(__uint_as_float(r[8 * i + 6]) * mul, __uint_as_float(r[8 * i + 7]) * mul);
                  o4[i] = v;
                }
            }
          }
        }
      }
    }
  } else {
    regs_inc<L::kRegsEw>();
    // ================================================================ elementwise warps 0-7
    const int quad = warp & 3;                // TMEM lane quadrant
    const int half = warp >> 2;               // query columns [64*half, 64*half+64)
    const int t = quad * 32 + lane;           // TMEM lane: key row
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int key = kt * kBN + t;
    const bool key_ok = key < kv_len;
    const float sl2 = p.scale_log2;
    // The next tile's row terms are loaded at the end of the current tile and used only when they
    // are written to shared memory at the start of the next one, ahead of the wait for its S^T.
    // Rows past the sequence read its last row and are replaced there.
    float lse_next = 0.f, d_next = 0.f;
    bool row_next = false;
    auto load_rows = [&](int it) {
      if (threadIdx.x < 128 && it < n_it) {
        const int qt = qt0 + it % per_head;
        const size_t row_base = static_cast<size_t>(hq0 + it / per_head) * N + seq_start;
        const int q = qt * kBM + threadIdx.x;
        row_next = q < seq_len;
        const size_t r = row_base + (row_next ? q : seq_len - 1);
        lse_next = p.lse[r];
        d_next = p.delta[r];
      }
    };
    load_rows(0);
    for (int it = 0; it < n_it; ++it) {
      const int qt = qt0 + it % per_head;
      float* lse_buf = sLse + (it & 1) * 128;
      float* d_buf = sD + (it & 1) * 128;
      // stored negated, so each element needs one paired FMA (and one paired add) against them
      if (threadIdx.x < 128) {
        lse_buf[threadIdx.x] = row_next ? -(lse_next * 1.4426950408889634f) : -INFINITY;
        d_buf[threadIdx.x] = row_next ? -d_next : 0.f;
      }
      mbar_arrive_warp(rows_ready);
      if (!mbar_wait_warp(rows_ready, it & 1, abort_flag, p.status)) break;
      // ---- phase 1: P^T = exp2(S^T * scale * log2e - LSE * log2e), hi/lo back into TMEM
      if (!mbar_wait_warp(s_full, it & 1, abort_flag, p.status)) break;
      tc_fence_after();
      float pv[64];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(tl + L::kColS + half * 64, r0);
        tmem_ld32(tl + L::kColS + half * 64 + 32, r1);
        tmem_ld_wait();
        tmem_reg_fence(r0);
        tmem_reg_fence(r1);
        // P = 2^(S scale log2e - LSE log2e): the row terms as float4 from shared memory, the
        // argument as one paired FMA per two queries.  In two parts of 32 query columns, each
        // written back to TMEM and handed over (p_full[cc]) before the next is computed, so the
        // first half of the dV MMAs runs while the second part is computed.
        const float4* nl4 = reinterpret_cast<const float4*>(lse_buf + half * 64);
        const uint64_t scl = f2_pack(sl2, sl2);
        // queries q < key - off are masked under causal (only tiles on the diagonal have any; a
        // query row that sees no key at all has every column masked), and keys past the
        // sequence give P = 0: the selects run only where a thread has such columns
        // columns c < lim are masked (a key past the sequence: all 64)
        const int lim = !key_ok ? 64 : (CAUSAL ? key - off - qt * kBM - half * 64 : -1);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t(&r)[32] = cc == 0 ? r0 : r1;
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 nl = nl4[8 * cc + j4];
            const int i = 32 * cc + 4 * j4;
            const float2 x01 = f2_unpack(f2_fma(f2_pack(__uint_as_float(r[4 * j4]), __uint_as_float(r[4 * j4 + 1])), scl,
                                                f2_pack(nl.x, nl.y)));
            const float2 x23 = f2_unpack(f2_fma(f2_pack(__uint_as_float(r[4 * j4 + 2]), __uint_as_float(r[4 * j4 + 3])),
                                                scl, f2_pack(nl.z, nl.w)));
            pv[i] = ex2_approx(x01.x);
            pv[i + 1] = ex2_approx(x01.y);
            pv[i + 2] = ex2_approx(x23.x);
            pv[i + 3] = ex2_approx(x23.y);
          }
          if (lim > 32 * cc) {
#pragma unroll
            for (int i = 32 * cc; i < 32 * cc + 32; ++i) pv[i] = i < lim ? 0.f : pv[i];
          }
          uint32_t ph[16], pl[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) split_pack<T>(pv[cc * 32 + 2 * i], pv[cc * 32 + 2 * i + 1], ph[i], pl[i]);
          tmem_st16(tl + L::kColS + half * 64 + cc * 32, ph);
          tmem_st16(tl + L::kColS + half * 64 + cc * 32 + 16, pl);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive_warp(p_full + cc);
        }
      }
      // ---- phase 2: dS^T = P^T (dP^T - D), hi/lo into shared memory.  dp_full also means the
      // previous tile's dK and dQ MMAs have completed (dP^T is issued after its dQ read-out), so
      // the dS hi area is free; the dS lo area waits for the reductions of the dQ chunks staged in it.
      if (!mbar_wait_warp(dp_full, it & 1, abort_flag, p.status)) break;
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld32(tl + L::kColdP + half * 64, r0);
      tmem_ld32(tl + L::kColdP + half * 64 + 32, r1);
      tmem_ld_wait();
      tmem_reg_fence(r0);
      tmem_reg_fence(r1);
      tc_fence_before();  // the dP columns are consumed (the dQ MMA may overwrite them)
      // dS = P (dP - D), with D (stored negated) read as float4, split hi/lo and written in two
      // parts of 32 query columns, each handed over (ds_full[h]) as soon as it is in shared
      // memory, so the first half of the dK MMAs goes in while the second part is computed
      const float4* nd4 = reinterpret_cast<const float4*>(d_buf + half * 64);
      bool stop = false;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t(&r)[32] = h == 0 ? r0 : r1;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 nd = nd4[8 * h + j4];
          const int i = 32 * h + 4 * j4;
          pv[i] *= __uint_as_float(r[4 * j4]) + nd.x;
          pv[i + 1] *= __uint_as_float(r[4 * j4 + 1]) + nd.y;
          pv[i + 2] *= __uint_as_float(r[4 * j4 + 2]) + nd.z;
          pv[i + 3] *= __uint_as_float(r[4 * j4 + 3]) + nd.w;
        }
        uint4 lo[4];
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          const int gi = 4 * h + g4;
          const int gq = half * 8 + gi;  // 16-byte granule index over the 128 queries
          const uint32_t off = (gq >> 3) * L::kChunkBytes + t * 128 + ((((gq & 7) ^ (t & 7))) << 4);
          uint4 a;
          split_pack<T>(pv[gi * 8 + 0], pv[gi * 8 + 1], a.x, lo[g4].x);
          split_pack<T>(pv[gi * 8 + 2], pv[gi * 8 + 3], a.y, lo[g4].y);
          split_pack<T>(pv[gi * 8 + 4], pv[gi * 8 + 5], a.z, lo[g4].z);
          split_pack<T>(pv[gi * 8 + 6], pv[gi * 8 + 7], a.w, lo[g4].w);
          *reinterpret_cast<uint4*>(sdSh + off) = a;
        }
        if (h == 0 && L::kLoStageChunks > 0 && it >= 1 &&
            !mbar_wait_warp(dsl_free, (it - 1) & 1, abort_flag, p.status)) {
          stop = true;
          break;
        }
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          const int gq = half * 8 + 4 * h + g4;
          const uint32_t off = (gq >> 3) * L::kChunkBytes + t * 128 + ((((gq & 7) ^ (t & 7))) << 4);
          *reinterpret_cast<uint4*>(sdSl + off) = lo[g4];
        }
        fence_async_smem();
        mbar_arrive_warp(ds_full + h);
      }
      if (stop) break;
      // the next tile's LSE and D: their latency passes while this warp waits for the next S^T
      load_rows(it + 1);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <typename T, int DP, bool CAUSAL>
cudaError_t launch_bwd_tc_t(const BwdMaps& maps, const BwdParams& p, cudaStream_t stream) {
  using L = BwdLayout<DP>;
  auto kern = bwd_tc_kernel<T, DP, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
  if (e != cudaSuccess) return e;
  // The in-kernel register split assumes the launch allocation; never launch otherwise.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != static_cast<int>(L::kLaunchRegs)) return cudaErrorInvalidConfiguration;
  const dim3 grid(p.cu_seqlens ? p.nseq * p.Hkv : p.B * p.Hkv, p.n_ktiles);
  kern<<<grid, L::kThreads, L::kSmemAlloc, stream>>>(maps.q, maps.k, maps.v, maps.dout, maps.dq_acc, p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_tc_dtype(const BwdMaps& maps, const BwdParams& p, bool causal, cudaStream_t stream) {
  if (p.d <= 64)
    return causal ? launch_bwd_tc_t<T, 64, true>(maps, p, stream) : launch_bwd_tc_t<T, 64, false>(maps, p, stream);
  return causal ? launch_bwd_tc_t<T, 128, true>(maps, p, stream) : launch_bwd_tc_t<T, 128, false>(maps, p, stream);
}

}  // namespace attn
