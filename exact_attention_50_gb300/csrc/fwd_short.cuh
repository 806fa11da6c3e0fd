// fwd_short.cuh -- tcgen05 forward for short sequences (N <= 64) with many (batch, head) pairs.
//
// A short sequence fills a small corner of a 128 x 128 score tile.  This kernel packs several
// independent problems into one tile instead (the attention-operator article, section 2.3: for
// the short sequences of diffusion models a single warp-sized block holds the whole Q.K^T and
// the row max / sum stay in registers).  A unit is one (batch, kv head): its R = G * N query
// rows (the G query heads of the kv head are adjacent in [B, Hq, N, d]) against its N keys.
//   packed (R <= 128): P = 128 / R units per tile; rows [u0 R, u0 R + P R) of the flat
//                      [B*Hkv*R, d] query matrix against keys [u0 N, u0 N + P N) of the flat
//                      [B*Hkv*N, d] key / value matrices, block-diagonal mask (a row sees only
//                      the keys of its own unit);
//   unpacked (R > 128): one unit's 128-row block against the unit's N keys.
// One S tile per work item: S = scale Q K^T in TMEM, a plain (not online) softmax in registers
// -- one thread per row, the warp loading only the key columns its rows can see -- P (16-bit)
// back into TMEM, O = P V in TMEM, O / l staged in the item's Q slot and written by TMA tile
// stores whose box is exactly the item's rows.  The loads use boxes of exactly the item's rows
// and keys too, so the shared memory past them is never written: it is zeroed once at start,
// which keeps the unused key rows of V at 0 (they meet P = 0 in the P V product).
//
// Persistent: one CTA per SM walks the items; a ring of Q/K/V stages keeps the next items'
// loads in flight while the current one computes (the kernel is HBM-bound: about 4 d bytes of
// traffic per 4 N d FLOPs of a row).  224 threads:
//   warp 0     TMA producer (lane 0), TMEM allocator
//   warp 1     MMA issuer (lane 0): S(t) once its stage has landed and the softmax has read
//              S(t-1); P V (t) once P(t) is written and the epilogue has read O(t-1)
//   warps 2-5  softmax and epilogue, thread = row (TMEM lane quadrant = warp % 4)
//   warp 6     output tile stores (lane 0), then frees the stage
#pragma once
#include "fwd_tc.cuh"

namespace attn {

template <int DP>
struct ShortLayout {
  static constexpr int kStages = DP == 128 ? 2 : 4;
  static constexpr int kChunkBytes = 128 * 128;  // 128 rows x 64 16-bit elements
  static constexpr int kTileBytes = (DP / 64) * kChunkBytes;
  static constexpr int kStageBytes = 3 * kTileBytes;  // Q (later the O staging), K, V
  static constexpr int kOffBar = kStages * kStageBytes;
  // full[S], empty[S], staged[S], s_full, s_free, p_full, pv_done, o_free, drain.  staged is
  // per stage so it can never run two phases ahead of the store warp: an item's stage is
  // loaded again only after the store warp has written the item out.
  static constexpr int kNumBars = 3 * kStages + 6;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem base, abort flag, wait limit (u64)
  static constexpr int kSmemAlloc = kOffMisc + 16;
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory over the per-CTA limit");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColP = 128, kColO = 256;
  static constexpr int kThreads = 224;
};

// Where work item t of a short launch sits: its first unit, its first row inside that unit
// (unpacked: a multiple of 128) and how many units it holds.
struct ShortItem {
  int u0, q0, units;
};

__device__ __forceinline__ ShortItem short_item(const ShortParams& p, int t) {
  ShortItem it;
  if (p.packed) {
    it.u0 = t * p.P;
    it.q0 = 0;
    it.units = min(p.P, p.U - it.u0);
  } else {
    it.u0 = t / p.row_tiles;
    it.q0 = (t % p.row_tiles) * kBM;
    it.units = 1;
  }
  return it;
}

template <typename T, int DP, bool CAUSAL>
__global__ void __launch_bounds__(224, 1)
    fwd_short_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const ShortParams p) {
  using L = ShortLayout<DP>;
  constexpr int S = L::kStages;
  constexpr int kChunks = DP / 64;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) raise_status(p.status, ATTN_ERR_CUDA);
    return;
  }
  uint8_t* smem = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* staged = bars + 2 * S;  // [S]: the softmax warps have staged the item's O tile
  uint64_t* s_full = bars + 3 * S;
  uint64_t* s_free = s_full + 1;
  uint64_t* p_full = s_free + 1;
  uint64_t* pv_done = p_full + 1;
  uint64_t* o_free = pv_done + 1;
  uint64_t* drain = o_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  const uint32_t abort_flag = smem_u32(smem + L::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto sQ = [&](int s) { return smem + s * L::kStageBytes; };
  auto sK = [&](int s) { return smem + s * L::kStageBytes + L::kTileBytes; };
  auto sV = [&](int s) { return smem + s * L::kStageBytes + 2 * L::kTileBytes; };

  // Zero the stages once: the loads only ever write the item's rows and keys.
  for (int i = threadIdx.x; i < L::kOffBar / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_async_smem();
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
      mbar_init(staged + i, 4);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(o_free, 4);
    mbar_init(drain, 1);
    abort_set(abort_flag, 0);
    wait_limit_set(abort_flag, p.wait_ns);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(tmem_slot, L::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_items = p.n_items;
  const uint32_t q_bytes = static_cast<uint32_t>(kChunks * p.box_q * 128);
  const uint32_t kv_bytes = static_cast<uint32_t>(kChunks * p.box_k * 128);

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t n = 0;
      for (int t = blockIdx.x; t < n_items; t += gridDim.x, ++n) {
        const int s = n % S;
        if (n >= static_cast<uint32_t>(S) && !mbar_wait(empty + s, ((n / S) - 1) & 1, abort_flag, p.status)) break;
        const ShortItem it = short_item(p, t);
        mbar_expect_tx(full + s, q_bytes + 2 * kv_bytes);
        for (int c = 0; c < kChunks; ++c) {
          if (p.packed) {
            tma_load_2d(sQ(s) + c * L::kChunkBytes, &tmQ, full + s, c * 64, it.u0 * p.R);
            tma_load_2d(sK(s) + c * L::kChunkBytes, &tmK, full + s, c * 64, it.u0 * p.N);
            tma_load_2d(sV(s) + c * L::kChunkBytes, &tmV, full + s, c * 64, it.u0 * p.N);
          } else {
            tma_load_3d(sQ(s) + c * L::kChunkBytes, &tmQ, full + s, c * 64, it.q0, it.u0);
            tma_load_3d(sK(s) + c * L::kChunkBytes, &tmK, full + s, c * 64, 0, it.u0);
            tma_load_3d(sV(s) + c * L::kChunkBytes, &tmV, full + s, c * 64, 0, it.u0);
          }
        }
      }
      if (abort_read(abort_flag)) {
        for (uint32_t j = n > static_cast<uint32_t>(S) ? n - S : 0; j < n; ++j) mbar_drain(full + j % S, (j / S) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr bool kB = Elem<T>::kBf16;
      constexpr uint32_t idS = idesc_f16(kB, false, false, 128, 128);
      constexpr uint32_t idO = idesc_f16(kB, false, true, 128, DP);
      const uint64_t dQ = smem_desc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t dK = smem_desc_sw128(smem_u32(smem + L::kTileBytes), 16, 1024);
      const uint64_t dV = smem_desc_sw128(smem_u32(smem + 2 * L::kTileBytes), L::kChunkBytes, 1024);
      constexpr uint32_t kStage16 = L::kStageBytes >> 4;
      const int mine = n_items > static_cast<int>(blockIdx.x) ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
      int ns = 0, np = 0;
      bool ok = true;
      unsigned long long t_idle = 0;
      while (np < mine) {
        bool progress = false;
        // S(ns): its stage has landed, and the softmax has read S(ns - 1)
        if (ns < mine && mbar_test(full + ns % S, (ns / S) & 1) && (ns == 0 || mbar_test(s_free, (ns - 1) & 1))) {
          tc_fence_after();
          const uint64_t qx = opaque(dQ + (ns % S) * kStage16), kx = opaque(dK + (ns % S) * kStage16);
#pragma unroll
          for (int ks = 0; ks < DP / 16; ++ks) {
            const uint32_t off = ((ks >> 2) * L::kChunkBytes + (ks & 3) * 32) >> 4;
            mma_ss(tmem + L::kColS, qx + off, kx + off, idS, ks > 0 ? 1u : 0u);
          }
          mma_commit(s_full);
          ++ns;
          progress = true;
        }
        // P V (np): P(np) written, and the epilogue has read O(np - 1)
        if (np < ns && mbar_test(p_full, np & 1) && (np == 0 || mbar_test(o_free, (np - 1) & 1))) {
          tc_fence_after();
          const uint64_t vx = opaque(dV + (np % S) * kStage16);
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks)
            mma_ts(tmem + L::kColO, tmem + L::kColP + ks * 8, vx + ((ks * 2048) >> 4), idO, ks > 0 ? 1u : 0u);
          mma_commit(pv_done);
          ++np;
          progress = true;
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
      if (!ok) {
        mma_commit(drain);
        mbar_drain(drain, 0);
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    // ================================================================ output stores
    if (lane == 0) {
      const bool tile_out = !p.out_f32;
      if (tile_out) tma_prefetch_desc(&tmO);
      uint32_t n = 0;
      for (int t = blockIdx.x; t < n_items; t += gridDim.x, ++n) {
        const int s = n % S;
        if (!mbar_wait(staged + s, (n / S) & 1, abort_flag, p.status)) break;
        if (tile_out) {
          const ShortItem it = short_item(p, t);
          for (int c = 0; c < kChunks; ++c) {
            if (p.packed)
              tma_store_2d(&tmO, sQ(s) + c * L::kChunkBytes, c * 64, it.u0 * p.R);
            else
              tma_store_3d(&tmO, sQ(s) + c * L::kChunkBytes, c * 64, it.q0, it.u0);
          }
          bulk_commit();
          bulk_wait_read<0>();
        }
        mbar_arrive(empty + s);
      }
      bulk_wait_all();
    }
    __syncwarp();
  } else {
    // ================================================================ softmax + epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // TMEM lane = row of the tile
    const uint32_t tl = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float sl2 = p.scale_log2;
    uint32_t n = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_items; t += gridDim.x, ++n) {
      const int s = n % S;
      const ShortItem it = short_item(p, t);
      // this row's unit, query index and visible keys [k_lo, k_hi) among the tile's columns
      int ur, qr, k_lo;
      if (p.packed) {
        ur = r / p.R;
        qr = r % p.R;
        k_lo = ur * p.N;
      } else {
        ur = 0;
        qr = it.q0 + r;
        k_lo = 0;
      }
      const bool row_ok = ur < it.units && qr < p.R;
      const int i = qr % p.N;
      const int k_hi = row_ok ? k_lo + (CAUSAL ? i + 1 : p.N) : k_lo;
      // the warp loads the union of its rows' key columns, 32 at a time
      const int w_lo = __reduce_min_sync(0xffffffffu, row_ok ? k_lo : 128);
      const int w_hi = __reduce_max_sync(0xffffffffu, k_hi);
      const int c_lo = w_lo / 32, c_hi = (w_hi + 31) / 32;  // chunk range [c_lo, c_hi)
      if (!mbar_wait_warp(s_full, n & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c >= c_lo && c < c_hi) {
          uint32_t v[32];
          tmem_ld32(tl + L::kColS + c * 32, v);
          tmem_ld_wait();
          tmem_reg_fence(v);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int key = c * 32 + j;
            x[c * 32 + j] = (key >= k_lo && key < k_hi) ? __uint_as_float(v[j]) * sl2 : -INFINITY;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c * 32 + j] = -INFINITY;
        }
      }
      tc_fence_before();
      mbar_arrive_warp(s_free);
      float m = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (c >= c_lo && c < c_hi) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) m = max3f(m, x[c * 32 + j], x[c * 32 + j + 1]);
        }
      const float mb = (m == -INFINITY) ? 0.f : m;
      float l = 0.f;
      // P over all 128 key columns (zeros outside the row's keys), 16-bit pairs in TMEM
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
        if (c >= c_lo && c < c_hi) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float e0 = ex2_approx(x[c * 32 + j] - mb), e1 = ex2_approx(x[c * 32 + j + 1] - mb);
            l += e0 + e1;
            pk[j / 2] = Elem<T>::pack(e0, e1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = 0u;
        }
        tmem_st16(tl + L::kColP + c * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(p_full);
      // ---- epilogue: O / l, LSE
      if (!mbar_wait_warp(pv_done, n & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const long long row = static_cast<long long>(it.u0) * p.R + (p.packed ? r : qr);  // flat [U*R] row
      uint32_t o[32];
      if (!p.out_f32) {
        // into this item's Q slot, in the 128-byte swizzled layout of the store map's boxes
        uint8_t* srow = sQ(s) + r * 128;
#pragma unroll
        for (int c = 0; c < DP / 32; ++c) {
          tmem_ld32(tl + L::kColO + c * 32, o);
          tmem_ld_wait();
          tmem_reg_fence(o);
          if (c == DP / 32 - 1) {
            tc_fence_before();
            mbar_arrive_warp(o_free);
          }
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 v;
            v.x = Elem<T>::pack(__uint_as_float(o[8 * g + 0]) * inv_l, __uint_as_float(o[8 * g + 1]) * inv_l);
            v.y = Elem<T>::pack(__uint_as_float(o[8 * g + 2]) * inv_l, __uint_as_float(o[8 * g + 3]) * inv_l);
            v.z = Elem<T>::pack(__uint_as_float(o[8 * g + 4]) * inv_l, __uint_as_float(o[8 * g + 5]) * inv_l);
            v.w = Elem<T>::pack(__uint_as_float(o[8 * g + 6]) * inv_l, __uint_as_float(o[8 * g + 7]) * inv_l);
            const int gran = (c & 1) * 4 + g;  // 16-byte granule within the 64-column chunk
            *reinterpret_cast<uint4*>(srow + (c >> 1) * L::kChunkBytes + ((gran ^ (r & 7)) << 4)) = v;
          }
        }
        fence_async_smem();
      } else {
#pragma unroll
        for (int c = 0; c < DP / 32; ++c) {
          tmem_ld32(tl + L::kColO + c * 32, o);
          tmem_ld_wait();
          tmem_reg_fence(o);
          if (c == DP / 32 - 1) {
            tc_fence_before();
            mbar_arrive_warp(o_free);
          }
          if (row_ok && c * 32 < p.d) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + row * p.d + c * 32);
            const int ncol = min(32, p.d - c * 32);
#pragma unroll
            for (int g = 0; g < 8; ++g)
              if (g * 4 < ncol)
                dst[g] = make_float4(__uint_as_float(o[4 * g]) * inv_l, __uint_as_float(o[4 * g + 1]) * inv_l,
                                     __uint_as_float(o[4 * g + 2]) * inv_l, __uint_as_float(o[4 * g + 3]) * inv_l);
          }
        }
      }
      if (row_ok && p.lse) p.lse[row] = (m == -INFINITY) ? -INFINITY : (m + __log2f(l)) * 0.69314718055994531f;
      mbar_arrive_warp(staged + s);
    }
    (void)ok;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <typename T, int DP, bool CAUSAL>
cudaError_t launch_fwd_short_t(const FwdMaps& maps, const ShortParams& p, cudaStream_t stream) {
  using L = ShortLayout<DP>;
  auto kern = fwd_short_kernel<T, DP, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemAlloc);
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < sm_count() ? p.n_items : sm_count();
  kern<<<grid, L::kThreads, L::kSmemAlloc, stream>>>(maps.q, maps.k, maps.v, maps.o, p);
  return cudaGetLastError();
}

}  // namespace attn
