// ptx.cuh -- hand-written inline PTX for sm_103a: mbarriers, TMA tile loads, tcgen05 (TMEM
// allocation, MMA, commit, loads/stores) and the shared-memory / instruction descriptors.
//
// Every wait on an mbarrier is bounded: after the CTA's wait limit (kWaitTimeoutNs unless the
// launch sets another) of %globaltimer time it records ATTN_ERR_TIMEOUT in the device status
// word, raises the CTA's abort flag and returns false, so a broken pipeline ends with an error
// status instead of a hung GPU.
#pragma once
#include <cstdint>
#include <cuda.h>
#include "attn.h"

namespace attn {

constexpr unsigned long long kWaitTimeoutNs = 4000000000ull;  // default: 4 s per single wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Records the first error raised on the device since the last status read.
__device__ __forceinline__ void raise_status(unsigned* status, unsigned code) {
  if (status) atomicCAS(status, 0u, code);
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The CTA's abort flag is a 32-bit word in shared memory, addressed through the shared window.
__device__ __forceinline__ int abort_read(uint32_t flag) {
  int v;
  asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(v) : "r"(flag) : "memory");
  return v;
}
__device__ __forceinline__ void abort_set(uint32_t flag, int v) {
  asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(flag), "r"(v) : "memory");
}

// The CTA's wait limit in ns: a 64-bit word in shared memory 4 bytes after the abort flag
// (8-byte aligned), written once at the start of the kernel.
__device__ __forceinline__ void wait_limit_set(uint32_t flag, unsigned long long ns) {
  asm volatile("st.shared.u64 [%0], %1;" ::"r"(flag + 4), "l"(ns ? ns : kWaitTimeoutNs) : "memory");
}
__device__ __forceinline__ unsigned long long wait_limit(uint32_t flag) {
  unsigned long long ns;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(ns) : "r"(flag + 4) : "memory");
  return ns;
}

// Non-blocking probe: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false (after raising the abort
// flag and, on a timeout, the device status) when the CTA must stop.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t abort_flag, unsigned* status) {
  const uint32_t b = smem_u32(bar);
  if (mbar_try_wait(b, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 63u) == 0u) {
      if (abort_read(abort_flag)) return false;
      if (globaltimer() - t0 > wait_limit(abort_flag)) {
        raise_status(status, ATTN_ERR_TIMEOUT);
        abort_set(abort_flag, 1);
        return false;
      }
    }
  }
}

// Bounded wait taken by a whole warp: every lane gets the same answer (false if any lane's
// wait failed), so the warp leaves a loop together and later warp-wide operations stay safe.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, uint32_t abort_flag,
                                               unsigned* status) {
  const bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// One arrival for the whole warp (the barrier counts warps, not threads).  Arrivals on one
// mbarrier are atomic updates of one shared-memory word and serialise, so a warp arrives once:
// the __syncwarp orders every lane's earlier work (after the caller's fences) before lane 0's
// release-arrive.
__device__ __forceinline__ void mbar_arrive_warp(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// A short bounded wait used only on the abort path, to let copies already in flight land
// before the CTA exits.  Never raises a status.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t b = smem_u32(bar);
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(b, parity)) {
    if (globaltimer() - t0 > 200000000ull) return;  // 0.2 s
  }
}

// ------------------------------------------------------------------ TMA (tiled, no multicast)
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Tile store shared -> global (bulk group; elements outside the tensor are not written).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Element-wise add of a shared-memory tile into a global tensor (2-D tiled map), performed as
// a reduction in L2; completion is tracked by bulk groups.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* m, const void* src, int c0, int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N of the most recently committed bulk groups are still reading their
// shared-memory sources (all older groups have finished reading).
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every committed bulk group has completed (its writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's generic-proxy and async-proxy (bulk copy) accesses to global memory.
__device__ __forceinline__ void fence_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Bounded wait (one thread) until the counter at p reaches `target` (counters only grow).
// Returns false after raising the abort flag, and on a timeout the device status.
__device__ __forceinline__ bool wait_turn(const int* p, int target, uint32_t abort_flag, unsigned* status) {
  if (ld_acquire_gpu(p) >= target) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    __nanosleep(100);
    if (ld_acquire_gpu(p) >= target) return true;
    if (abort_read(abort_flag)) return false;
    if (globaltimer() - t0 > wait_limit(abort_flag)) {
      raise_status(status, ATTN_ERR_TIMEOUT);
      abort_set(abort_flag, 1);
      return false;
    }
  }
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tensor core, TMA).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (fp16 or bf16 in, fp32 accumulate).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16: A (M x 16, K-major, two 16-bit values per
// 32-bit column) is read from tensor memory.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on the mbarrier when every tcgen05 async operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

#define ATTN_R32(p)                                                                                    \
  "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3]), "=r"(p[4]), "=r"(p[5]), "=r"(p[6]), "=r"(p[7]),     \
      "=r"(p[8]), "=r"(p[9]), "=r"(p[10]), "=r"(p[11]), "=r"(p[12]), "=r"(p[13]), "=r"(p[14]),         \
      "=r"(p[15]), "=r"(p[16]), "=r"(p[17]), "=r"(p[18]), "=r"(p[19]), "=r"(p[20]), "=r"(p[21]),       \
      "=r"(p[22]), "=r"(p[23]), "=r"(p[24]), "=r"(p[25]), "=r"(p[26]), "=r"(p[27]), "=r"(p[28]),       \
      "=r"(p[29]), "=r"(p[30]), "=r"(p[31])
#define ATTN_W32(p)                                                                                    \
  "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7]), "r"(p[8]),   \
      "r"(p[9]), "r"(p[10]), "r"(p[11]), "r"(p[12]), "r"(p[13]), "r"(p[14]), "r"(p[15]), "r"(p[16]),   \
      "r"(p[17]), "r"(p[18]), "r"(p[19]), "r"(p[20]), "r"(p[21]), "r"(p[22]), "r"(p[23]), "r"(p[24]),  \
      "r"(p[25]), "r"(p[26]), "r"(p[27]), "r"(p[28]), "r"(p[29]), "r"(p[30]), "r"(p[31])
#define ATTN_RW32(p)                                                                                   \
  "+r"(p[0]), "+r"(p[1]), "+r"(p[2]), "+r"(p[3]), "+r"(p[4]), "+r"(p[5]), "+r"(p[6]), "+r"(p[7]),     \
      "+r"(p[8]), "+r"(p[9]), "+r"(p[10]), "+r"(p[11]), "+r"(p[12]), "+r"(p[13]), "+r"(p[14]),         \
      "+r"(p[15]), "+r"(p[16]), "+r"(p[17]), "+r"(p[18]), "+r"(p[19]), "+r"(p[20]), "+r"(p[21]),       \
      "+r"(p[22]), "+r"(p[23]), "+r"(p[24]), "+r"(p[25]), "+r"(p[26]), "+r"(p[27]), "+r"(p[28]),       \
      "+r"(p[29]), "+r"(p[30]), "+r"(p[31])

// 32 consecutive columns of this warp's 32 TMEM lanes: thread t gets lane (base + t).
// The values are valid only after tmem_ld_wait(); tmem_reg_fence() then pins their uses after it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : ATTN_R32(r)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_reg_fence(uint32_t (&r)[32]) { asm volatile("" : ATTN_RW32(r)::"memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32};" ::"r"(taddr),
      ATTN_W32(r)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor (tcgen05 format): start address, leading and stride byte
// offsets (all >> 4), the fixed version field (bits 46-47 = 1), base offset 0 (every swizzle
// atom starts 1024-byte aligned), layout type 2 = 128-byte swizzle (bits 61-63).
//   K-major operand: rows of 128 B (64 16-bit elements), 8-row groups SBO = 1024 B apart;
//                    LBO is not used by the 128-byte swizzled K-major layout.
//   MN-major operand: 64 MN-contiguous elements per 128-B row; 8 K-rows per atom with
//                    SBO = 1024 B between 8-row groups along K and LBO = distance between
//                    consecutive 64-element atoms along MN.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation, dense.
//   bits 4-5 D format (1 = f32); 7-9 A format and 10-12 B format (0 = f16, 1 = bf16);
//   bit 15 A major, bit 16 B major (0 = K-major, 1 = MN-major); 17-22 N >> 3; 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, bool a_mn_major, bool b_mn_major, int M, int N) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

// Hides a value from the optimiser at this point: expressions derived from it are computed
// here instead of being hoisted out of the enclosing loop and kept live in registers.
__device__ __forceinline__ uint64_t opaque(uint64_t x) {
  asm volatile("" : "+l"(x));
  return x;
}

// ------------------------------------------------------------------ register split
// Per-warpgroup register budget changes; every warp of the warpgroup executes the same one.
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ global reductions
// Four fp32 adds into global memory with no return value (relaxed, gpu scope).
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// ------------------------------------------------------------------ math
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x on the FMA/ALU pipes, to take part of the exponentials off the special-function unit.
// Range reduction in the manner of Cody and Waite: x = n + f with n = round(x), f in [-1/2, 1/2]
// (adding 1.5 * 2^23 leaves round(x) in the low mantissa bits); 2^f from a degree-3 polynomial
// whose coefficients were fitted for this library by the Remez exchange algorithm (minimax
// relative error 7.5e-5 on [-1/2, 1/2]); 2^n added into the exponent field.  x is clamped to
// -126 so the result stays normal: inputs below that give 2^-126 instead of (almost) 0.
__device__ __forceinline__ float exp2_fma(float x) {
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  constexpr float c0 = 0.99992806f, c1 = 0.69326097f, c2 = 0.24261113f, c3 = 0.05517167f;
  x = fmaxf(x, -126.0f);
  const float t = x + kRound;
  const float n = t - kRound;
  const float f = x - n;
  const float p = fmaf(fmaf(fmaf(c3, f, c2), f, c1), f, c0);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// ------------------------------------------------------------------ paired fp32 arithmetic
// Two fp32 values in one 64-bit register pair: the f32x2 instructions do two operations per
// issue slot, which halves the instruction count of elementwise fp32 work.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three values in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// exp2_fma on a pair, with the range reduction and polynomial in paired instructions.
__device__ __forceinline__ uint64_t exp2_fma2(uint64_t x) {
  constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
  const float2 xf = f2_unpack(x);
  const uint64_t xc = f2_pack(fmaxf(xf.x, -126.0f), fmaxf(xf.y, -126.0f));
  const uint64_t t = f2_add(xc, f2_pack(kRound, kRound));
  const uint64_t n = f2_add(t, f2_pack(-kRound, -kRound));
  const uint64_t f = f2_fma(n, f2_pack(-1.0f, -1.0f), xc);
  uint64_t q = f2_fma(f2_pack(0.05517167f, 0.05517167f), f, f2_pack(0.24261113f, 0.24261113f));
  q = f2_fma(q, f, f2_pack(0.69326097f, 0.69326097f));
  q = f2_fma(q, f, f2_pack(0.99992806f, 0.99992806f));
  const float2 qf = f2_unpack(q), tf = f2_unpack(t);
  return f2_pack(__int_as_float(__float_as_int(qf.x) + (__float_as_int(tf.x) << 23)),
                 __int_as_float(__float_as_int(qf.y) + (__float_as_int(tf.y) << 23)));
}

}  // namespace attn
