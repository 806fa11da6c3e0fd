// attn_noalloc.cu -- the backward for callers that cannot allocate device memory.
//
// attn_bwd needs a scratch workspace (an fp32 dQ accumulator and the fp32 row terms D) that the
// caller allocates.  Some callers cannot: a plugin or host application whose device memory is
// reserved up front by another allocator and may not grow on the hot path, or a runtime that
// forbids allocation calls after start-up.  attn_bwd_noalloc serves them from a fixed scratch
// array that lives in this library's own module: it is reserved on every GPU that loads the
// library and held until the process exits.  No allocation call is made on any path here.
//
// The host side never touches the array by name (in host code the name is only a stand-in, not
// a device address): the first call on each device looks up the array's device address with
// cudaGetSymbolAddress while that device is current and caches it; later calls reuse it.
#include <cuda_runtime.h>
#include <mutex>
#include "attn.h"

namespace {

constexpr size_t kScratchBytes = 64ull << 20;  // 64 MiB: see attn_bwd_noalloc in attn.h

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

// Device address of g_bwd_scratch on the current device (looked up once per device).
void* scratch_address() {
  static std::mutex mu;
  static void* cache[256] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess) return nullptr;
    cache[dev] = ptr;
  }
  return cache[dev];
}

}  // namespace

extern "C" attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                          const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                                          int Hq, int Hkv, int N, int d, int causal, float scale,
                                          attn_dtype_t dtype, unsigned flags, void* stream) {
  if (B < 0 || Hq <= 0 || N < 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || N == 0)  // empty: nothing to compute, no scratch needed
    return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, nullptr, 0, B, Hq, Hkv, N, d, causal, scale, dtype, flags,
                    stream);
  if (attn_bwd_workspace_bytes(B, Hq, N, d) > kScratchBytes) return ATTN_ERR_UNSUPPORTED;
  void* scratch = scratch_address();
  if (!scratch) return ATTN_ERR_CUDA;
  // attn_bwd zeroes the part of the scratch that must start at zero (the dQ accumulator) and
  // overwrites the rest, so what an earlier call left in the array does not matter.
  return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, kScratchBytes, B, Hq, Hkv, N, d, causal, scale,
                  dtype, flags, stream);
}
