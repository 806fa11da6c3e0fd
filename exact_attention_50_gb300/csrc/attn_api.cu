// attn_api.cu -- the C ABI (include/attn.h): argument validation, TMA tensor-map encoding,
// the per-device status word and dispatch to the kernels.  Nothing here allocates device
// memory; every launch goes on the caller's stream.
#include <cudaTypedefs.h>
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <initializer_list>
#include <mutex>
#include "kernels.h"

namespace {

using attn::BwdMaps;
using attn::BwdParams;
using attn::FwdMaps;
using attn::FwdParams;

// First error recorded by a kernel on this device (0 = none); cleared by attn_get_device_status.
__device__ unsigned g_attn_status;

constexpr float kLog2e = 1.4426950408889634f;

unsigned* status_word() {
  static std::mutex mu;
  static unsigned* cache[256] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_attn_status) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned*>(ptr);
  }
  return cache[dev];
}

// The limit of any single device-side wait, in ns: ATTN_WAIT_LIMIT_MS from the environment when
// the first call is made (10 .. 600000 ms), else 4 s.  A pipeline wait or a deterministic
// backward's turn wait that exceeds it stops its CTA and reports ATTN_ERR_TIMEOUT.
unsigned long long wait_limit_ns() {
  static unsigned long long ns = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    ns = 4000000000ull;
    if (const char* e = std::getenv("ATTN_WAIT_LIMIT_MS")) {
      char* end = nullptr;
      const long ms = std::strtol(e, &end, 10);
      if (end != e && *end == '\0' && ms >= 10 && ms <= 600000) ns = static_cast<unsigned long long>(ms) * 1000000ull;
    }
  });
  return ns;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// 128-byte-swizzled tile map with a {64 elements, rows} box over the innermost (head_dim) and
// the row dimension.  rank 3 = dense {d, N, B*H}; rank 4 = packed varlen {d, H, 3, T}.
bool make_map(CUtensorMap* map, const void* base, attn_dtype_t dt, int rank, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType t =
      dt == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = fn(map, t, rank, const_cast<void*>(base), dims, strides_bytes, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The fp32 dQ accumulator [rows, d] as a 2-D map with a {32, 128} box (128 bytes per row).
bool make_acc_map(CUtensorMap* map, const float* base, long long rows, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(d) * 4};
  const uint32_t box[2] = {32, 128};
  const uint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_dense_map(CUtensorMap* map, const void* base, attn_dtype_t dt, int heads_total, int N, int d) {
  const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(N), static_cast<uint64_t>(heads_total)};
  const uint64_t strides[2] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(N) * d * 2};
  const uint32_t box[3] = {64, 128, 1};
  return make_map(map, base, dt, 3, dims, strides, box);
}

// {d, rows, heads} over a [rows, heads, d]-like layout with the given element strides (a plane
// of packed qkv, or a [T, H, d] tensor): the same box and coordinates as the dense maps.
bool make_rows_map(CUtensorMap* map, const void* base, attn_dtype_t dt, int rows, int heads, int d,
                   long long row_stride, long long head_stride) {
  const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(rows), static_cast<uint64_t>(heads)};
  const uint64_t strides[2] = {static_cast<uint64_t>(row_stride) * 2, static_cast<uint64_t>(head_stride) * 2};
  const uint32_t box[3] = {64, 128, 1};
  return make_map(map, base, dt, 3, dims, strides, box);
}

bool make_packed_map(CUtensorMap* map, const void* base, attn_dtype_t dt, int T, int H, int d) {
  const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(H), 3, static_cast<uint64_t>(T)};
  const uint64_t strides[3] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(H) * d * 2,
                               3ull * H * d * 2};
  const uint32_t box[4] = {64, 1, 1, 128};
  return make_map(map, base, dt, 4, dims, strides, box);
}

attn_status_t check_common(int d, float scale, attn_dtype_t dt) {
  if (dt != ATTN_F32 && dt != ATTN_F16 && dt != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (!(scale >= 0.f) || std::isinf(scale)) return ATTN_ERR_INVALID_ARG;
  if (d <= 0) return ATTN_ERR_INVALID_ARG;
  if (d % 16 != 0 || d > 128) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

float resolve_scale(float scale, int d) { return scale == 0.f ? 1.f / std::sqrt(static_cast<float>(d)) : scale; }

attn_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// The short-sequence kernel serves dense fp16 / bf16 forwards with N <= 64 unless the environment
// sets ATTN_SHORT_KERNEL=0 (a switch to time the general kernel on the same shapes).
bool short_kernel_enabled() {
  const char* e = std::getenv("ATTN_SHORT_KERNEL");
  return !(e && e[0] == '0' && e[1] == '\0');
}

// Dense forward of short sequences on the packing kernel: one unit is a (batch, kv head) with its
// R = G * N query rows (adjacent in [B, Hq, N, d]) and its N keys.
attn_status_t fwd_short(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int N, int d, int causal, float scale, attn_dtype_t dtype, unsigned flags, cudaStream_t s) {
  const long long U = static_cast<long long>(B) * Hkv;
  const int G = Hq / Hkv;
  const long long R = static_cast<long long>(G) * N;
  if (U * R > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  attn::ShortParams p{};
  p.o = o;
  p.lse = lse;
  p.status = status_word();
  p.wait_ns = wait_limit_ns();
  if (!p.status) return ATTN_ERR_CUDA;
  p.U = static_cast<int>(U); p.N = N; p.R = static_cast<int>(R); p.G = G; p.d = d;
  p.packed = R <= attn::kBM ? 1 : 0;
  p.P = p.packed ? attn::kBM / p.R : 1;
  p.row_tiles = p.packed ? 1 : (p.R + attn::kBM - 1) / attn::kBM;
  p.n_items = p.packed ? (p.U + p.P - 1) / p.P : p.U * p.row_tiles;
  p.box_q = p.packed ? p.P * p.R : attn::kBM;
  p.box_k = p.packed ? p.P * N : N;
  p.scale_log2 = resolve_scale(scale, d) * kLog2e;
  p.out_f32 = (flags & ATTN_FLAG_OUT_F32) ? 1 : 0;
  FwdMaps maps;
  const uint64_t es = 2;
  if (p.packed) {
    const uint64_t dq[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(U * R)};
    const uint64_t dk[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(U * N)};
    const uint64_t st[1] = {static_cast<uint64_t>(d) * es};
    const uint32_t bq[2] = {64, static_cast<uint32_t>(p.box_q)}, bk[2] = {64, static_cast<uint32_t>(p.box_k)};
    if (!make_map(&maps.q, q, dtype, 2, dq, st, bq) || !make_map(&maps.k, k, dtype, 2, dk, st, bk) ||
        !make_map(&maps.v, v, dtype, 2, dk, st, bk) || (!p.out_f32 && !make_map(&maps.o, o, dtype, 2, dq, st, bq)))
      return ATTN_ERR_CUDA;
  } else {
    const uint64_t dq[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(R), static_cast<uint64_t>(U)};
    const uint64_t dk[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(N), static_cast<uint64_t>(U)};
    const uint64_t sq[2] = {static_cast<uint64_t>(d) * es, static_cast<uint64_t>(R) * d * es};
    const uint64_t sk[2] = {static_cast<uint64_t>(d) * es, static_cast<uint64_t>(N) * d * es};
    const uint32_t bq[3] = {64, attn::kBM, 1}, bk[3] = {64, static_cast<uint32_t>(N), 1};
    if (!make_map(&maps.q, q, dtype, 3, dq, sq, bq) || !make_map(&maps.k, k, dtype, 3, dk, sk, bk) ||
        !make_map(&maps.v, v, dtype, 3, dk, sk, bk) || (!p.out_f32 && !make_map(&maps.o, o, dtype, 3, dq, sq, bq)))
      return ATTN_ERR_CUDA;
  }
  if (p.out_f32) maps.o = maps.q;  // unused: fp32 rows are stored by the threads
  return from_cuda(attn::launch_fwd_short(maps, p, dtype, causal != 0, s));
}

}  // namespace

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int N, int d, int causal, float scale, attn_dtype_t dtype, unsigned flags, void* stream) {
  attn_status_t st = check_common(d, scale, dtype);
  if (st != ATTN_OK) return st;
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (flags & ~ATTN_FLAG_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * Hq > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  const bool f32 = dtype == ATTN_F32;
  const int rows_per_tile = f32 ? 32 : attn::kBM;
  const int n_qtiles = (N + rows_per_tile - 1) / rows_per_tile;
  if (n_qtiles > 65535) return ATTN_ERR_UNSUPPORTED;

  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.status = status_word();
  p.wait_ns = wait_limit_ns();
  if (!p.status) return ATTN_ERR_CUDA;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = N; p.d = d; p.G = Hq / Hkv;
  p.n_qtiles = n_qtiles;
  p.scale = resolve_scale(scale, d);
  p.scale_log2 = p.scale * kLog2e;
  p.out_f32 = (flags & ATTN_FLAG_OUT_F32) ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (f32) return from_cuda(attn::launch_fwd_f32(q, k, v, p, causal != 0, attn::kModeDense, s));
  if (N <= 64 && short_kernel_enabled())
    return fwd_short(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, dtype, flags, s);
  FwdMaps maps;
  if (!make_dense_map(&maps.q, q, dtype, B * Hq, N, d) || !make_dense_map(&maps.k, k, dtype, B * Hkv, N, d) ||
      !make_dense_map(&maps.v, v, dtype, B * Hkv, N, d))
    return ATTN_ERR_CUDA;
  // the epilogue's tile stores (16-bit output); an fp32 output is stored by the threads
  if (p.out_f32)
    maps.o = maps.q;
  else if (!make_dense_map(&maps.o, o, dtype, B * Hq, N, d))
    return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_fwd_tc(maps, p, dtype, causal != 0, attn::kModeDense, s));
}

attn_status_t attn_fwd_varlen(const void* qkv, const int32_t* cu_seqlens, int nseq, int total_tokens,
                              int max_seqlen, void* out, float* lse, int H, int d, int causal, float scale,
                              attn_dtype_t dtype, unsigned flags, void* stream) {
  attn_status_t st = check_common(d, scale, dtype);
  if (st != ATTN_OK) return st;
  if (nseq < 0 || total_tokens < 0 || max_seqlen < 0 || H <= 0) return ATTN_ERR_INVALID_ARG;
  if (flags & ~ATTN_FLAG_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (nseq == 0) return total_tokens == 0 ? ATTN_OK : ATTN_ERR_INVALID_ARG;
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return ATTN_ERR_INVALID_ARG;
  if (total_tokens == 0) return ATTN_OK;  // every sequence is empty
  if (max_seqlen == 0) return ATTN_ERR_INVALID_ARG;
  if (!qkv || !out || !aligned(qkv, 16) || !aligned(out, 16) || !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
  if (nseq > 65535) return ATTN_ERR_UNSUPPORTED;
  const bool f32 = dtype == ATTN_F32;
  const int rows_per_tile = f32 ? 32 : attn::kBM;
  const int n_qtiles = (max_seqlen + rows_per_tile - 1) / rows_per_tile;
  if (n_qtiles > 65535) return ATTN_ERR_UNSUPPORTED;

  FwdParams p{};
  p.o = out;
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.status = status_word();
  p.wait_ns = wait_limit_ns();
  if (!p.status) return ATTN_ERR_CUDA;
  p.B = 1; p.Hq = H; p.Hkv = H; p.N = 0; p.d = d; p.G = 1;
  p.nseq = nseq; p.total_tokens = total_tokens; p.max_seqlen = max_seqlen;
  p.n_qtiles = n_qtiles;
  p.scale = resolve_scale(scale, d);
  p.scale_log2 = p.scale * kLog2e;
  p.out_f32 = (flags & ATTN_FLAG_OUT_F32) ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t plane = static_cast<size_t>(H) * d;
  if (f32) {
    const float* base = static_cast<const float*>(qkv);
    return from_cuda(attn::launch_fwd_f32(base, base + plane, base + 2 * plane, p, causal != 0, attn::kModeVarlen, s));
  }
  FwdMaps maps;
  if (!make_packed_map(&maps.q, qkv, dtype, total_tokens, H, d)) return ATTN_ERR_CUDA;
  maps.k = maps.q;
  maps.v = maps.q;
  // the epilogue's tile stores of full 128-row tiles (16-bit output): {d, T, H} over [T, H, d]
  if (p.out_f32)
    maps.o = maps.q;
  else if (!make_rows_map(&maps.o, out, dtype, total_tokens, H, d, static_cast<long long>(H) * d, d))
    return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_fwd_tc(maps, p, dtype, causal != 0, attn::kModeVarlen, s));
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int N, int d) {
  if (B <= 0 || Hq <= 0 || N <= 0 || d <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * N;
  return round256(rows * d * sizeof(float)) + 2 * round256(rows * sizeof(float));
}

namespace {

// Shared validation of the backward's sizes and workspace; fills the common BwdParams fields.
attn_status_t bwd_setup(BwdParams* p, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d,
                        float scale, attn_dtype_t dtype, unsigned flags, int grid_rows = -1) {
  attn_status_t st = check_common(d, scale, dtype);
  if (st != ATTN_OK) return st;
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (flags & ~(ATTN_FLAG_OUT_F32 | ATTN_FLAG_DETERMINISTIC)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return ATTN_OK;
  if (!workspace || !aligned(workspace, 256)) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_workspace_bytes(B, Hq, N, d)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * Hq > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (((grid_rows < 0 ? N : grid_rows) + 31) / 32 > 65535) return ATTN_ERR_UNSUPPORTED;  // grid y extent
  const size_t rows = static_cast<size_t>(B) * Hq * N;
  p->dq_acc = static_cast<float*>(workspace);
  p->delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + round256(rows * d * sizeof(float)));
  p->dq_turn = reinterpret_cast<int*>(reinterpret_cast<char*>(p->delta) + round256(rows * sizeof(float)));
  p->deterministic = (flags & ATTN_FLAG_DETERMINISTIC) ? 1 : 0;
  p->wait_ns = wait_limit_ns();
  p->B = B; p->Hq = Hq; p->Hkv = Hkv; p->N = N; p->Nk = N; p->d = d; p->G = Hq / Hkv;
  p->n_ktiles = (N + attn::kBN - 1) / attn::kBN;
  const BwdParams::Rows dense{d, static_cast<long long>(N) * d};
  p->lay_q = p->lay_kv = p->lay_o = p->lay_dq = p->lay_dkv = dense;
  p->cu_seqlens = nullptr;
  p->scale = resolve_scale(scale, d);
  p->scale_log2 = p->scale * kLog2e;
  p->out_f32 = (flags & ATTN_FLAG_OUT_F32) ? 1 : 0;
  return ATTN_OK;
}

bool all_aligned16(std::initializer_list<const void*> ptrs) {
  for (const void* ptr : ptrs)
    if (!ptr || !aligned(ptr, 16)) return false;
  return true;
}

}  // namespace

attn_status_t attn_bwd_prepare(const void* o, const void* dout, void* workspace, size_t workspace_bytes, int B,
                               int Hq, int N, int d, attn_dtype_t dtype, void* stream) {
  BwdParams p{};
  attn_status_t st = bwd_setup(&p, workspace, workspace_bytes, B, Hq, Hq, N, d, 0.f, dtype, 0);
  if (st != ATTN_OK || B == 0 || N == 0) return st;
  if (!all_aligned16({o, dout})) return ATTN_ERR_INVALID_ARG;
  p.o = o;
  p.dout = dout;
  if (!(p.status = status_word())) return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_bwd_preprocess(p, dtype, dtype != ATTN_F32, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_bwd_main(const void* q, const void* k, const void* v, const void* dout, const float* lse, void* dq,
                            void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                            int N, int d, int causal, float scale, attn_dtype_t dtype, unsigned flags,
                            void* stream) {
  BwdParams p{};
  attn_status_t st = bwd_setup(&p, workspace, workspace_bytes, B, Hq, Hkv, N, d, scale, dtype, flags);
  if (st != ATTN_OK || B == 0 || N == 0) return st;
  if (!all_aligned16({q, k, v, dout, dk, dv}) || !lse || !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
  if (dtype == ATTN_F32 && !all_aligned16({dq})) return ATTN_ERR_INVALID_ARG;
  p.q = q; p.k = k; p.v = v; p.dout = dout; p.lse = lse;
  p.dq = dq; p.dk = dk; p.dv = dv;
  if (!(p.status = status_word())) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == ATTN_F32) return from_cuda(attn::launch_bwd_f32(p, causal != 0, s));
  BwdMaps maps;
  if (!make_dense_map(&maps.q, q, dtype, B * Hq, N, d) || !make_dense_map(&maps.k, k, dtype, B * Hkv, N, d) ||
      !make_dense_map(&maps.v, v, dtype, B * Hkv, N, d) || !make_dense_map(&maps.dout, dout, dtype, B * Hq, N, d) ||
      !make_acc_map(&maps.dq_acc, p.dq_acc, static_cast<long long>(B) * Hq * N, d))
    return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_bwd_tc(maps, p, dtype, causal != 0, s));
}

attn_status_t attn_bwd_finish(void* dq, void* workspace, size_t workspace_bytes, int B, int Hq, int N, int d,
                              float scale, attn_dtype_t dtype, unsigned flags, void* stream) {
  BwdParams p{};
  attn_status_t st = bwd_setup(&p, workspace, workspace_bytes, B, Hq, Hq, N, d, scale, dtype, flags);
  if (st != ATTN_OK || B == 0 || N == 0) return st;
  if (dtype == ATTN_F32) return ATTN_OK;  // the fp32 main step wrote dq itself
  if (!all_aligned16({dq})) return ATTN_ERR_INVALID_ARG;
  p.dq = dq;
  if (!(p.status = status_word())) return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_bwd_postprocess(p, dtype, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                       void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                       int N, int d, int causal, float scale, attn_dtype_t dtype, unsigned flags, void* stream) {
  BwdParams p{};
  attn_status_t st = bwd_setup(&p, workspace, workspace_bytes, B, Hq, Hkv, N, d, scale, dtype, flags);
  if (st != ATTN_OK || B == 0 || N == 0) return st;
  if (!all_aligned16({q, k, v, o, dout, dq, dk, dv}) || !lse || !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
  st = attn_bwd_prepare(o, dout, workspace, workspace_bytes, B, Hq, N, d, dtype, stream);
  if (st == ATTN_OK)
    st = attn_bwd_main(q, k, v, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, d, causal, scale,
                       dtype, flags, stream);
  if (st == ATTN_OK) st = attn_bwd_finish(dq, workspace, workspace_bytes, B, Hq, N, d, scale, dtype, flags, stream);
  return st;
}

size_t attn_bwd_varlen_workspace_bytes(int total_tokens, int H, int d) {
  return attn_bwd_workspace_bytes(1, H, total_tokens, d);
}

size_t attn_bwd_cross_workspace_bytes(int B, int Hq, int Nq, int Nk, int d, attn_dtype_t dtype, unsigned flags) {
  (void)dtype;
  (void)flags;
  if (B <= 0 || Hq <= 0 || Nq <= 0 || Nk <= 0 || d <= 0) return 0;
  return attn_bwd_workspace_bytes(B, Hq, Nq, d);
}

// Cross-attention backward: the backward kernels walk Nq query rows against Nk keys per head
// directly, with the bottom-right causal alignment (query i sees key j iff j <= i + Nk - Nq).
attn_status_t attn_bwd_cross(const void* q, const void* k, const void* v, const void* o, const void* dout,
                             const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                             attn_dtype_t dtype, unsigned flags, void* stream) {
  attn_status_t st = check_common(d, scale, dtype);
  if (st != ATTN_OK) return st;
  if (B < 0 || Nq < 0 || Nk < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (flags & ~(ATTN_FLAG_OUT_F32 | ATTN_FLAG_DETERMINISTIC)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || (Nq == 0 && Nk == 0)) return ATTN_OK;
  if (Nq == Nk)
    return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, Nk, d, causal, scale,
                    dtype, flags, stream);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t eo = (dtype == ATTN_F32 || (flags & ATTN_FLAG_OUT_F32)) ? 4 : 2;
  if (Nq == 0) {  // no query: dk = dv = 0
    if (!all_aligned16({dk, dv})) return ATTN_ERR_INVALID_ARG;
    const size_t bytes = static_cast<size_t>(B) * Hkv * Nk * d * eo;
    if (cudaMemsetAsync(dk, 0, bytes, s) != cudaSuccess || cudaMemsetAsync(dv, 0, bytes, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  if (Nk == 0) {  // no key: every query row sees nothing, dq = 0
    if (!all_aligned16({dq})) return ATTN_ERR_INVALID_ARG;
    return from_cuda(cudaMemsetAsync(dq, 0, static_cast<size_t>(B) * Hq * Nq * d * eo, s));
  }
  if (!all_aligned16({q, k, v, o, dout, dq, dk, dv}) || !lse || !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
  if ((Nk + 31) / 32 > 65535) return ATTN_ERR_UNSUPPORTED;
  BwdParams p{};
  st = bwd_setup(&p, workspace, workspace_bytes, B, Hq, Hkv, Nq, d, scale, dtype, flags);
  if (st != ATTN_OK) return st;
  p.Nk = Nk;
  p.n_ktiles = (Nk + attn::kBN - 1) / attn::kBN;
  p.lay_kv = p.lay_dkv = BwdParams::Rows{d, static_cast<long long>(Nk) * d};
  p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse;
  p.dq = dq; p.dk = dk; p.dv = dv;
  if (!(p.status = status_word())) return ATTN_ERR_CUDA;
  cudaError_t e = attn::launch_bwd_preprocess(p, dtype, dtype != ATTN_F32, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  if (dtype == ATTN_F32) return from_cuda(attn::launch_bwd_f32(p, causal != 0, s));
  BwdMaps maps;
  if (!make_dense_map(&maps.q, q, dtype, B * Hq, Nq, d) || !make_dense_map(&maps.k, k, dtype, B * Hkv, Nk, d) ||
      !make_dense_map(&maps.v, v, dtype, B * Hkv, Nk, d) || !make_dense_map(&maps.dout, dout, dtype, B * Hq, Nq, d) ||
      !make_acc_map(&maps.dq_acc, p.dq_acc, static_cast<long long>(B) * Hq * Nq, d))
    return ATTN_ERR_CUDA;
  e = attn::launch_bwd_tc(maps, p, dtype, causal != 0, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_bwd_postprocess(p, dtype, s));
}

attn_status_t attn_bwd_varlen(const void* qkv, const void* out, const void* dout, const float* lse,
                              const int32_t* cu_seqlens, int nseq, int total_tokens, int max_seqlen, void* dqkv,
                              void* workspace, size_t workspace_bytes, int H, int d, int causal, float scale,
                              attn_dtype_t dtype, unsigned flags, void* stream) {
  attn_status_t st = check_common(d, scale, dtype);
  if (st != ATTN_OK) return st;
  if (nseq < 0 || total_tokens < 0 || max_seqlen < 0 || H <= 0) return ATTN_ERR_INVALID_ARG;
  if (flags & ~(ATTN_FLAG_OUT_F32 | ATTN_FLAG_DETERMINISTIC)) return ATTN_ERR_INVALID_ARG;
  if (nseq == 0) return total_tokens == 0 ? ATTN_OK : ATTN_ERR_INVALID_ARG;
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return ATTN_ERR_INVALID_ARG;
  if (total_tokens == 0) return ATTN_OK;  // every sequence is empty
  if (max_seqlen == 0) return ATTN_ERR_INVALID_ARG;
  if (!all_aligned16({qkv, out, dout, dqkv}) || !lse || !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_bwd_varlen_workspace_bytes(total_tokens, H, d)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(nseq) * H > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;

  // The sequences are the diagonal blocks of a B = 1, N = total_tokens problem with Hq = Hkv = H.
  BwdParams p{};
  st = bwd_setup(&p, workspace, workspace_bytes, 1, H, H, total_tokens, d, scale, dtype, flags, max_seqlen);
  if (st != ATTN_OK) return st;
  const long long hd = static_cast<long long>(H) * d;
  const BwdParams::Rows packed{3 * hd, d}, rows{hd, d};
  p.lay_q = p.lay_kv = p.lay_dq = p.lay_dkv = packed;
  p.lay_o = rows;
  p.cu_seqlens = cu_seqlens;
  p.nseq = nseq;
  p.max_seqlen = max_seqlen;
  p.n_ktiles = (max_seqlen + attn::kBN - 1) / attn::kBN;
  const size_t es = dtype == ATTN_F32 ? 4 : 2;                 // input element size
  const size_t eo = (dtype == ATTN_F32 || p.out_f32) ? 4 : es;  // output element size
  const char* in = static_cast<const char*>(qkv);
  char* outp = static_cast<char*>(dqkv);
  p.q = in;
  p.k = in + hd * es;
  p.v = in + 2 * hd * es;
  p.o = out;
  p.dout = dout;
  p.lse = lse;
  p.dq = outp;
  p.dk = outp + hd * eo;
  p.dv = outp + 2 * hd * eo;
  if (!(p.status = status_word())) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = attn::launch_bwd_preprocess(p, dtype, dtype != ATTN_F32, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  if (dtype == ATTN_F32) return from_cuda(attn::launch_bwd_f32(p, causal != 0, s));
  BwdMaps maps;
  if (!make_rows_map(&maps.q, p.q, dtype, total_tokens, H, d, 3 * hd, d) ||
      !make_rows_map(&maps.k, p.k, dtype, total_tokens, H, d, 3 * hd, d) ||
      !make_rows_map(&maps.v, p.v, dtype, total_tokens, H, d, 3 * hd, d) ||
      !make_rows_map(&maps.dout, dout, dtype, total_tokens, H, d, hd, d) ||
      !make_acc_map(&maps.dq_acc, p.dq_acc, static_cast<long long>(H) * total_tokens, d))
    return ATTN_ERR_CUDA;
  e = attn::launch_bwd_tc(maps, p, dtype, causal != 0, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return from_cuda(attn::launch_bwd_postprocess(p, dtype, s));
}

namespace {
// Key ranges of the KV-cache forward: the requested count (0: enough work items for about
// eight per SM of a 152-SM GPU), at most one per 128-key tile and at most 128; ranges are
// whole tiles, and trailing empty ranges are dropped.
struct KvSplit {
  int n_splits, tiles_per_split;
};
KvSplit kv_split(int B, int Hq, int Hkv, int Nq, int Nk, int num_splits) {
  const long tiles = (static_cast<long>(Nk) + attn::kBN - 1) / attn::kBN;
  if (tiles <= 0) return {1, 1};
  long want = num_splits;
  if (want <= 0) {
    const long rb = (static_cast<long>(Hq / Hkv) * Nq + attn::kBM - 1) / attn::kBM;
    const long base = static_cast<long>(B) * Hkv * rb;
    want = (8L * 152 + base - 1) / base;
  }
  want = std::min(want, std::min(tiles, 128L));
  if (want < 1) want = 1;
  const long tps = (tiles + want - 1) / want;
  return {static_cast<int>((tiles + tps - 1) / tps), static_cast<int>(tps)};
}
}  // namespace

int attn_fwd_kvcache_splits(int B, int Hq, int Hkv, int Nq, int Nk, int num_splits) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq <= 0 || Nk < 0 || num_splits < 0) return 0;
  return kv_split(B, Hq, Hkv, Nq, Nk, num_splits).n_splits;
}

size_t attn_fwd_kvcache_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int num_splits) {
  const int n = attn_fwd_kvcache_splits(B, Hq, Hkv, Nq, Nk, num_splits);
  if (n <= 0 || d <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * Nq;
  return round256(static_cast<size_t>(n) * rows * d * sizeof(float)) + round256(static_cast<size_t>(n) * rows * sizeof(float));
}

attn_status_t attn_fwd_kvcache(const void* q, const void* k_cache, const void* v_cache, const int32_t* cache_seqlens,
                               void* o, float* lse, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                               int Nq, int Nk, int d, int causal, float scale, int num_splits, attn_dtype_t dtype,
                               unsigned flags, void* stream) {
  attn_status_t st = check_common(d, scale, dtype);
  if (st != ATTN_OK) return st;
  if (B < 0 || Nq < 0 || Nk < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_splits < 0) return ATTN_ERR_INVALID_ARG;
  if (flags & ~ATTN_FLAG_OUT_F32) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Nq == 0) return ATTN_OK;
  // an empty cache (Nk == 0) is never read: its pointers may be null
  if (!q || !o || (Nk > 0 && (!k_cache || !v_cache)) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(o, 16) || !aligned(lse, 4) || !aligned(cache_seqlens, 4))
    return ATTN_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < attn_fwd_kvcache_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, num_splits))
    return ATTN_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  const long long R = static_cast<long long>(G) * Nq;
  const long long bh = static_cast<long long>(B) * Hkv;
  if (R > 0x7fffffffLL || bh * R > 0x7fffffffLL || static_cast<long long>(B) * Hq > 0x7fffffffLL)
    return ATTN_ERR_UNSUPPORTED;
  const KvSplit sp = kv_split(B, Hq, Hkv, Nq, Nk, num_splits);
  const bool f32 = dtype == ATTN_F32;
  const long long n_rb = (R + attn::kBM - 1) / attn::kBM;
  if (f32 ? (Nq + 31) / 32 > 65535 : n_rb * bh * sp.n_splits > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  const size_t rows = static_cast<size_t>(B) * Hq * Nq;

  FwdParams p{};
  p.o = o;
  p.lse = lse;
  p.status = status_word();
  p.wait_ns = wait_limit_ns();
  if (!p.status) return ATTN_ERR_CUDA;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.N = Nk; p.d = d; p.G = G;
  p.Nq = Nq; p.Nk = Nk; p.R = static_cast<int>(R);
  p.cache_seqlens = cache_seqlens;
  p.n_splits = sp.n_splits;
  p.tiles_per_split = sp.tiles_per_split;
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        round256(static_cast<size_t>(sp.n_splits) * rows * d * sizeof(float)));
  p.n_qtiles = static_cast<int>(n_rb);
  p.scale = resolve_scale(scale, d);
  p.scale_log2 = p.scale * kLog2e;
  p.out_f32 = (flags & ATTN_FLAG_OUT_F32) ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Nk > 0) {  // an empty cache: no key for any row, the combine writes O = 0, LSE = -inf
    cudaError_t e;
    if (f32) {
      e = attn::launch_fwd_f32(q, k_cache, v_cache, p, causal != 0, attn::kModeKv, s);
    } else {
      FwdMaps maps;
      if (!make_dense_map(&maps.q, q, dtype, static_cast<int>(bh), static_cast<int>(R), d) ||
          !make_dense_map(&maps.k, k_cache, dtype, static_cast<int>(bh), Nk, d) ||
          !make_dense_map(&maps.v, v_cache, dtype, static_cast<int>(bh), Nk, d))
        return ATTN_ERR_CUDA;
      maps.o = maps.q;  // unused: the partials are stored by the threads
      e = attn::launch_fwd_tc(maps, p, dtype, causal != 0, attn::kModeKv, s);
    }
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return from_cuda(attn::launch_kv_combine(p, dtype, causal != 0, s));
}

attn_status_t attn_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned* w = status_word();
  if (!w) return ATTN_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return static_cast<attn_status_t>(v);
}

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case ATTN_ERR_DEVICE_INPUT: return "invalid cu_seqlens / max_seqlen detected on the device";
  }
  return "unknown status";
}

int attn_version(void) { return 100; }

}  // extern "C"
