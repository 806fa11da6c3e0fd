/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact attention library (libattn_gb300.so).
 *
 * The library computes exact scaled-dot-product attention IO-aware: Q.K^T is tiled, the
 * softmax runs online (running row max and sum) and P.V accumulates on chip, so the N x N
 * score matrix never reaches HBM.  Sources for what each call computes:
 *   - "AMD GPU에서도 동작하는 FlashAttention 구현체, Aule-Attention" (jeff.news/article/688),
 *     API list: tensors [batch, heads, seq_len, head_dim]; causal masks future tokens; scale
 *     defaults to 1/sqrt(head_dim); head_dim <= 128; float16, bfloat16 and float32; query heads
 *     a multiple of kv heads (GQA).
 *   - "跨平台注意力神器AuleAttention把FlashAttention从CUDA解放出来" (jdon.com/83460), sections on
 *     calling flash_attention (causal forward, loss.backward()) and on GQA / MQA.
 *   - Turing varlen article (ewbang.com/community/article/details/1000323363), section on the
 *     core code: flash_attn_varlen_qkvpacked_func's packed qkv [total_tokens,3,heads,head_dim],
 *     cu_seqlens [batch+1] and output [total_tokens,heads,head_dim].
 *   - Attention-operator article (m.xxqk.cn/news/636956) section 2.2: Q/K/V tiles staged on
 *     chip, the softmax max-subtracted in registers, only the output written back.
 *   - FlashAttention-T review (ai-stack.site), best practices 2 and 4 (scale/mask fused into the
 *     GEMM loop; online max/sum kept so the backward can restore the normalisation) and FAQ 4
 *     (the backward recomputes scores rather than storing them).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous, 16-byte
 *     aligned.  The library allocates no device memory in these calls; the backward's scratch
 *     is a caller-provided workspace.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream).  Argument errors are returned before anything is launched.
 *   - Errors found on the device (a pipeline wait that timed out, invalid cu_seqlens) are
 *     recorded in a per-device status word and returned by attn_get_device_status().  Every
 *     device-side wait is bounded: 4 s by default, or ATTN_WAIT_LIMIT_MS milliseconds (10 to
 *     600000) from the environment as read at the library's first call.  A CTA whose wait runs
 *     out stops and reports ATTN_ERR_TIMEOUT; the CUDA context stays usable.
 *   - scale == 0 selects the default 1/sqrt(d); a negative or NaN scale is rejected.
 *   - d must be a multiple of 16 in [16, 128]; Hq must be a multiple of Hkv; query head h uses
 *     kv head h / (Hq / Hkv).
 *   - dtype selects the element type of q/k/v/o/dout/dq/dk/dv.  ATTN_F16 / ATTN_BF16 run on the
 *     5th-generation tensor cores (tcgen05) with fp32 accumulation and an fp32 softmax;
 *     ATTN_F32 runs an fp32 CUDA-core path.
 *   - flags: ATTN_FLAG_OUT_F32 makes the outputs (o; dq, dk, dv) float32 regardless of dtype:
 *     the fp32 value the kernel holds before the final rounding to dtype.
 */
#ifndef EXACT_ATTENTION_GB300_ATTN_H
#define EXACT_ATTENTION_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_F32 = 0, ATTN_F16 = 1, ATTN_BF16 = 2 } attn_dtype_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, Hq % Hkv != 0, ... */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid but not provided: d not a multiple of 16 or above 128 */
  ATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed (launch, tensor map, ...) */
  ATTN_ERR_TIMEOUT = 4,      /* device: a pipeline wait exceeded its time limit; CTA stopped */
  ATTN_ERR_DEVICE_INPUT = 5  /* device: cu_seqlens not non-decreasing from 0, a sequence
                                longer than max_seqlen, or a cache length outside [0, Nk] */
} attn_status_t;

#define ATTN_FLAG_OUT_F32 1u
/* Backward only (attn_bwd, attn_bwd_main, attn_bwd_varlen, attn_bwd_noalloc): dq is bitwise
 * reproducible from run to run.  The key tiles add their parts of each 128-row dQ tile into the
 * fp32 accumulator in key-tile order (each waits, on the device and bounded, for the one
 * before it) instead of in the order they arrive; slower.  dk, dv and the fp32 path are
 * reproducible in either mode. */
#define ATTN_FLAG_DETERMINISTIC 2u

/*
 * Forward: O = softmax(scale * Q K^T, causally masked) V for every (batch, query head), tiled so
 * the N x N scores stay on chip.  Defining passages: the attention-operator article
 * (m.xxqk.cn/news/636956) section 2.1 (S = Q K^T, softmax, P V) and section 2.2 (the tiled form
 * that writes only O back); the Aule-Attention summary (jeff.news/article/688), API list (layout
 * [batch, heads, seq_len, head_dim], causal, default scale 1/sqrt(head_dim), head_dim <= 128,
 * GQA); the FlashAttention-T review, best practice 4 (running max and sum, kept so the
 * normalisation can be restored: the LSE below).
 *   q    [B, Hq,  N, d]   k, v [B, Hkv, N, d]   (dtype)
 *   o    [B, Hq,  N, d]   (dtype, or float32 with ATTN_FLAG_OUT_F32)
 *   lse  [B, Hq,  N] float32, nullable: natural-log log-sum-exp of the scaled, masked scores
 *        of each query row (LSE_i = m_i + ln sum_j exp(S_ij - m_i)), as the backward needs it.
 *   causal != 0 masks key j for query i when j > i.
 * B == 0 or N == 0 is a valid empty call that launches nothing.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                       int Hkv, int N, int d, int causal, float scale, attn_dtype_t dtype, unsigned flags,
                       void* stream);

/*
 * Forward on packed variable-length sequences (flash_attn_varlen_qkvpacked_func semantics:
 * Turing varlen article (ewbang.com/community/article/details/1000323363), the function's
 * argument list and its pseudo-code, which runs every sequence of cu_seqlens as its own
 * attention problem and returns the packed [total_tokens, heads, head_dim] output).
 *   qkv         [total_tokens, 3, H, d] (dtype): plane 0 = q, 1 = k, 2 = v
 *   cu_seqlens  DEVICE int32 [nseq + 1]: 0-based prefix sums, cu_seqlens[nseq] == total_tokens;
 *               sequence s is tokens [cu_seqlens[s], cu_seqlens[s+1]); indices (and the causal
 *               mask) are relative to the sequence start.  Zero-length sequences are allowed.
 *   max_seqlen  an upper bound on every sequence length (sizes the launch grid)
 *   out         [total_tokens, H, d] (dtype, or float32 with ATTN_FLAG_OUT_F32)
 *   lse         [H, total_tokens] float32, nullable
 * A cu_seqlens array that is not non-decreasing from 0, or a sequence longer than max_seqlen,
 * is detected on the device: the affected work is skipped and attn_get_device_status()
 * returns ATTN_ERR_DEVICE_INPUT.
 */
attn_status_t attn_fwd_varlen(const void* qkv, const int32_t* cu_seqlens, int nseq, int total_tokens,
                              int max_seqlen, void* out, float* lse, int H, int d, int causal, float scale,
                              attn_dtype_t dtype, unsigned flags, void* stream);

/* Bytes of device workspace attn_bwd needs for these sizes (an fp32 dQ accumulator
 * [B,Hq,N,d], the fp32 row terms D_i = dO_i . O_i [B,Hq,N] and int32 turn counters [B,Hq,N]
 * for ATTN_FLAG_DETERMINISTIC, each 256-byte aligned). */
size_t attn_bwd_workspace_bytes(int B, int Hq, int N, int d);

/*
 * Backward: given dout = dL/dO, writes dq [B,Hq,N,d], dk and dv [B,Hkv,N,d] (dtype, or float32
 * with ATTN_FLAG_OUT_F32).  Defining passages: the Aule-Attention article (jdon.com/83460),
 * the training example (loss.backward() through flash_attention gives the gradients of q, k
 * and v); the FlashAttention-T review, FAQ 4 (the backward recomputes the score matrix from
 * Q, K and the saved normalisation instead of storing it).  With P_ij = exp(S_ij - LSE_i),
 * D_i = dO_i . O_i and dS_ij = P_ij (dO_i . V_j - D_i): dV_j = sum_i P_ij dO_i,
 * dK_j = scale sum_i dS_ij Q_i, dQ_i = scale sum_j dS_ij K_j.  q, k, v, o are the forward's inputs and output and lse its
 * float32 LSE; P is recomputed from q, k and lse (nothing of size N x N is stored).  dk and
 * dv of a kv head sum the contributions of every query head of its group.
 *   workspace  DEVICE, at least attn_bwd_workspace_bytes(B, Hq, N, d) bytes, 256-byte aligned;
 *              contents on entry are ignored, on exit undefined.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                       int B, int Hq, int Hkv, int N, int d, int causal, float scale, attn_dtype_t dtype,
                       unsigned flags, void* stream);

/*
 * The backward as three steps on one stream (attn_bwd runs all three; calling them separately
 * lets a caller time or schedule them).  All take the same workspace.
 *   attn_bwd_prepare: D_i = dO_i . O_i (fp32) into the workspace, and for fp16/bf16 zeroes
 *                     the fp32 dQ accumulator.
 *   attn_bwd_main:    the fused recompute-and-reduce kernel: dk, dv (final) and, for
 *                     fp16/bf16, the dQ accumulator in the workspace.  For ATTN_F32 it writes
 *                     dq (float32) directly.
 *   attn_bwd_finish:  dq = scale * accumulator, rounded to dtype (or float32 with
 *                     ATTN_FLAG_OUT_F32); nothing for ATTN_F32.
 * The argument rules are those of attn_bwd.
 */
attn_status_t attn_bwd_prepare(const void* o, const void* dout, void* workspace, size_t workspace_bytes, int B,
                               int Hq, int N, int d, attn_dtype_t dtype, void* stream);
attn_status_t attn_bwd_main(const void* q, const void* k, const void* v, const void* dout, const float* lse, void* dq,
                            void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                            int N, int d, int causal, float scale, attn_dtype_t dtype, unsigned flags,
                            void* stream);
attn_status_t attn_bwd_finish(void* dq, void* workspace, size_t workspace_bytes, int B, int Hq, int N, int d,
                              float scale, attn_dtype_t dtype, unsigned flags, void* stream);

/* Bytes of device workspace attn_bwd_varlen needs (an fp32 dQ accumulator [H, total_tokens, d],
 * the fp32 row terms [H, total_tokens] and int32 turn counters [H, total_tokens], each
 * 256-byte aligned). */
size_t attn_bwd_varlen_workspace_bytes(int total_tokens, int H, int d);

/*
 * Backward of attn_fwd_varlen (the training side of flash_attn_varlen_qkvpacked_func, per the
 * Turing varlen article's packed layout; the recompute follows the FlashAttention-T review,
 * FAQ 4).  Each sequence is differentiated on its own, as attn_bwd would for a batch of one.
 *   qkv, cu_seqlens, nseq, total_tokens, max_seqlen, H, d, causal, scale, dtype: as given to
 *               attn_fwd_varlen
 *   out, lse    its output [total_tokens, H, d] (dtype) and LSE [H, total_tokens] float32
 *   dout        dL/dout [total_tokens, H, d] (dtype)
 *   dqkv        [total_tokens, 3, H, d]: plane 0 = dq, 1 = dk, 2 = dv (dtype, or float32 with
 *               ATTN_FLAG_OUT_F32); rows of zero-length sequences are not written
 *   workspace   DEVICE, at least attn_bwd_varlen_workspace_bytes(total_tokens, H, d) bytes,
 *               256-byte aligned; contents on entry are ignored, on exit undefined.
 * Argument errors return a status before any launch; a cu_seqlens array that is not
 * non-decreasing from 0 or a sequence longer than max_seqlen is detected on the device: the
 * affected work is skipped and attn_get_device_status() returns ATTN_ERR_DEVICE_INPUT.
 */
attn_status_t attn_bwd_varlen(const void* qkv, const void* out, const void* dout, const float* lse,
                              const int32_t* cu_seqlens, int nseq, int total_tokens, int max_seqlen, void* dqkv,
                              void* workspace, size_t workspace_bytes, int H, int d, int causal, float scale,
                              attn_dtype_t dtype, unsigned flags, void* stream);

/*
 * Backward of cross-attention (the KV-cache forward above without cache lengths): gradients of
 * q [B,Hq,Nq,d] and of k, v [B,Hkv,Nk,d] for the forward's output o and LSE (natural log,
 * [B,Hq,Nq]) and dL/do, for any Nq and Nk, with the same bottom-right causal alignment: query i
 * sees key j iff j <= i + Nk - Nq.  The FlashAttention-T review names blocked KV-cache
 * computation (FAQ 4) and the prefill phase (practical advice 2); the gradients are the
 * backward's formulas restricted to the keys each query sees.  The backward kernels walk the
 * Nq x Nk problem directly (no padded copies); a query row that sees no key (Nq > Nk under the
 * causal mask, or Nk == 0) gets dq = 0, and with Nq == 0, dk = dv = 0.
 *   workspace  DEVICE, at least attn_bwd_cross_workspace_bytes(B, Hq, Nq, Nk, d, dtype, flags)
 *              bytes (that of attn_bwd for Nq query rows), 256-byte aligned
 * Nq == Nk is attn_bwd.  Flags, layouts and the other argument rules are those of attn_bwd.
 */
size_t attn_bwd_cross_workspace_bytes(int B, int Hq, int Nq, int Nk, int d, attn_dtype_t dtype, unsigned flags);
attn_status_t attn_bwd_cross(const void* q, const void* k, const void* v, const void* o, const void* dout,
                             const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                             attn_dtype_t dtype, unsigned flags, void* stream);

/*
 * KV cache / cross-attention forward: Nq queries per (batch, query head) against a cache of up to
 * Nk keys per (batch, kv head) (the FlashAttention-T review, FAQ 4: at inference the KV cache is
 * computed in blocks; its practical advice 2: the prefill and decode phases).  Decode is Nq = 1
 * (or a few), prefill against a cache and cross-attention are larger Nq.
 *   q              [B, Hq, Nq, d] (dtype)
 *   k_cache, v_cache [B, Hkv, Nk, d] (dtype)
 *   cache_seqlens  DEVICE int32 [B] or NULL: batch b's cache holds its first cache_seqlens[b]
 *                  keys (0 <= cache_seqlens[b] <= Nk); NULL means Nk keys for every batch
 *   o              [B, Hq, Nq, d] (dtype, or float32 with ATTN_FLAG_OUT_F32)
 *   lse            [B, Hq, Nq] float32 (natural log), or NULL
 *   causal         query i sees key j only when j <= L - Nq + i (L = the batch's cache length):
 *                  the queries are the last Nq positions of the sequence (bottom-right
 *                  alignment); with Nq == L this is the self-attention mask of attn_fwd
 *   num_splits     key ranges per (batch, kv head), merged by their LSE (split-KV); 0 picks a
 *                  count from the sizes (attn_fwd_kvcache_splits); at most one per 128 keys
 *   workspace      DEVICE, at least attn_fwd_kvcache_workspace_bytes(...) bytes with the same
 *                  sizes and num_splits, 256-byte aligned; contents on entry are ignored
 * A query row that sees no key (an empty cache, or L < Nq under the causal mask) gets O = 0 and
 * LSE = -inf.  B == 0 or Nq == 0 is a no-op.  A cache_seqlens entry outside [0, Nk] is detected
 * on the device: that batch is treated as empty and attn_get_device_status() returns
 * ATTN_ERR_DEVICE_INPUT.  Other argument rules are those of attn_fwd.
 */
int attn_fwd_kvcache_splits(int B, int Hq, int Hkv, int Nq, int Nk, int num_splits);
size_t attn_fwd_kvcache_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int num_splits);
attn_status_t attn_fwd_kvcache(const void* q, const void* k_cache, const void* v_cache, const int32_t* cache_seqlens,
                               void* o, float* lse, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                               int Nq, int Nk, int d, int causal, float scale, int num_splits, attn_dtype_t dtype,
                               unsigned flags, void* stream);

/*
 * attn_bwd_noalloc -- the backward (same arguments, layouts and results as attn_bwd) for callers
 * that cannot allocate device memory when they call it: for example a plugin or host program
 * whose GPU memory is reserved up front by another allocator and may not grow on its hot path,
 * or a runtime that forbids allocation calls after start-up.  The pages describe no such call;
 * it exists only for such callers.
 *   - Scratch comes from a fixed 64 MiB array inside this library (not from the caller and not
 *     from any allocator).  Every GPU that loads the library holds that array until the process
 *     exits.  No call on this path allocates or frees device memory.
 *   - Sizes are limited by it: when attn_bwd_workspace_bytes(B, Hq, N, d) exceeds 64 MiB
 *     (67108864 bytes; at d = 128 that is about 129,000 query rows B*Hq*N) the call returns
 *     ATTN_ERR_UNSUPPORTED and launches nothing.
 *   - The first call on each device looks up the array's device address (a one-time set-up on
 *     that device, made while it is current); make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents; each call clears the
 *     part that must start at zero itself.  Calls whose execution overlaps on the GPU (other
 *     streams, or other host threads) race on the array and give wrong results: order them.
 *   - The cached address belongs to the device's primary context (the one the CUDA runtime
 *     uses).  Do not call it from a different driver context, and not after cudaDeviceReset
 *     in the same process: the address would no longer be valid there.
 */
attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                               int d, int causal, float scale, attn_dtype_t dtype, unsigned flags, void* stream);

/* Synchronises `stream`, then returns and clears the first error the current device's
 * kernels recorded (ATTN_OK when none).  Returns ATTN_ERR_CUDA if the synchronisation fails. */
attn_status_t attn_get_device_status(void* stream);

/* A static, human-readable name for a status code. */
const char* attn_status_string(attn_status_t status);

/* Library ABI version (major * 100 + minor). */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_GB300_ATTN_H */
