"""PyTorch-facing API over the C ABI.  PyTorch supplies device memory and the current stream;
every step of the computation runs in libattn_gb300.so's kernels.

- ``flash_attention(q, k, v, causal=True, scale=None)``: [batch, heads, seq, head_dim] tensors,
  GQA when k/v have fewer heads, differentiable (Aule-Attention API, jeff.news/article/688:
  causal defaults to True, scale to 1/sqrt(head_dim)).
- ``flash_attn_varlen_qkvpacked_func(qkv, cu_seqlens, max_seqlen, ...)``: packed variable-length
  forward with the flash_attn signature (Turing varlen article, ewbang.com/...1000323363:
  causal defaults to False; window_size, softcap, alibi_slopes and return_attn_probs are
  rejected; dropout is not provided).
- ``fwd``, ``bwd``, ``fwd_varlen``: explicit calls that also return the LSE / take workspaces.
"""
from __future__ import annotations

import math

import torch

from . import _lib

_DT = {torch.float32: _lib.ATTN_F32, torch.float16: _lib.ATTN_F16, torch.bfloat16: _lib.ATTN_BF16}


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}: float16, bfloat16 or float32")
    return _DT[t.dtype]


def _require(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _scale_arg(scale) -> float:
    if scale is None:
        return 0.0
    scale = float(scale)
    if not (scale > 0.0) or math.isinf(scale):
        raise ValueError("scale must be a positive finite number (None = 1/sqrt(head_dim))")
    return scale


def get_device_status() -> int:
    """Synchronises the current stream and returns/clears the device status word."""
    return _lib.attn_get_device_status(_stream())


def fwd(q, k, v, causal: bool, scale=None, out_f32: bool = False, with_lse: bool = True):
    """Dense forward.  q [B,Hq,N,d]; k, v [B,Hkv,N,d].  Returns (o, lse or None)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, q.dtype)
    if q.dim() != 4 or k.shape != v.shape or k.dim() != 4:
        raise ValueError("q must be [B,Hq,N,d] and k, v [B,Hkv,N,d]")
    B, Hq, N, d = q.shape
    if k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError("q and k/v disagree on batch, sequence length or head_dim")
    Hkv = k.shape[1]
    o = torch.empty(q.shape, dtype=torch.float32 if out_f32 else q.dtype, device=q.device)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if with_lse else None
    st = _lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                       lse.data_ptr() if lse is not None else None, B, Hq, Hkv, N, d, causal,
                       _scale_arg(scale), _dtype_code(q), _lib.ATTN_FLAG_OUT_F32 if out_f32 else 0, _stream())
    _lib._check(st, "attn_fwd")
    return o, lse


def _bwd_flags(out_f32: bool, deterministic: bool) -> int:
    return (_lib.ATTN_FLAG_OUT_F32 if out_f32 else 0) | (_lib.ATTN_FLAG_DETERMINISTIC if deterministic else 0)


def bwd(q, k, v, o, lse, dout, causal: bool, scale=None, out_f32: bool = False, workspace=None,
        deterministic: bool = False):
    """Dense backward.  Returns (dq, dk, dv).  deterministic: dq bitwise reproducible (slower)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _require(t, n, q.dtype)
    _require(lse, "lse", torch.float32)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if o.shape != q.shape or dout.shape != q.shape or lse.shape != (B, Hq, N):
        raise ValueError("o and dout must be shaped like q, lse [B,Hq,N]")
    odt = torch.float32 if out_f32 else q.dtype
    dq = torch.empty(q.shape, dtype=odt, device=q.device)
    dk = torch.empty(k.shape, dtype=odt, device=q.device)
    dv = torch.empty(v.shape, dtype=odt, device=q.device)
    nbytes = _lib.attn_bwd_workspace_bytes(B, Hq, N, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    st = _lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), workspace.numel(),
                       B, Hq, Hkv, N, d, causal, _scale_arg(scale), _dtype_code(q),
                       _bwd_flags(out_f32, deterministic), _stream())
    _lib._check(st, "attn_bwd")
    return dq, dk, dv


def bwd_cross(q, k, v, o, lse, dout, causal: bool, scale=None, out_f32: bool = False, workspace=None,
              deterministic: bool = False):
    """Cross-attention backward (any Nq, Nk; bottom-right causal alignment: query i sees key j
    iff j <= i + Nk - Nq).  q, o, dout [B,Hq,Nq,d]; k, v [B,Hkv,Nk,d]; lse [B,Hq,Nq] from
    fwd_kvcache without cache lengths.  Query rows that see no key get dq = 0.
    Returns (dq, dk, dv)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _require(t, n, q.dtype)
    _require(lse, "lse", torch.float32)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    if v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape or lse.shape != (B, Hq, Nq):
        raise ValueError("o and dout must be shaped like q, v like k, lse [B,Hq,Nq]")
    odt = torch.float32 if out_f32 else q.dtype
    dq = torch.empty(q.shape, dtype=odt, device=q.device)
    dk = torch.empty(k.shape, dtype=odt, device=q.device)
    dv = torch.empty(v.shape, dtype=odt, device=q.device)
    flags = _bwd_flags(out_f32, deterministic)
    nbytes = _lib.attn_bwd_cross_workspace_bytes(B, Hq, Nq, Nk, d, _dtype_code(q), flags)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    st = _lib.attn_bwd_cross(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), workspace.numel(),
                             B, Hq, Hkv, Nq, Nk, d, causal, _scale_arg(scale), _dtype_code(q), flags, _stream())
    _lib._check(st, "attn_bwd_cross")
    return dq, dk, dv


def fwd_varlen(qkv, cu_seqlens, max_seqlen: int, causal: bool, scale=None, out_f32: bool = False,
               with_lse: bool = True):
    """Packed varlen forward.  qkv [T,3,H,d], cu_seqlens int32 [nseq+1] (device).
    Returns (out [T,H,d], lse [H,T] or None)."""
    _require(qkv, "qkv")
    _require(cu_seqlens, "cu_seqlens", torch.int32)
    if qkv.dim() != 4 or qkv.shape[1] != 3:
        raise ValueError("qkv must be [total_tokens, 3, heads, head_dim]")
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be 1-D with batch_size + 1 entries")
    T, _, H, d = qkv.shape
    nseq = cu_seqlens.numel() - 1
    out = torch.empty((T, H, d), dtype=torch.float32 if out_f32 else qkv.dtype, device=qkv.device)
    lse = torch.empty((H, T), dtype=torch.float32, device=qkv.device) if with_lse else None
    st = _lib.attn_fwd_varlen(qkv.data_ptr(), cu_seqlens.data_ptr(), nseq, T, int(max_seqlen), out.data_ptr(),
                              lse.data_ptr() if lse is not None else None, H, d, causal, _scale_arg(scale),
                              _dtype_code(qkv), _lib.ATTN_FLAG_OUT_F32 if out_f32 else 0, _stream())
    _lib._check(st, "attn_fwd_varlen")
    return out, lse


def bwd_varlen(qkv, out, lse, dout, cu_seqlens, max_seqlen: int, causal: bool, scale=None, out_f32: bool = False,
               workspace=None, deterministic: bool = False):
    """Packed varlen backward.  qkv [T,3,H,d], out / dout [T,H,d], lse [H,T] (from fwd_varlen),
    cu_seqlens int32 [nseq+1] (device).  Returns dqkv [T,3,H,d]."""
    _require(qkv, "qkv")
    for t, n in ((out, "out"), (dout, "dout")):
        _require(t, n, qkv.dtype)
    _require(lse, "lse", torch.float32)
    _require(cu_seqlens, "cu_seqlens", torch.int32)
    T, _, H, d = qkv.shape
    if out.shape != (T, H, d) or dout.shape != (T, H, d) or lse.shape != (H, T):
        raise ValueError("out and dout must be [T,H,d], lse [H,T]")
    nseq = cu_seqlens.numel() - 1
    dqkv = torch.zeros(qkv.shape, dtype=torch.float32 if out_f32 else qkv.dtype, device=qkv.device)
    nbytes = _lib.attn_bwd_varlen_workspace_bytes(T, H, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=qkv.device)
    st = _lib.attn_bwd_varlen(qkv.data_ptr(), out.data_ptr(), dout.data_ptr(), lse.data_ptr(), cu_seqlens.data_ptr(),
                              nseq, T, int(max_seqlen), dqkv.data_ptr(), workspace.data_ptr(), workspace.numel(), H,
                              d, causal, _scale_arg(scale), _dtype_code(qkv),
                              _bwd_flags(out_f32, deterministic), _stream())
    _lib._check(st, "attn_bwd_varlen")
    return dqkv


def kvcache_workspace_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, num_splits: int = 0) -> int:
    """Bytes of the device workspace fwd_kvcache needs for these sizes and num_splits."""
    return _lib.attn_fwd_kvcache_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, num_splits)


def fwd_kvcache(q, k_cache, v_cache, cache_seqlens=None, causal: bool = False, scale=None, num_splits: int = 0,
                out_f32: bool = False, with_lse: bool = True, workspace=None):
    """KV-cache / cross-attention forward.  q [B,Hq,Nq,d]; k_cache, v_cache [B,Hkv,Nk,d];
    cache_seqlens int32 [B] on the device (None: Nk keys each).  causal aligns the queries with
    the last Nq keys of each cache.  num_splits: key ranges per (batch, kv head), 0 = chosen
    from the sizes.  Returns (o [B,Hq,Nq,d], lse [B,Hq,Nq] or None)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _require(t, n, q.dtype)
    if q.dim() != 4 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("q must be [B,Hq,Nq,d] and k_cache, v_cache [B,Hkv,Nk,d]")
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, dk = k_cache.shape
    if k_cache.shape[0] != B or dk != d:
        raise ValueError("q and the caches disagree on batch or head_dim")
    lens_ptr = None
    if cache_seqlens is not None:
        _require(cache_seqlens, "cache_seqlens", torch.int32)
        if cache_seqlens.shape != (B,) or cache_seqlens.device != q.device:
            raise ValueError("cache_seqlens must be int32 [B] on q's device")
        lens_ptr = cache_seqlens.data_ptr()
    o = torch.empty(q.shape, dtype=torch.float32 if out_f32 else q.dtype, device=q.device)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device) if with_lse else None
    need = _lib.attn_fwd_kvcache_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, num_splits) if B * Nq > 0 else 0
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    elif workspace.numel() < need:
        raise ValueError(f"workspace too small: {workspace.numel()} < {need} bytes")
    st = _lib.attn_fwd_kvcache(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), lens_ptr, o.data_ptr(),
                               lse.data_ptr() if lse is not None else None, workspace.data_ptr(), workspace.numel(),
                               B, Hq, Hkv, Nq, Nk, d, causal, _scale_arg(scale), num_splits, _dtype_code(q),
                               _lib.ATTN_FLAG_OUT_F32 if out_f32 else 0, _stream())
    _lib._check(st, "attn_fwd_kvcache")
    return o, lse


class _AttnFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale, deterministic):
        # queries and keys of different lengths: cross-attention (bottom-right causal alignment)
        ctx.cross = q.dim() == 4 and k.dim() == 4 and q.shape[2] != k.shape[2]
        if ctx.cross:
            o, lse = fwd_kvcache(q, k, v, None, causal, scale)
        else:
            o, lse = fwd(q, k, v, causal, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale, ctx.deterministic = causal, scale, deterministic
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse = ctx.saved_tensors
        call = bwd_cross if ctx.cross else bwd
        dq, dk, dv = call(q, k, v, o, lse, dout.contiguous(), ctx.causal, ctx.scale, deterministic=ctx.deterministic)
        return dq, dk, dv, None, None, None


def flash_attention(q, k, v, causal: bool = True, scale=None, deterministic: bool = False):
    """Exact attention of [B,Hq,Nq,d] queries over [B,Hkv,Nk,d] keys/values (Hq % Hkv == 0).
    Nq != Nk is cross-attention, with the causal mask aligned to the last Nq keys.
    deterministic makes the backward's dq bitwise reproducible (slower)."""
    return _AttnFn.apply(q, k, v, causal, scale, bool(deterministic))


class _VarlenFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, qkv, cu_seqlens, max_seqlen, causal, scale, deterministic):
        out, lse = fwd_varlen(qkv, cu_seqlens, max_seqlen, causal, scale)
        ctx.save_for_backward(qkv, out, lse, cu_seqlens)
        ctx.max_seqlen, ctx.causal, ctx.scale, ctx.deterministic = max_seqlen, causal, scale, deterministic
        return out

    @staticmethod
    def backward(ctx, dout):
        qkv, out, lse, cu_seqlens = ctx.saved_tensors
        dqkv = bwd_varlen(qkv, out, lse, dout.contiguous(), cu_seqlens, ctx.max_seqlen, ctx.causal, ctx.scale,
                          deterministic=ctx.deterministic)
        return dqkv, None, None, None, None, None


def flash_attn_varlen_qkvpacked_func(qkv, cu_seqlens, max_seqlen, dropout_p=0.0, softmax_scale=None,
                                     causal=False, window_size=(-1, -1), softcap=0.0, alibi_slopes=None,
                                     deterministic=False, return_attn_probs=False):
    """flash_attn's packed varlen call: qkv [total_tokens,3,H,d], cu_seqlens [batch+1] -> [total_tokens,H,d]."""
    if tuple(window_size) != (-1, -1):
        raise ValueError("window_size is not supported (must be (-1, -1))")
    if softcap != 0.0:
        raise ValueError("softcap is not supported (must be 0.0)")
    if alibi_slopes is not None:
        raise ValueError("alibi_slopes is not supported (must be None)")
    if return_attn_probs:
        raise ValueError("return_attn_probs is not supported (must be False)")
    if dropout_p != 0.0:
        raise ValueError("dropout is not supported (dropout_p must be 0.0)")
    if not isinstance(qkv, torch.Tensor) or qkv.dim() != 4 or qkv.shape[1] != 3:
        raise ValueError("Bad qkv shape")
    if cu_seqlens is None or cu_seqlens.dim() != 1:
        raise ValueError("Bad cu_seqlens")
    if cu_seqlens.numel() - 1 <= 0:
        raise ValueError("Bad batch size")
    if qkv.shape[0] != int(cu_seqlens[-1].item()):
        raise ValueError("Token count mismatch")
    return _VarlenFn.apply(qkv, cu_seqlens.to(torch.int32), int(max_seqlen), bool(causal), softmax_scale,
                           bool(deterministic))
