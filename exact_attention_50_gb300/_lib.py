"""ctypes binding of libattn_gb300.so: the C ABI of include/attn.h, one Python function per
entry point with the same name.  Argument marshalling only; all compute runs in the library.
There is no fallback: if the library is missing or fails to load, every call raises."""
from __future__ import annotations

import ctypes
import os

from . import build as _build

ATTN_F32, ATTN_F16, ATTN_BF16 = 0, 1, 2
ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_DEVICE_INPUT = 5
ATTN_FLAG_OUT_F32 = 1
ATTN_FLAG_DETERMINISTIC = 2

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Loads the built library (build it with exact_attention_50_gb300.build.build())."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing "
                               "(run exact_attention_50_gb300.build.build())")
        lib = ctypes.CDLL(path)
        vp, i, f, u = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, u, vp]
        lib.attn_fwd.restype = i
        lib.attn_fwd_varlen.argtypes = [vp, vp, i, i, i, vp, vp, i, i, i, f, i, u, vp]
        lib.attn_fwd_varlen.restype = i
        lib.attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
        lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_bwd.argtypes = [vp] * 10 + [ctypes.c_size_t, i, i, i, i, i, i, f, i, u, vp]
        lib.attn_bwd.restype = i
        lib.attn_bwd_prepare.argtypes = [vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, vp]
        lib.attn_bwd_prepare.restype = i
        lib.attn_bwd_main.argtypes = [vp] * 9 + [ctypes.c_size_t, i, i, i, i, i, i, f, i, u, vp]
        lib.attn_bwd_main.restype = i
        lib.attn_bwd_finish.argtypes = [vp, vp, ctypes.c_size_t, i, i, i, i, f, i, u, vp]
        lib.attn_bwd_finish.restype = i
        lib.attn_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, i, u, vp]
        lib.attn_bwd_noalloc.restype = i
        lib.attn_bwd_varlen_workspace_bytes.argtypes = [i, i, i]
        lib.attn_bwd_varlen_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp, vp, ctypes.c_size_t, i, i, i, f, i, u, vp]
        lib.attn_bwd_varlen.restype = i
        lib.attn_fwd_kvcache_splits.argtypes = [i, i, i, i, i, i]
        lib.attn_fwd_kvcache_splits.restype = i
        lib.attn_fwd_kvcache_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.attn_fwd_kvcache_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_fwd_kvcache.argtypes = [vp] * 7 + [ctypes.c_size_t] + [i] * 7 + [f, i, i, u, vp]
        lib.attn_fwd_kvcache.restype = i
        lib.attn_bwd_cross_workspace_bytes.argtypes = [i, i, i, i, i, i, u]
        lib.attn_bwd_cross_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_bwd_cross.argtypes = [vp] * 10 + [ctypes.c_size_t] + [i] * 7 + [f, i, u, vp]
        lib.attn_bwd_cross.restype = i
        lib.attn_get_device_status.argtypes = [vp]
        lib.attn_get_device_status.restype = i
        lib.attn_status_string.argtypes = [i]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_version.restype = i
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, where)


def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, dtype, flags, stream) -> int:
    return load().attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, int(causal), float(scale), dtype, flags, stream)


def attn_fwd_varlen(qkv, cu_seqlens, nseq, total_tokens, max_seqlen, out, lse, H, d, causal, scale, dtype,
                    flags, stream) -> int:
    return load().attn_fwd_varlen(qkv, cu_seqlens, nseq, total_tokens, max_seqlen, out, lse, H, d, int(causal),
                                  float(scale), dtype, flags, stream)


def attn_fwd_kvcache_splits(B, Hq, Hkv, Nq, Nk, num_splits) -> int:
    return load().attn_fwd_kvcache_splits(B, Hq, Hkv, Nq, Nk, num_splits)


def attn_fwd_kvcache_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, num_splits) -> int:
    return load().attn_fwd_kvcache_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, num_splits)


def attn_fwd_kvcache(q, k_cache, v_cache, cache_seqlens, o, lse, workspace, workspace_bytes, B, Hq, Hkv, Nq, Nk, d,
                     causal, scale, num_splits, dtype, flags, stream) -> int:
    return load().attn_fwd_kvcache(q, k_cache, v_cache, cache_seqlens, o, lse, workspace, workspace_bytes, B, Hq, Hkv,
                                   Nq, Nk, d, int(causal), float(scale), int(num_splits), dtype, flags, stream)


def attn_bwd_cross_workspace_bytes(B, Hq, Nq, Nk, d, dtype, flags) -> int:
    return load().attn_bwd_cross_workspace_bytes(B, Hq, Nq, Nk, d, dtype, flags)


def attn_bwd_cross(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, Nq, Nk, d, causal,
                   scale, dtype, flags, stream) -> int:
    return load().attn_bwd_cross(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, Nq, Nk,
                                 d, int(causal), float(scale), dtype, flags, stream)


def attn_bwd_workspace_bytes(B, Hq, N, d) -> int:
    return load().attn_bwd_workspace_bytes(B, Hq, N, d)


def attn_bwd_varlen_workspace_bytes(total_tokens, H, d) -> int:
    return load().attn_bwd_varlen_workspace_bytes(total_tokens, H, d)


def attn_bwd_varlen(qkv, out, dout, lse, cu_seqlens, nseq, total_tokens, max_seqlen, dqkv, workspace,
                    workspace_bytes, H, d, causal, scale, dtype, flags, stream) -> int:
    return load().attn_bwd_varlen(qkv, out, dout, lse, cu_seqlens, nseq, total_tokens, max_seqlen, dqkv, workspace,
                                  workspace_bytes, H, d, int(causal), float(scale), dtype, flags, stream)


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, d, causal, scale,
             dtype, flags, stream) -> int:
    return load().attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, d,
                           int(causal), float(scale), dtype, flags, stream)


def attn_bwd_prepare(o, dout, workspace, workspace_bytes, B, Hq, N, d, dtype, stream) -> int:
    return load().attn_bwd_prepare(o, dout, workspace, workspace_bytes, B, Hq, N, d, dtype, stream)


def attn_bwd_main(q, k, v, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, d, causal, scale,
                  dtype, flags, stream) -> int:
    return load().attn_bwd_main(q, k, v, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, d,
                                int(causal), float(scale), dtype, flags, stream)


def attn_bwd_finish(dq, workspace, workspace_bytes, B, Hq, N, d, scale, dtype, flags, stream) -> int:
    return load().attn_bwd_finish(dq, workspace, workspace_bytes, B, Hq, N, d, float(scale), dtype, flags, stream)


def attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, dtype, flags,
                     stream) -> int:
    """attn_bwd without a caller workspace (a fixed 64 MiB scratch array inside the library)."""
    return load().attn_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, int(causal), float(scale),
                                   dtype, flags, stream)


def attn_get_device_status(stream) -> int:
    return load().attn_get_device_status(stream)


def attn_status_string(status: int) -> str:
    return status_string(status)


def attn_version() -> int:
    return load().attn_version()
