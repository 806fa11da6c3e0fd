"""Plain fp64 CPU attention oracle (ctypes loader for attn_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the benchmark's
CPU-baseline leg.  The product package never imports this module, and this module imports
nothing from the product package.

Every function takes and returns float64 NumPy arrays in the layouts of the C source:
dense Q/O/dO/dQ [B,Hq,N,d], K/V/dK/dV [B,Hkv,N,d], LSE [B,Hq,N]; varlen qkv [T,3,H,d],
out [T,H,d], LSE [H,T]; KV cache q/o [B,Hq,Nq,d], k/v [B,Hkv,Nk,d], LSE [B,Hq,Nq].  ``scale=None`` means the default 1/sqrt(d).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)


def compile_source(src_path: str, out_path: str, extra_flags=()) -> str:
    """Compile one oracle C source into a shared library with plain gcc and OpenMP."""
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", *extra_flags,
           "-o", tmp, src_path, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so beside it."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    c_int, c_long, c_double = ctypes.c_int, ctypes.c_long, ctypes.c_double
    lib.oracle_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp] + [c_int] * 6 + [c_double]
    lib.oracle_fwd_rows.argtypes = [_dp, _dp, _dp, _i64p, c_long, _dp, _dp] + [c_int] * 6 + [c_double]
    lib.oracle_probs.argtypes = [_dp, _dp, _dp] + [c_int] * 8 + [c_double]
    lib.oracle_bwd.argtypes = [_dp] * 7 + [c_int] * 6 + [c_double]
    lib.oracle_bwd_sampled.argtypes = ([_dp] * 4 + [_i64p, c_long, _dp, _i64p, c_long, _dp, _dp]
                                       + [c_int] * 6 + [c_double])
    lib.oracle_fwd_varlen.argtypes = [_dp, _i32p, c_int, c_int, _dp, _dp, c_int, c_int, c_int, c_double]
    lib.oracle_fwd_kvcache.argtypes = [_dp, _dp, _dp, _i32p, _dp, _dp] + [c_int] * 7 + [c_double]
    lib.oracle_bwd_cross.argtypes = [_dp] * 7 + [c_int] * 7 + [c_double]
    lib.oracle_num_threads.restype = c_int
    lib.oracle_set_num_threads.argtypes = [c_int]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def load_library(path: str):
    """Bind another build of the oracle source (the mutation tests plant bugs in copies)."""
    return _bind(ctypes.CDLL(path))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _scale(scale):
    return 0.0 if scale is None else float(scale)


def num_threads(lib=None) -> int:
    return (lib or _load()).oracle_num_threads()


def set_num_threads(n: int, lib=None) -> None:
    (lib or _load()).oracle_set_num_threads(int(n))


def _dims(q, k):
    B, Hq, N, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if (Bk, Nk, dk) != (B, N, d):
        raise ValueError("q and k shapes disagree")
    return B, Hq, Hkv, N, d


def fwd(q, k, v, causal: bool, scale=None, lib=None):
    """Returns (O, LSE) for dense inputs."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, N, d = _dims(q, k)
    o = np.empty_like(q)
    lse = np.empty((B, Hq, N))
    lib = lib or _load()
    rc = lib.oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                            B, Hq, Hkv, N, d, int(causal), _scale(scale))
    if rc:
        raise ValueError(f"oracle_fwd rejected its arguments ({rc})")
    return o, lse


def fwd_rows(q, k, v, rows, causal: bool, scale=None, lib=None):
    """O and LSE of selected rows; rows is an int array [n,3] of (b, h, i)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, N, d = _dims(q, k)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    o = np.empty((rows.shape[0], d))
    lse = np.empty(rows.shape[0])
    lib = lib or _load()
    rc = lib.oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), rows.ctypes.data_as(_i64p),
                                 rows.shape[0], _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                                 int(causal), _scale(scale))
    if rc:
        raise ValueError(f"oracle_fwd_rows rejected its arguments ({rc})")
    return o, lse


def probs(q, k, b: int, h: int, causal: bool, scale=None, lib=None):
    """The [N,N] probability matrix P of one (batch, query head)."""
    q, k = _f64(q), _f64(k)
    B, Hq, Hkv, N, d = _dims(q, k)
    P = np.empty((N, N))
    lib = lib or _load()
    rc = lib.oracle_probs(_ptr(q), _ptr(k), _ptr(P), b, h, B, Hq, Hkv, N, d,
                              int(causal), _scale(scale))
    if rc:
        raise ValueError(f"oracle_probs rejected its arguments ({rc})")
    return P


def bwd(q, k, v, dout, causal: bool, scale=None, lib=None):
    """Returns (dQ, dK, dV) for dense inputs and upstream gradient dout."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Hkv, N, d = _dims(q, k)
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    lib = lib or _load()
    rc = lib.oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk),
                            _ptr(dv), B, Hq, Hkv, N, d, int(causal), _scale(scale))
    if rc:
        raise ValueError(f"oracle_bwd rejected its arguments ({rc})")
    return dq, dk, dv


def bwd_sampled(q, k, v, dout, q_rows, k_rows, causal: bool, scale=None, lib=None):
    """dQ of selected query rows (b,h,i) and dK, dV of selected key rows (b,g,j)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Hkv, N, d = _dims(q, k)
    q_rows = np.ascontiguousarray(np.asarray(q_rows, dtype=np.int64).reshape(-1, 3))
    k_rows = np.ascontiguousarray(np.asarray(k_rows, dtype=np.int64).reshape(-1, 3))
    dq = np.empty((q_rows.shape[0], d))
    dk = np.empty((k_rows.shape[0], d))
    dv = np.empty((k_rows.shape[0], d))
    lib = lib or _load()
    rc = lib.oracle_bwd_sampled(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                    q_rows.ctypes.data_as(_i64p), q_rows.shape[0], _ptr(dq),
                                    k_rows.ctypes.data_as(_i64p), k_rows.shape[0], _ptr(dk),
                                    _ptr(dv), B, Hq, Hkv, N, d, int(causal), _scale(scale))
    if rc:
        raise ValueError(f"oracle_bwd_sampled rejected its arguments ({rc})")
    return dq, dk, dv


def fwd_varlen(qkv, cu_seqlens, causal: bool, scale=None, lib=None):
    """Returns (out [T,H,d], LSE [H,T]) for packed qkv [T,3,H,d] and cu_seqlens [nseq+1]."""
    qkv = _f64(qkv)
    T, three, H, d = qkv.shape
    if three != 3:
        raise ValueError("qkv must be [T,3,H,d]")
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    out = np.empty((T, H, d))
    lse = np.empty((H, T))
    lib = lib or _load()
    rc = lib.oracle_fwd_varlen(_ptr(qkv), cu.ctypes.data_as(_i32p), cu.shape[0] - 1, T,
                                   _ptr(out), _ptr(lse), H, d, int(causal), _scale(scale))
    if rc:
        raise ValueError(f"oracle_fwd_varlen rejected its arguments ({rc})")
    return out, lse


def fwd_kvcache(q, k, v, cache_seqlens, causal: bool, scale=None, lib=None):
    """Returns (O [B,Hq,Nq,d], LSE [B,Hq,Nq]) for queries q against caches k, v [B,Hkv,Nk,d]
    holding cache_seqlens[b] valid keys (None: all Nk); causal aligns the queries with the
    last Nq cache positions.  Rows that see no key: O = 0, LSE = -inf."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if (Bk, dk) != (B, d) or v.shape != k.shape:
        raise ValueError("q, k and v shapes disagree")
    lens = None
    if cache_seqlens is not None:
        lens = np.ascontiguousarray(np.asarray(cache_seqlens, dtype=np.int32).reshape(-1))
        if lens.shape[0] != B:
            raise ValueError("cache_seqlens must have B entries")
    o = np.empty((B, Hq, Nq, d))
    lse = np.empty((B, Hq, Nq))
    lib = lib or _load()
    rc = lib.oracle_fwd_kvcache(_ptr(q), _ptr(k), _ptr(v),
                                None if lens is None else lens.ctypes.data_as(_i32p),
                                _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d, int(causal), _scale(scale))
    if rc:
        raise ValueError(f"oracle_fwd_kvcache rejected its arguments ({rc})")
    return o, lse


def bwd_cross(q, k, v, dout, causal: bool, scale=None, lib=None):
    """(dQ [B,Hq,Nq,d], dK, dV [B,Hkv,Nk,d]) of the cross-attention forward (fwd_kvcache with
    full caches) for the upstream gradient dout [B,Hq,Nq,d]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk_ = k.shape
    if (Bk, dk_) != (B, d) or v.shape != k.shape or dout.shape != q.shape:
        raise ValueError("q, k, v and dout shapes disagree")
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    lib = lib or _load()
    rc = lib.oracle_bwd_cross(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                              B, Hq, Hkv, Nq, Nk, d, int(causal), _scale(scale))
    if rc:
        raise ValueError(f"oracle_bwd_cross rejected its arguments ({rc})")
    return dq, dk, dv
