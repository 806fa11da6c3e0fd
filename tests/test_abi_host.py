"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports every
function include/attn.h declares, and rejects bad arguments with status codes before it
touches the device."""
import ctypes
import math
import os
import re

import pytest

from exact_attention_50_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_varlen", "attn_bwd", "attn_bwd_workspace_bytes", "attn_get_device_status",
              "attn_status_string", "attn_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_version_and_status_strings(lib):
    assert _lib.attn_version() >= 100
    for code in range(6):
        assert _lib.status_string(code)
    assert _lib.status_string(42) == "unknown status"


def _fwd(**kw):
    a = dict(q=8, k=8, v=8, o=8, lse=None, B=1, Hq=2, Hkv=1, N=16, d=64, causal=0, scale=0.0,
             dtype=_lib.ATTN_BF16, flags=0, stream=None)
    a.update(kw)
    # fake, 16-byte aligned host addresses: every case below must be rejected before any use
    for key in ("q", "k", "v", "o"):
        if a[key] == 8:
            a[key] = 4096
    return _lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"], a["d"],
                         a["causal"], a["scale"], a["dtype"], a["flags"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), _lib.ATTN_ERR_INVALID_ARG),
    (dict(o=None), _lib.ATTN_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), _lib.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), _lib.ATTN_ERR_INVALID_ARG),
    (dict(N=-5), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(d=24), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(d=144), _lib.ATTN_ERR_UNSUPPORTED),
    (dict(scale=-1.0), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=math.nan), _lib.ATTN_ERR_INVALID_ARG),
    (dict(scale=math.inf), _lib.ATTN_ERR_INVALID_ARG),
    (dict(dtype=7), _lib.ATTN_ERR_INVALID_ARG),
    (dict(flags=4), _lib.ATTN_ERR_INVALID_ARG),
    (dict(q=4100), _lib.ATTN_ERR_INVALID_ARG),   # not 16-byte aligned
    (dict(lse=4098), _lib.ATTN_ERR_INVALID_ARG),  # not 4-byte aligned
    (dict(B=0), _lib.ATTN_OK),                    # empty: nothing to launch
    (dict(N=0), _lib.ATTN_OK),
])
def test_fwd_rejects_bad_arguments(lib, kw, code):
    assert _fwd(**kw) == code


def test_varlen_validation(lib):
    f = lambda **kw: _lib.attn_fwd_varlen(kw.get("qkv", 4096), kw.get("cu", 4096), kw.get("nseq", 2),
                                          kw.get("T", 12), kw.get("maxlen", 7), kw.get("out", 4096), None,
                                          kw.get("H", 2), kw.get("d", 64), 0, 0.0, _lib.ATTN_BF16, 0, None)
    assert f(nseq=-1) == _lib.ATTN_ERR_INVALID_ARG
    assert f(nseq=0, T=0) == _lib.ATTN_OK
    assert f(nseq=0, T=3) == _lib.ATTN_ERR_INVALID_ARG
    assert f(cu=None) == _lib.ATTN_ERR_INVALID_ARG
    assert f(T=0) == _lib.ATTN_OK
    assert f(maxlen=0) == _lib.ATTN_ERR_INVALID_ARG
    assert f(qkv=None) == _lib.ATTN_ERR_INVALID_ARG
    assert f(H=0) == _lib.ATTN_ERR_INVALID_ARG
    assert f(d=40) == _lib.ATTN_ERR_UNSUPPORTED


def test_bwd_workspace_and_validation(lib):
    ws = _lib.attn_bwd_workspace_bytes(2, 4, 100, 64)
    rows = 2 * 4 * 100
    r256 = lambda x: (x + 255) // 256 * 256
    assert ws == r256(rows * 64 * 4) + 2 * r256(rows * 4)  # dQ acc, D, turn counters
    assert _lib.attn_bwd_workspace_bytes(0, 4, 100, 64) == 0
    args = [4096] * 10 + [ws, 2, 4, 2, 100, 64, 1, 0.0, _lib.ATTN_BF16, 0, None]
    small = list(args)
    small[10] = ws - 1
    assert _lib.attn_bwd(*small) == _lib.ATTN_ERR_INVALID_ARG
    nolse = list(args)
    nolse[5] = None
    assert _lib.attn_bwd(*nolse) == _lib.ATTN_ERR_INVALID_ARG
    misaligned_ws = list(args)
    misaligned_ws[9] = 4096 + 128
    assert _lib.attn_bwd(*misaligned_ws) == _lib.ATTN_ERR_INVALID_ARG
    empty = list(args)
    empty[14] = 0
    assert _lib.attn_bwd(*empty) == _lib.ATTN_OK


def test_python_wrapper_rejects_unsupported_flags():
    import torch
    from exact_attention_50_gb300 import flash_attn_varlen_qkvpacked_func
    qkv = torch.zeros(12, 3, 2, 64)
    cu = torch.tensor([0, 5, 12], dtype=torch.int32)
    for kw in (dict(window_size=(4, 4)), dict(softcap=1.0), dict(alibi_slopes=torch.zeros(2)),
               dict(return_attn_probs=True), dict(dropout_p=0.1)):
        with pytest.raises(ValueError):
            flash_attn_varlen_qkvpacked_func(qkv, cu, 7, **kw)
    with pytest.raises(ValueError, match="Token count mismatch"):
        flash_attn_varlen_qkvpacked_func(torch.zeros(11, 3, 2, 64), cu, 7)


def test_bwd_varlen_workspace_and_validation(lib):
    T, H, d = 300, 2, 64
    ws = _lib.attn_bwd_varlen_workspace_bytes(T, H, d)
    assert ws == _lib.attn_bwd_workspace_bytes(1, H, T, d)
    f = lambda **kw: _lib.attn_bwd_varlen(kw.get("qkv", 4096), kw.get("out", 4096), kw.get("dout", 4096),
                                          kw.get("lse", 4096), kw.get("cu", 4096), kw.get("nseq", 2),
                                          kw.get("T", T), kw.get("maxlen", 200), kw.get("dqkv", 4096),
                                          kw.get("ws", 4096), kw.get("wsb", ws), kw.get("H", H), kw.get("d", d),
                                          0, 0.0, _lib.ATTN_BF16, kw.get("flags", 0), None)
    assert f(nseq=-1) == _lib.ATTN_ERR_INVALID_ARG
    assert f(nseq=0, T=0) == _lib.ATTN_OK
    assert f(nseq=0, T=3) == _lib.ATTN_ERR_INVALID_ARG
    assert f(T=0) == _lib.ATTN_OK
    assert f(cu=None) == _lib.ATTN_ERR_INVALID_ARG
    assert f(maxlen=0) == _lib.ATTN_ERR_INVALID_ARG
    assert f(dqkv=None) == _lib.ATTN_ERR_INVALID_ARG
    assert f(lse=None) == _lib.ATTN_ERR_INVALID_ARG
    assert f(dout=4100) == _lib.ATTN_ERR_INVALID_ARG   # not 16-byte aligned
    assert f(ws=4096 + 128) == _lib.ATTN_ERR_INVALID_ARG  # not 256-byte aligned
    assert f(wsb=ws - 1) == _lib.ATTN_ERR_INVALID_ARG
    assert f(H=0) == _lib.ATTN_ERR_INVALID_ARG
    assert f(d=40) == _lib.ATTN_ERR_UNSUPPORTED
    assert f(flags=4) == _lib.ATTN_ERR_INVALID_ARG


def test_kvcache_splits_workspace_and_validation(lib):
    S = _lib.attn_fwd_kvcache_splits
    # 0 = about eight work items per SM of a 152-SM GPU: 64 (batch, kv head) blocks of one row
    # block over 256 key tiles -> 19 ranges of 14 tiles
    assert S(8, 32, 8, 1, 32768, 0) == 19
    assert S(1, 8, 8, 1, 300, 0) == 3           # at most one range per 128-key tile
    assert S(2, 4, 2, 1, 1000, 5) == 4          # 8 tiles in ranges of 2: the empty 5th is dropped
    assert S(1, 1, 1, 1, 128, 7) == 1
    assert S(1, 1, 1, 1, 0, 0) == 1             # an empty cache still has one (empty) range
    assert S(1, 3, 2, 1, 64, 0) == 0 and S(1, 2, 1, 0, 64, 0) == 0 and S(1, 2, 1, 1, 64, -1) == 0
    r256 = lambda x: (x + 255) // 256 * 256
    ws = _lib.attn_fwd_kvcache_workspace_bytes(2, 4, 2, 3, 1000, 64, 5)
    rows = 2 * 4 * 3
    assert ws == r256(4 * rows * 64 * 4) + r256(4 * rows * 4)

    def f(**kw):
        a = dict(q=4096, k=4096, v=4096, lens=None, o=4096, lse=None, ws=4096, wsb=ws, B=2, Hq=4, Hkv=2, Nq=3,
                 Nk=1000, d=64, causal=1, scale=0.0, splits=5, dtype=_lib.ATTN_BF16, flags=0)
        a.update(kw)
        return _lib.attn_fwd_kvcache(a["q"], a["k"], a["v"], a["lens"], a["o"], a["lse"], a["ws"], a["wsb"], a["B"],
                                     a["Hq"], a["Hkv"], a["Nq"], a["Nk"], a["d"], a["causal"], a["scale"],
                                     a["splits"], a["dtype"], a["flags"], None)
    assert f(B=0) == _lib.ATTN_OK and f(Nq=0) == _lib.ATTN_OK
    assert f(q=None) == _lib.ATTN_ERR_INVALID_ARG
    assert f(k=None) == _lib.ATTN_ERR_INVALID_ARG and f(v=None) == _lib.ATTN_ERR_INVALID_ARG
    assert f(k=4100) == _lib.ATTN_ERR_INVALID_ARG      # not 16-byte aligned
    assert f(lens=4098) == _lib.ATTN_ERR_INVALID_ARG   # not 4-byte aligned
    assert f(lse=4098) == _lib.ATTN_ERR_INVALID_ARG
    assert f(ws=None) == _lib.ATTN_ERR_INVALID_ARG
    assert f(ws=4096 + 128) == _lib.ATTN_ERR_INVALID_ARG
    assert f(wsb=ws - 1) == _lib.ATTN_ERR_INVALID_ARG
    assert f(Hq=3) == _lib.ATTN_ERR_INVALID_ARG
    assert f(Nk=-1) == _lib.ATTN_ERR_INVALID_ARG
    assert f(splits=-1) == _lib.ATTN_ERR_INVALID_ARG
    assert f(d=40) == _lib.ATTN_ERR_UNSUPPORTED
    assert f(flags=2) == _lib.ATTN_ERR_INVALID_ARG
    assert f(scale=-1.0) == _lib.ATTN_ERR_INVALID_ARG


def test_bwd_cross_workspace_and_validation(lib):
    W = _lib.attn_bwd_cross_workspace_bytes
    # the kernels walk Nq x Nk directly: the workspace is attn_bwd's for the Nq query rows
    for Nq, Nk in ((100, 100), (100, 300), (301, 300), (1, 5000)):
        for flags in (0, _lib.ATTN_FLAG_OUT_F32):
            assert W(2, 4, Nq, Nk, 64, _lib.ATTN_BF16, flags) == _lib.attn_bwd_workspace_bytes(2, 4, Nq, 64)
    assert W(2, 4, 0, 300, 64, _lib.ATTN_BF16, 0) == 0
    ws = W(2, 4, 100, 300, 64, _lib.ATTN_BF16, 0)

    def f(**kw):
        a = dict(p=4096, lse=4096, ws=4096, wsb=ws, B=2, Hq=4, Hkv=2, Nq=100, Nk=300, d=64, flags=0)
        a.update(kw)
        return _lib.attn_bwd_cross(a["p"], a["p"], a["p"], a["p"], a["p"], a["lse"], a["p"], a["p"], a["p"], a["ws"],
                                   a["wsb"], a["B"], a["Hq"], a["Hkv"], a["Nq"], a["Nk"], a["d"], 1, 0.0,
                                   _lib.ATTN_BF16, a["flags"], None)
    assert f(B=0) == _lib.ATTN_OK and f(Nq=0, Nk=0) == _lib.ATTN_OK
    assert f(Nq=301, wsb=W(2, 4, 301, 300, 64, _lib.ATTN_BF16, 0) - 1) == _lib.ATTN_ERR_INVALID_ARG
    assert f(p=4100) == _lib.ATTN_ERR_INVALID_ARG
    assert f(lse=None) == _lib.ATTN_ERR_INVALID_ARG
    assert f(wsb=ws - 1) == _lib.ATTN_ERR_INVALID_ARG
    assert f(ws=4096 + 128) == _lib.ATTN_ERR_INVALID_ARG
    assert f(Hq=3) == _lib.ATTN_ERR_INVALID_ARG
    assert f(flags=4) == _lib.ATTN_ERR_INVALID_ARG
