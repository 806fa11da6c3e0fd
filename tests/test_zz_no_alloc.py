"""The allocation-free backward entry point (attn_bwd_noalloc), for callers that cannot allocate
device memory when they call it.  It must give the results of attn_bwd with a caller-allocated
workspace, on consecutive calls (the fixed scratch array keeps the previous call's contents),
and refuse sizes beyond its fixed capacity without launching anything.  This file sorts last so
that a run stopping at its first failure has already run every other test."""
import pytest
import torch

from exact_attention_50_gb300 import _lib, build
from exact_attention_50_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    _lib.load()
    return torch.device("cuda:0")


def _fwd(q, k, v, causal, dtype_code, stream):
    B, Hq, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, N, dtype=torch.float32, device=q.device)
    st = _lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, k.shape[1], N,
                       d, causal, 0.0, dtype_code, 0, stream)
    assert st == _lib.ATTN_OK
    return o, lse


def _grads(q, k, v, dtype):
    return tuple(torch.empty(t.shape, dtype=dtype, device=t.device) for t in (q, k, v))


@pytest.mark.parametrize("dtype,causal,deterministic", [("bf16", True, False), ("f16", False, False),
                                                        ("bf16", True, True)])
def test_noalloc_backward_matches_workspace_backward_twice(dev, dtype, causal, deterministic):
    """Same kernels on the same inputs as attn_bwd: dK and dV bitwise equal on both calls; dQ
    bitwise equal in the deterministic mode (whose per-tile turn counters live in the shared
    scratch array and must be reset by each call).  Otherwise the dQ tiles are added into the
    fp32 accumulator in arrival order, so the two runs are compared on their fp32 results
    (ATTN_FLAG_OUT_F32): dK and dV bitwise, dQ within 1e-5, where fp32 reordering noise of
    values of order one lies (about 1e-6) and a scratch-layout error would not."""
    B, Hq, Hkv, N, d = 2, 8, 2, 1000, 128
    code = {"bf16": _lib.ATTN_BF16, "f16": _lib.ATTN_F16}[dtype]
    flags = _lib.ATTN_FLAG_DETERMINISTIC if deterministic else _lib.ATTN_FLAG_OUT_F32
    odt = W.DTYPES[dtype] if deterministic else torch.float32
    stream = torch.cuda.current_stream().cuda_stream
    q, k, v, dout = (t.to(dev) for t in W.dense_inputs(B, Hq, Hkv, N, d, dtype, seed=5))
    o, lse = _fwd(q, k, v, causal, code, stream)
    # the existing entry point, workspace allocated by the caller
    nbytes = _lib.attn_bwd_workspace_bytes(B, Hq, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ref = _grads(q, k, v, odt)
    st = _lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                       *(g.data_ptr() for g in ref), ws.data_ptr(), nbytes, B, Hq, Hkv, N, d, causal, 0.0, code,
                       flags, stream)
    assert st == _lib.ATTN_OK
    # the allocation-free entry point, twice in a row
    for call in range(2):
        out = _grads(q, k, v, odt)
        st = _lib.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                                   lse.data_ptr(), *(g.data_ptr() for g in out), B, Hq, Hkv, N, d, causal, 0.0, code,
                                   flags, stream)
        assert st == _lib.ATTN_OK
        torch.cuda.synchronize()
        assert _lib.attn_get_device_status(stream) == _lib.ATTN_OK
        for name, a, r in zip(("dQ", "dK", "dV"), out, ref):
            assert bool(torch.isfinite(a).all()), (call, name)
            if name == "dQ" and not deterministic:
                err = float((a.double() - r.double()).abs().max())
                assert err <= 1e-5, f"call {call} dQ: {err:.3e} from attn_bwd"
            else:
                assert torch.equal(a, r), f"call {call} {name}: not bitwise equal to attn_bwd"


def test_noalloc_refuses_sizes_beyond_its_scratch(dev):
    # 1 x 32 x 8192 rows at d = 128 needs about 137 MB of scratch, more than the fixed 64 MiB
    B, Hq, Hkv, N, d = 1, 32, 8, 8192, 128
    assert _lib.attn_bwd_workspace_bytes(B, Hq, N, d) > 64 * 2 ** 20
    p = 4096  # never dereferenced: the size check comes first
    st = _lib.attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, Hq, Hkv, N, d, 1, 0.0, _lib.ATTN_BF16, 0, None)
    assert st == _lib.ATTN_ERR_UNSUPPORTED
