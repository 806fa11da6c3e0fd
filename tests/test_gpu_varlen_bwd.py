"""GPU parity of the packed varlen backward (attn_bwd_varlen), through the C ABI: every sequence
against the fp64 oracle's dense backward of that sequence alone, dK / dV identical to the
library's dense backward of the sequence alone (the sequences are independent problems), the
device-side cu_seqlens check, and autograd through flash_attn_varlen_qkvpacked_func."""
import pytest
import torch

import oracle
from exact_attention_50_gb300 import _lib, build
from exact_attention_50_gb300 import attention as A
from exact_attention_50_gb300 import workloads as W
from tests.parity import assert_close_f32, assert_close_native, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    _lib.load()
    return torch.device("cuda:0")


def dense(x):
    """[L, H, d] rows of one sequence -> the dense [1, H, L, d] layout."""
    return x.permute(1, 0, 2).unsqueeze(0).contiguous()


def inputs(lengths, H, d, dtype, seed):
    qkv, cu, lengths, _ = W.varlen_inputs(lengths, H, d, dtype, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    dout = torch.randn(qkv.shape[0], H, d, generator=g).to(W.DTYPES[dtype])
    return qkv, cu, lengths, dout


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 64), ("bf16", 80)])
@pytest.mark.parametrize("causal", [True, False])
def test_varlen_bwd_matches_oracle(dev, dtype, d, causal):
    # an empty sequence, a single token, exact and ragged tiles
    qkv, cu, lengths, dout = inputs([130, 0, 1, 257, 128], 2, d, dtype, seed=21)
    tdt = W.DTYPES[dtype]
    qkv_d, cu_d, dout_d = qkv.to(dev), cu.to(dev), dout.to(dev)
    maxlen = max(lengths)
    out, lse = A.fwd_varlen(qkv_d, cu_d, maxlen, causal)
    g32 = A.bwd_varlen(qkv_d, out, lse, dout_d, cu_d, maxlen, causal, out_f32=True)
    gn = A.bwd_varlen(qkv_d, out, lse, dout_d, cu_d, maxlen, causal)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    cu_l = cu.tolist()
    for s, L in enumerate(lengths):
        if L == 0:
            continue
        a, b = cu_l[s], cu_l[s + 1]
        q, k, v = (dense(qkv[a:b, i]) for i in range(3))
        refs = oracle.bwd(to_np(q), to_np(k), to_np(v), to_np(dense(dout[a:b])), causal)
        for plane, name, r in zip(range(3), ("dQ", "dK", "dV"), refs):
            what = f"varlen bwd {dtype} d={d} causal={causal} seq {s} (L={L}) {name}"
            assert_close_f32(dense(g32[a:b, plane]), r, tdt, what + " (fp32)")
            assert_close_native(dense(gn[a:b, plane]), r, tdt, what)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_varlen_bwd_equals_dense_per_sequence(dev, dtype):
    """dK and dV of each sequence are bitwise those of a dense backward of that sequence alone
    (same kernel decomposition; dQ is reduced with atomics, so it is compared within tolerance)."""
    qkv, cu, lengths, dout = inputs([300, 77, 129], 3, 128 if dtype == "bf16" else 64, dtype, seed=22)
    tdt = W.DTYPES[dtype]
    qkv_d, cu_d, dout_d = qkv.to(dev), cu.to(dev), dout.to(dev)
    maxlen = max(lengths)
    out, lse = A.fwd_varlen(qkv_d, cu_d, maxlen, True)
    dqkv = A.bwd_varlen(qkv_d, out, lse, dout_d, cu_d, maxlen, True)
    cu_l = cu.tolist()
    for s in range(len(lengths)):
        a, b = cu_l[s], cu_l[s + 1]
        q, k, v = (dense(qkv_d[a:b, i]) for i in range(3))
        o_s, lse_s = dense(out[a:b]), lse[:, a:b].unsqueeze(0).contiguous()
        dq, dk, dv = A.bwd(q, k, v, o_s, lse_s, dense(dout_d[a:b]), True)
        assert torch.equal(dense(dqkv[a:b, 1]), dk), f"seq {s} dK differs from the dense backward"
        assert torch.equal(dense(dqkv[a:b, 2]), dv), f"seq {s} dV differs from the dense backward"
        err = (dense(dqkv[a:b, 0]).double() - dq.double()).abs().max().item()
        assert err <= (1e-6 if dtype == "f32" else 2.0 ** -7 * 4), f"seq {s} dQ differs by {err}"
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK


def test_varlen_bwd_invalid_cu_seqlens_reported_by_device(dev):
    qkv, cu, lengths, dout = inputs([40, 60], 2, 64, "bf16", seed=23)
    qkv_d, cu_d, dout_d = qkv.to(dev), cu.to(dev), dout.to(dev)
    out, lse = A.fwd_varlen(qkv_d, cu_d, 60, False)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    bad = torch.tensor([0, 70, 100], dtype=torch.int32, device=dev)  # a sequence longer than max_seqlen
    A.bwd_varlen(qkv_d, out, lse, dout_d, bad, 60, False)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_ERR_DEVICE_INPUT
    assert A.get_device_status() == _lib.ATTN_OK  # reading clears it


def test_varlen_autograd_matches_direct_call(dev):
    from exact_attention_50_gb300 import flash_attn_varlen_qkvpacked_func
    qkv, cu, lengths, dout = inputs([5, 7, 150], 4, 64, "f16", seed=24)
    qkv_d = qkv.to(dev).requires_grad_()
    cu_d, dout_d = cu.to(dev), dout.to(dev)
    out = flash_attn_varlen_qkvpacked_func(qkv_d, cu_d, max(lengths), causal=True)
    out.backward(dout_d)
    o2, lse2 = A.fwd_varlen(qkv_d.detach(), cu_d, max(lengths), True)
    direct = A.bwd_varlen(qkv_d.detach(), o2, lse2, dout_d, cu_d, max(lengths), True)
    assert torch.equal(out.detach(), o2)
    dq_err = (qkv_d.grad[:, 0].double() - direct[:, 0].double()).abs().max().item()
    assert torch.equal(qkv_d.grad[:, 1:], direct[:, 1:]) and dq_err <= 2e-3
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
