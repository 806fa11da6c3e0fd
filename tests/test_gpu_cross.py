"""GPU parity of the cross-attention backward (attn_bwd_cross, Nq < Nk, bottom-right causal
alignment) against the fp64 oracle, its identity with attn_bwd at Nq = Nk, autograd through
flash_attention with Nq != Nk, the deterministic flag, and the refusal of Nq > Nk."""
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


def inputs(B, Hq, Hkv, Nq, Nk, d, dtype, seed):
    q, k, v, _ = W.kvcache_inputs(B, Hq, Hkv, Nq, Nk, d, dtype, None, seed=seed)
    g = W.generator(seed + 500)
    dout = torch.randn(B, Hq, Nq, d, generator=g, dtype=torch.float32).to(W.DTYPES[dtype])
    return q, k, v, dout


@pytest.mark.parametrize("dtype,d,Nq,Nk", [("bf16", 128, 300, 520), ("f16", 64, 130, 700), ("f32", 64, 33, 100),
                                           ("bf16", 80, 1, 257)])
@pytest.mark.parametrize("causal", [False, True])
def test_cross_bwd_matches_oracle(dev, dtype, d, Nq, Nk, causal):
    tdt = W.DTYPES[dtype]
    q, k, v, dout = inputs(2, 4, 2, Nq, Nk, d, dtype, seed=61)
    qd, kd, vd, dd = q.to(dev), k.to(dev), v.to(dev), dout.to(dev)
    o, lse = A.fwd_kvcache(qd, kd, vd, None, causal)
    g32 = A.bwd_cross(qd, kd, vd, o, lse, dd, causal, out_f32=True)
    gn = A.bwd_cross(qd, kd, vd, o, lse, dd, causal)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    refs = oracle.bwd_cross(to_np(q), to_np(k), to_np(v), to_np(dout), causal)
    for name, a, b, r in zip(("dQ", "dK", "dV"), g32, gn, refs):
        what = f"cross bwd {dtype} d={d} Nq={Nq} Nk={Nk} causal={causal} {name}"
        assert_close_f32(a, r, tdt, what + " (fp32)")
        assert_close_native(b, r, tdt, what)


def test_square_cross_is_dense_backward(dev):
    q, k, v, dout = (t.to(dev) for t in W.dense_inputs(1, 4, 2, 384, 128, "bf16", seed=62))
    o, lse = A.fwd(q, k, v, True)
    a = A.bwd_cross(q, k, v, o, lse, dout, True, deterministic=True)
    b = A.bwd(q, k, v, o, lse, dout, True, deterministic=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_cross_autograd_and_determinism(dev):
    from exact_attention_50_gb300 import flash_attention
    q, k, v, dout = (t.to(dev) for t in inputs(1, 8, 2, 200, 650, 128, "bf16", seed=63))
    grads = []
    for _ in range(2):
        qq, kk, vv = (t.detach().clone().requires_grad_() for t in (q, k, v))
        out = flash_attention(qq, kk, vv, causal=True, deterministic=True)
        out.backward(dout)
        grads.append((qq.grad, kk.grad, vv.grad))
    o2, lse2 = A.fwd_kvcache(q, k, v, None, True)
    direct = A.bwd_cross(q, k, v, o2, lse2, dout, True, deterministic=True)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    assert torch.equal(out.detach(), o2)
    assert all(torch.equal(x, y) for x, y in zip(grads[0], grads[1]))
    assert all(torch.equal(x, y) for x, y in zip(grads[0], direct))


def test_cross_bwd_refuses_more_queries_than_keys(dev):
    q, k, v, dout = (t.to(dev) for t in inputs(1, 2, 1, 10, 5, 64, "bf16", seed=64))
    o, lse = A.fwd_kvcache(q, k, v, None, False)
    with pytest.raises(_lib.AttnError):
        A.bwd_cross(q, k, v, o, lse, dout, False)
