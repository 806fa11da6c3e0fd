"""GPU checks of the deterministic backward (ATTN_FLAG_DETERMINISTIC): dq, dk and dv are bitwise
the same from run to run (dense, GQA, ragged N, causal or not; varlen; many key tiles per dQ
tile), they match the oracle within tolerance, and differ from the default mode's result only
by the fp32 summation order of dQ."""
import pytest
import torch

import oracle
from exact_attention_50_gb300 import _lib, build
from exact_attention_50_gb300 import attention as A
from exact_attention_50_gb300 import workloads as W
from tests.parity import assert_close_f32, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    _lib.load()
    return torch.device("cuda:0")


def status_ok():
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK


@pytest.mark.parametrize("causal", [True, False])
def test_dense_repeatable_and_matches_oracle(dev, causal):
    B, Hq, Hkv, N, d = 2, 8, 2, 1100, 128  # 9 key tiles, a ragged last one
    q, k, v, dout = (t.to(dev) for t in W.dense_inputs(B, Hq, Hkv, N, d, "bf16", seed=51))
    o, lse = A.fwd(q, k, v, causal)
    runs = [A.bwd(q, k, v, o, lse, dout, causal, out_f32=True, deterministic=True) for _ in range(3)]
    status_ok()
    for r in runs[1:]:
        for name, a, b in zip(("dQ", "dK", "dV"), runs[0], r):
            assert torch.equal(a, b), f"{name} differs between deterministic runs"
    default = A.bwd(q, k, v, o, lse, dout, causal, out_f32=True)
    status_ok()
    assert (runs[0][0] - default[0]).abs().max().item() <= 1e-4  # dQ: summation order only
    assert torch.equal(runs[0][1], default[1]) and torch.equal(runs[0][2], default[2])
    refs = oracle.bwd(to_np(q[:1]), to_np(k[:1]), to_np(v[:1]), to_np(dout[:1]), causal)
    for name, g, r in zip(("dQ", "dK", "dV"), runs[0], refs):
        assert_close_f32(g[:1], r, torch.bfloat16, f"deterministic bwd causal={causal} batch 0 {name}")


def test_many_key_tiles_per_dq_tile(dev):
    """32 key tiles add into the last dQ tiles of every head, in order."""
    q, k, v, dout = (t.to(dev) for t in W.dense_inputs(1, 4, 1, 4096, 64, "f16", seed=52))
    o, lse = A.fwd(q, k, v, True)
    a = A.bwd(q, k, v, o, lse, dout, True, deterministic=True)
    b = A.bwd(q, k, v, o, lse, dout, True, deterministic=True)
    status_ok()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_varlen_repeatable(dev):
    qkv, cu, lengths, dout = W.varlen_inputs([300, 77, 600, 129], 3, 64, "bf16", seed=53, with_dout=True)
    qkv, cu, dout = qkv.to(dev), cu.to(dev), dout.to(dev)
    out, lse = A.fwd_varlen(qkv, cu, max(lengths), True)
    g1 = A.bwd_varlen(qkv, out, lse, dout, cu, max(lengths), True, out_f32=True, deterministic=True)
    g2 = A.bwd_varlen(qkv, out, lse, dout, cu, max(lengths), True, out_f32=True, deterministic=True)
    gd = A.bwd_varlen(qkv, out, lse, dout, cu, max(lengths), True, out_f32=True)
    status_ok()
    assert torch.equal(g1, g2)
    assert (g1 - gd).abs().max().item() <= 1e-4


def test_autograd_flag(dev):
    from exact_attention_50_gb300 import flash_attention
    q, k, v, dout = (t.to(dev) for t in W.dense_inputs(1, 4, 2, 700, 128, "bf16", seed=54))
    grads = []
    for _ in range(2):
        qq, kk, vv = (t.detach().clone().requires_grad_() for t in (q, k, v))
        flash_attention(qq, kk, vv, causal=True, deterministic=True).backward(dout)
        grads.append((qq.grad, kk.grad, vv.grad))
    status_ok()
    assert all(torch.equal(x, y) for x, y in zip(*grads))
