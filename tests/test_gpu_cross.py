"""GPU parity of the cross-attention backward (attn_bwd_cross, Nq != Nk, bottom-right causal
alignment) against the fp64 oracle -- fewer queries than keys (prefill against a cache) and
more queries than keys (causal rows that see no key get no gradient) -- its identity with
attn_bwd at Nq = Nk, autograd through flash_attention with Nq != Nk and the deterministic flag."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_50_gb300 import _lib, build
from exact_attention_50_gb300 import attention as A
from exact_attention_50_gb300 import workloads as W
from tests.parity import TOL, assert_close_f32, assert_close_native, to_np

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
                                           ("bf16", 80, 1, 257), ("bf16", 128, 520, 300), ("f16", 64, 700, 130),
                                           ("f32", 64, 100, 33), ("bf16", 128, 257, 1), ("bf16", 64, 128, 256),
                                           ("f16", 128, 384, 128)])
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


def test_cross_bwd_empty_sides(dev):
    """No query: dk = dv = 0.  No key: every row sees nothing, dq = 0."""
    q, k, v, dout = (t.to(dev) for t in inputs(1, 2, 1, 10, 6, 64, "bf16", seed=64))
    z = q[:, :, :0].contiguous()
    dz = dout[:, :, :0].contiguous()
    lz = torch.empty(1, 2, 0, dtype=torch.float32, device=dev)
    dq, dk, dv = A.bwd_cross(z, k, v, z, lz, dz, True)
    assert dq.numel() == 0 and bool((dk == 0).all()) and bool((dv == 0).all())
    kz = k[:, :, :0].contiguous()
    lse = torch.full((1, 2, 10), float("-inf"), device=dev)
    o = torch.zeros_like(q)
    dq, dk, dv = A.bwd_cross(q, kz, kz, o, lse, dout, True)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    assert bool((dq == 0).all()) and dk.numel() == 0 and dv.numel() == 0


@pytest.mark.parametrize("causal", [False, True])
def test_cross_bwd_gqa_more_queries(dev, causal):
    """GQA with more queries than keys.  Under the causal mask most rows see only a few keys, so
    P is large and dS = P (dP - D) is sensitive to D_i = dO_i . O_i, which the backward forms
    from the stored bf16 O (off by up to 2^-8 |O| per element) as every caller's O is.  dV does
    not involve D and keeps the plain tolerance; dQ and dK get the tolerance plus the bound that
    rounding carries through exactly:
      |dD_i| <= sum_c |dO_ic| (2^-8 |O_ic| + e_O),  |d dQ_i| <= scale |dD_i| sum_j P_ij |K_j|,
      |d dK_j| <= scale sum_i P_ij |dD_i| |Q_i|  (e_O: the stored O's measured error)."""
    B, Hq, Hkv, Nq, Nk, d = 2, 8, 2, 333, 150, 128
    q, k, v, dout = inputs(B, Hq, Hkv, Nq, Nk, d, "bf16", seed=65)
    qd, kd, vd, dd = q.to(dev), k.to(dev), v.to(dev), dout.to(dev)
    o, lse = A.fwd_kvcache(qd, kd, vd, None, causal)
    g32 = A.bwd_cross(qd, kd, vd, o, lse, dd, causal, out_f32=True)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    qn, kn, vn, dn = (to_np(t) for t in (q, k, v, dout))
    refs = oracle.bwd_cross(qn, kn, vn, dn, causal)
    o_ref, lse_ref = oracle.fwd_kvcache(qn, kn, vn, None, causal)
    e_o = float(np.abs(to_np(o) - o_ref).max())
    dD = (np.abs(dn) * (2.0 ** -8 * np.abs(o_ref) + e_o)).sum(-1)  # [B,Hq,Nq]
    sc = 1 / np.sqrt(d)
    G = Hq // Hkv
    kx = np.repeat(kn, G, axis=1)  # the kv head of each query head
    S = sc * np.einsum("bhid,bhjd->bhij", qn, kx)
    if causal:
        S = np.where(np.arange(Nk)[None, :] > np.arange(Nq)[:, None] + (Nk - Nq), -np.inf, S)
    with np.errstate(invalid="ignore"):
        P = np.where(np.isfinite(lse_ref)[..., None], np.exp(S - lse_ref[..., None]), 0.0)
    bound_dq = TOL[torch.bfloat16] + sc * dD[..., None] * (P @ np.abs(kx))
    bound_dk_h = sc * np.einsum("bhij,bhi,bhid->bhjd", P, dD, np.abs(qn))
    bound_dk = TOL[torch.bfloat16] + bound_dk_h.reshape(B, Hkv, G, Nk, d).sum(2)
    dq32, dk32, dv32 = (to_np(t) for t in g32)
    assert_close_f32(dv32, refs[2], torch.bfloat16, f"cross bwd GQA Nq>Nk causal={causal} dV")
    for name, g, r, bnd in (("dQ", dq32, refs[0], bound_dq), ("dK", dk32, refs[1], bound_dk)):
        excess = float((np.abs(g - r) - bnd).max())
        assert excess <= 0, f"cross bwd GQA Nq>Nk causal={causal} {name}: exceeds the derived bound by {excess:.3e}"
    if causal:  # rows 0 .. Nq - Nk - 1 see no key
        assert bool((g32[0][:, :, :Nq - Nk] == 0).all())
