"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle, element by element,
on seeded inputs.  Small ragged shapes span several tiles and a partial tail; the full-size
workloads are checked in the launch configuration the benchmark times: whole batches, whole kv
groups and every varlen sequence element by element, plus sampled rows and keys of the parts
the oracle would take minutes over."""
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


def status_ok():
    assert A.get_device_status() == _lib.ATTN_OK


def gpu_fwd_bwd(q, k, v, dout, causal, scale, dev, with_bwd=True):
    """Runs the forward (fp32-flagged and native outputs) and optionally the backward."""
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o32, lse = A.fwd(qd, kd, vd, causal, scale, out_f32=True)
    o, lse_n = A.fwd(qd, kd, vd, causal, scale)
    res = {"o32": o32, "o": o, "lse": lse, "lse_n": lse_n}
    if with_bwd:
        dd = dout.to(dev)
        res["g32"] = A.bwd(qd, kd, vd, o, lse, dd, causal, scale, out_f32=True)
        res["g"] = A.bwd(qd, kd, vd, o, lse, dd, causal, scale)
    torch.cuda.synchronize()
    status_ok()
    return res


def check_dense(res, q, k, v, dout, causal, scale, dtype, what, with_bwd=True):
    o_ref, lse_ref = oracle.fwd(to_np(q), to_np(k), to_np(v), causal, scale)
    assert_close_f32(res["o32"], o_ref, dtype, what + " O(fp32)")
    assert_close_native(res["o"], o_ref, dtype, what + " O(native)")
    assert torch.equal(res["lse"], res["lse_n"])
    assert_close_f32(res["lse"], lse_ref, dtype if dtype == torch.float32 else torch.float16, what + " LSE")
    if with_bwd:
        refs = oracle.bwd(to_np(q), to_np(k), to_np(v), to_np(dout), causal, scale)
        for name, g32, g, r in zip(("dQ", "dK", "dV"), res["g32"], res["g"], refs):
            assert_close_f32(g32, r, dtype, f"{what} {name}(fp32)")
            assert_close_native(g, r, dtype, f"{what} {name}(native)")


# ------------------------------------------------------------------ fp32 (CUDA cores)

def test_tiny_f32_forward_workload(dev):
    """B=1, H=2, N=128, d=64, non-causal, scale 1/8, seed 0: within 1e-5 of the oracle."""
    wl = W.WORKLOADS["tiny_f32"]
    q, k, v, dout = W.dense_inputs(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, "f32", seed=0)
    res = gpu_fwd_bwd(q, k, v, dout, wl.causal, wl.scale, dev)
    check_dense(res, q, k, v, dout, wl.causal, wl.scale, torch.float32, "tiny_f32")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 1, 1, 16), (2, 4, 2, 77, 64), (1, 2, 2, 130, 128), (1, 3, 1, 33, 48)])
def test_f32_ragged_shapes(dev, shape, causal):
    B, Hq, Hkv, N, d = shape
    q, k, v, dout = W.dense_inputs(B, Hq, Hkv, N, d, "f32", seed=N)
    res = gpu_fwd_bwd(q, k, v, dout, causal, None, dev)
    check_dense(res, q, k, v, dout, causal, None, torch.float32, f"f32 {shape} causal={causal}")


# ------------------------------------------------------------------ fp16 / bf16 (tcgen05)

TC_SHAPES = [(1, 1, 1, 1, 64), (1, 2, 1, 100, 64), (2, 4, 2, 129, 128), (1, 2, 2, 300, 32),
             (1, 4, 1, 257, 96), (1, 2, 1, 64, 16), (1, 2, 2, 513, 128), (1, 8, 1, 200, 112)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", TC_SHAPES)
def test_tensor_core_ragged_shapes(dev, shape, causal, dtype):
    B, Hq, Hkv, N, d = shape
    q, k, v, dout = W.dense_inputs(B, Hq, Hkv, N, d, dtype, seed=7 * N + d)
    res = gpu_fwd_bwd(q, k, v, dout, causal, None, dev)
    check_dense(res, q, k, v, dout, causal, None, W.DTYPES[dtype], f"{dtype} {shape} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_online_rescaling_under_growing_scores(dev, d, causal):
    """Scores that grow (or shrink) across key tiles by tens of log2 units force the running
    max to move, and the O rescale to run, in tile after tile."""
    B, H, N = 1, 4, 1024
    g = W.generator(11)
    q = torch.randn(B, H, N, d, generator=g) * 2.0
    k = torch.randn(B, H, N, d, generator=g) + (torch.arange(N) / N * 6.0)[None, None, :, None]
    v = torch.randn(B, H, N, d, generator=g)
    dout = torch.randn(B, H, N, d, generator=g)
    q, k, v, dout = (t.to(torch.bfloat16) for t in (q, k, v, dout))
    res = gpu_fwd_bwd(q, k, v, dout, causal, None, dev)
    what = f"rescale d={d} causal={causal}"
    check_dense(res, q, k, v, dout, causal, None, torch.bfloat16, what, with_bwd=False)
    # Backward.  D_i = dO_i . O_i is formed from the stored bf16 O, which is off by at most
    # 2^-8 |O_ic| (round to nearest) plus the forward's own error e_O, so
    #   |dD_i| <= sum_c |dO_ic| (2^-8 |O_ic| + e_O).
    # Through dS_ij = P_ij (dP_ij - D_i) that moves dQ_ic by at most scale dD_i sum_j P_ij |K_jc|
    # and dK_jc by at most scale sum_i P_ij dD_i |Q_ic| -- exact-arithmetic consequences that
    # these large-offset keys (|K| up to ~9) make larger than with N(0,1) inputs.  dV does not
    # involve D and keeps the plain tolerance; dQ and dK get tolerance + that bound.
    qn, kn, vn, dn = (to_np(t) for t in (q, k, v, dout))
    sc = 1 / np.sqrt(d)
    o_ref, _ = oracle.fwd(qn, kn, vn, causal)
    e_o = float(np.abs(to_np(res["o32"]) - o_ref).max())
    dD = (np.abs(dn) * (2.0 ** -8 * np.abs(o_ref) + e_o)).sum(-1)          # [B,H,N]
    P = np.stack([oracle.probs(qn, kn, 0, h, causal) for h in range(H)])[None]  # [1,H,N,N]
    bound_dq = TOL[torch.bfloat16] + sc * dD[..., None] * (P @ np.abs(kn))
    bound_dk = TOL[torch.bfloat16] + sc * (np.swapaxes(P, -1, -2) @ (dD[..., None] * np.abs(qn)))
    refs = oracle.bwd(qn, kn, vn, dn, causal)
    dq32, dk32, dv32 = (to_np(t) for t in res["g32"])
    assert_close_f32(dv32, refs[2], torch.bfloat16, what + " dV")
    for name, g, r, bnd in (("dQ", dq32, refs[0], bound_dq), ("dK", dk32, refs[1], bound_dk)):
        excess = float((np.abs(g - r) - bnd).max())
        assert excess <= 0, f"{what} {name}: exceeds the derived bound by {excess:.3e}"


def test_mha_f16_workload_full(dev):
    """B=1, H=32, N=2048, d=64 fp16 forward (the pages' A10 shape), non-causal and causal."""
    wl = W.WORKLOADS["mha_f16"]
    q, k, v, _ = W.dense_inputs(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, "f16", seed=0, with_dout=False)
    for causal in (False, True):
        res = gpu_fwd_bwd(q, k, v, None, causal, wl.scale, dev, with_bwd=False)
        check_dense(res, q, k, v, None, causal, wl.scale, torch.float16, f"mha_f16 causal={causal}", with_bwd=False)


def test_gqa_bf16_workload_full(dev):
    """B=4, Hq=32, Hkv=8, N=2048, d=128 bf16 causal fwd+bwd, launched at full size; batch 0 is
    compared element by element in full, batch 3 on sampled rows and keys."""
    wl = W.WORKLOADS["gqa_bf16"]
    q, k, v, dout = W.dense_inputs(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, "bf16", seed=0)
    res = gpu_fwd_bwd(q, k, v, dout, True, None, dev)
    sub = {key: (val[:1] if isinstance(val, torch.Tensor) else tuple(x[:1] for x in val))
           for key, val in res.items()}
    check_dense(sub, q[:1], k[:1], v[:1], dout[:1], True, None, torch.bfloat16, "gqa_bf16 batch0")
    rng = np.random.default_rng(0)
    rows = np.stack([np.full(48, 3), rng.integers(0, wl.Hq, 48), rng.integers(0, wl.N, 48)], 1)
    rows[:4, 2] = [0, 1, wl.N - 1, 1000]
    o_r, l_r = oracle.fwd_rows(to_np(q), to_np(k), to_np(v), rows, True)
    o_g = to_np(res["o32"])[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close_f32(o_g, o_r, torch.bfloat16, "gqa_bf16 batch3 O rows")
    keys = np.stack([np.full(8, 3), rng.integers(0, wl.Hkv, 8), rng.integers(0, wl.N, 8)], 1)
    keys[:3, 2] = [0, 127, wl.N - 1]
    dq_r, dk_r, dv_r = oracle.bwd_sampled(to_np(q), to_np(k), to_np(v), to_np(dout), rows[:16], keys, True)
    dq32, dk32, dv32 = (to_np(x) for x in res["g32"])
    assert_close_f32(dq32[rows[:16, 0], rows[:16, 1], rows[:16, 2]], dq_r, torch.bfloat16, "batch3 dQ rows")
    assert_close_f32(dk32[keys[:, 0], keys[:, 1], keys[:, 2]], dk_r, torch.bfloat16, "batch3 dK keys")
    assert_close_f32(dv32[keys[:, 0], keys[:, 1], keys[:, 2]], dv_r, torch.bfloat16, "batch3 dV keys")


def test_long_context_bf16_workload_full_group(dev):
    """B=1, Hq=32, Hkv=8, N=32768, d=128 bf16 causal fwd+bwd, launched at full size.  KV group 0
    (its four query heads and its kv head) is compared with the oracle element by element in
    full: O and LSE of all 4 x 32768 rows, dQ of those rows, dK and dV of all 32768 keys, at the
    bf16 tolerance on the fp32 results and tol + half an ulp on the stored bf16 ones.  The other
    groups are checked on sampled rows (64 for the last group, 12 for the others, including the
    first and last rows) and on keys near the end of the sequence (8 for the last group, 2 for
    the others): a sampled key costs the oracle a row pass over every query that sees it, which
    for the early keys is the whole group, and those are covered in full by group 0."""
    wl = W.WORKLOADS["long_bf16"]
    q, k, v, dout = W.dense_inputs(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d, "bf16", seed=0)
    res = gpu_fwd_bwd(q, k, v, dout, True, None, dev)
    G = wl.Hq // wl.Hkv
    hs = slice(0, G)
    sub = {"o32": res["o32"][:, hs], "o": res["o"][:, hs], "lse": res["lse"][:, hs], "lse_n": res["lse_n"][:, hs],
           "g32": (res["g32"][0][:, hs], res["g32"][1][:, :1], res["g32"][2][:, :1]),
           "g": (res["g"][0][:, hs], res["g"][1][:, :1], res["g"][2][:, :1])}
    check_dense(sub, q[:, hs], k[:, :1], v[:, :1], dout[:, hs], True, None, torch.bfloat16, "long_bf16 group 0")
    rng = np.random.default_rng(5)
    for g in range(1, wl.Hkv):
        n_r, n_k = (64, 8) if g == wl.Hkv - 1 else (12, 2)
        hs = slice(g * G, (g + 1) * G)
        qs, ks, vs, ds = (to_np(t) for t in (q[:, hs], k[:, g:g + 1], v[:, g:g + 1], dout[:, hs]))
        rows = np.stack([np.zeros(n_r, int), rng.integers(0, G, n_r), rng.integers(0, wl.N, n_r)], 1)
        rows[:4, 2] = [0, 1, 127, wl.N - 1]
        # keys in the last 1024 of the sequence, including the last one and a tile boundary
        keys = np.stack([np.zeros(n_k, int), np.zeros(n_k, int), rng.integers(wl.N - 1024, wl.N, n_k)], 1)
        keys[:2, 2] = [wl.N - 1, wl.N - 129]
        o_r, l_r = oracle.fwd_rows(qs, ks, vs, rows, True)
        dq_r, dk_r, dv_r = oracle.bwd_sampled(qs, ks, vs, ds, rows, keys, True)
        o_g = to_np(res["o32"][:, hs])[rows[:, 0], rows[:, 1], rows[:, 2]]
        l_g = to_np(res["lse"][:, hs])[rows[:, 0], rows[:, 1], rows[:, 2]]
        dq_g = to_np(res["g32"][0][:, hs])[rows[:, 0], rows[:, 1], rows[:, 2]]
        dk_g = to_np(res["g32"][1][:, g:g + 1])[0, 0, keys[:, 2]]
        dv_g = to_np(res["g32"][2][:, g:g + 1])[0, 0, keys[:, 2]]
        assert_close_f32(o_g, o_r, torch.bfloat16, f"long O rows g={g}")
        assert_close_f32(l_g, l_r, torch.float16, f"long LSE rows g={g}")
        assert_close_f32(dq_g, dq_r, torch.bfloat16, f"long dQ rows g={g}")
        assert_close_f32(dk_g, dk_r, torch.bfloat16, f"long dK keys g={g}")
        assert_close_f32(dv_g, dv_r, torch.bfloat16, f"long dV keys g={g}")


# ------------------------------------------------------------------ varlen

def test_varlen_bf16_workload(dev):
    """16 sequences, lengths ~ U[64, 4096] (seed 0), qkv [T,3,16,128], causal: every sequence's
    rows are bit-identical to a dense forward of that sequence alone, and every sequence is
    compared with the oracle element by element."""
    wl = W.WORKLOADS["varlen_bf16"]
    qkv, cu, lengths, _ = W.varlen_inputs(wl.varlen, wl.Hq, wl.d, "bf16", seed=0)
    qkv_d, cu_d = qkv.to(dev), cu.to(dev)
    out32, lse = A.fwd_varlen(qkv_d, cu_d, max(lengths), True, out_f32=True)
    out, _ = A.fwd_varlen(qkv_d, cu_d, max(lengths), True)
    status_ok()
    cu_l = cu.tolist()
    for s in range(len(lengths)):
        a, b = cu_l[s], cu_l[s + 1]
        seq = qkv_d[a:b]
        qs, ks, vs = (seq[:, i].transpose(0, 1).unsqueeze(0).contiguous() for i in range(3))
        o32, l = A.fwd(qs, ks, vs, True, None, out_f32=True)
        o_n, _ = A.fwd(qs, ks, vs, True, None)
        assert torch.equal(out32[a:b], o32[0].transpose(0, 1)), f"sequence {s}: fp32 rows differ"
        assert torch.equal(out[a:b], o_n[0].transpose(0, 1)), f"sequence {s}: native rows differ"
        assert torch.equal(lse[:, a:b], l[0]), f"sequence {s}: LSE differs"
    status_ok()
    o_r, l_r = oracle.fwd_varlen(to_np(qkv), cu.numpy(), True)
    for s in range(len(lengths)):
        a, b = cu_l[s], cu_l[s + 1]
        assert_close_f32(out32[a:b], o_r[a:b], torch.bfloat16, f"varlen seq {s} O")
        assert_close_native(out[a:b], o_r[a:b], torch.bfloat16, f"varlen seq {s} O native")
        assert_close_f32(lse[:, a:b], l_r[:, a:b], torch.float16, f"varlen seq {s} LSE")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_varlen_small_with_empty_and_ragged(dev, dtype):
    lengths = [5, 0, 130, 1, 0, 257, 64]
    qkv, cu, lengths, _ = W.varlen_inputs(lengths, 3, 64, dtype, seed=3)
    for causal in (False, True):
        out32, lse = A.fwd_varlen(qkv.to(dev), cu.to(dev), max(lengths), causal, out_f32=True)
        status_ok()
        o_r, l_r = oracle.fwd_varlen(to_np(qkv), cu.numpy(), causal)
        assert_close_f32(out32, o_r, W.DTYPES[dtype], f"varlen small {dtype} causal={causal}")
        tol_lse = torch.float32 if dtype == "f32" else torch.float16
        assert_close_f32(lse, l_r, tol_lse, "varlen small LSE")


def test_varlen_guard_bands_untouched(dev):
    """Canary bytes before and after the output and LSE buffers survive a varlen call."""
    lengths = [100, 3, 260]
    qkv, cu, lengths, _ = W.varlen_inputs(lengths, 2, 128, "bf16", seed=4)
    T, H, d = qkv.shape[0], 2, 128
    pad = 4096
    canary = -12345.0
    obuf = torch.full((pad + T * H * d + pad,), canary, dtype=torch.bfloat16, device=dev)
    lbuf = torch.full((pad + H * T + pad,), canary, dtype=torch.float32, device=dev)
    out = obuf[pad:pad + T * H * d]
    lse = lbuf[pad:pad + H * T]
    qkv_d, cu_d = qkv.to(dev), cu.to(dev)
    st = _lib.attn_fwd_varlen(qkv_d.data_ptr(), cu_d.data_ptr(), len(lengths), T, max(lengths), out.data_ptr(),
                              lse.data_ptr(), H, d, 1, 0.0, _lib.ATTN_BF16, 0,
                              torch.cuda.current_stream().cuda_stream)
    assert st == _lib.ATTN_OK
    status_ok()
    assert bool((obuf[:pad] == canary).all()) and bool((obuf[pad + T * H * d:] == canary).all())
    assert bool((lbuf[:pad] == canary).all()) and bool((lbuf[pad + H * T:] == canary).all())
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all())


def test_varlen_invalid_cu_seqlens_reported_by_device(dev):
    qkv = torch.randn(20, 3, 2, 64, device=dev).to(torch.bfloat16)
    for cu in ([0, 10, 5, 20], [0, 10, 20, 20], [0, 19, 20]):
        cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
        maxlen = 12 if cu == [0, 19, 20] else 20
        A.fwd_varlen(qkv, cu_d, maxlen, False)
        st = A.get_device_status()
        if cu == [0, 10, 20, 20]:
            assert st == _lib.ATTN_OK  # a trailing empty sequence is valid
        else:
            assert st == _lib.ATTN_ERR_DEVICE_INPUT
    # the context is still usable afterwards
    out, _ = A.fwd_varlen(qkv, torch.tensor([0, 20], dtype=torch.int32, device=dev), 20, True)
    status_ok()
    assert bool(torch.isfinite(out).all())


# ------------------------------------------------------------------ API surface

def test_autograd_flash_attention_matches_explicit_calls(dev):
    q, k, v, dout = W.dense_inputs(2, 8, 2, 333, 64, "bf16", seed=21)
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    o = A.flash_attention(qd, kd, vd)  # causal=True by default
    o.backward(dout.to(dev))
    o2, lse = A.fwd(qd.detach(), kd.detach(), vd.detach(), True)
    g = A.bwd(qd.detach(), kd.detach(), vd.detach(), o2, lse, dout.to(dev), True)
    assert torch.equal(o, o2)
    for a, b in zip((qd.grad, kd.grad, vd.grad), g):
        assert torch.equal(a, b)
    status_ok()


def test_varlen_api_matches_page_example(dev):
    """cu_seqlens [0, 5, 12]: two sequences of 5 and 7 tokens (Turing varlen article)."""
    from exact_attention_50_gb300 import flash_attn_varlen_qkvpacked_func
    qkv, cu, lengths, _ = W.varlen_inputs([5, 7], 4, 64, "f16", seed=1)
    out = flash_attn_varlen_qkvpacked_func(qkv.to(dev), cu.to(dev), 7)
    status_ok()
    o_r, _ = oracle.fwd_varlen(to_np(qkv), [0, 5, 12], False)
    assert_close_native(out, o_r, torch.float16, "page example")


def test_empty_inputs_are_no_ops(dev):
    z = torch.empty(0, 2, 16, 64, device=dev, dtype=torch.bfloat16)
    o, lse = A.fwd(z, z, z, True)
    assert o.shape == z.shape
    z2 = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    o, lse = A.fwd(z2, z2, z2, False)
    g = A.bwd(z2, z2, z2, o, lse, z2, False)
    assert all(t.numel() == 0 for t in g)
    status_ok()
