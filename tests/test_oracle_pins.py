"""Pins for the CPU oracle: facts fixed by the mathematics or printed on the pages, none of
which re-types the oracle's own formula.  Each is chosen so a plausible mistake in the
oracle (a dropped term, a wrong sign, index or mask, a transposed operand) fails at least one;
test_oracle_mutants.py checks that claim by planting such mistakes in copies of the source.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- closed forms / special cases

@pytest.mark.parametrize("causal", [False, True])
def test_uniform_keys_give_mean_of_values(causal, lib=None):
    """All keys equal -> every score in a row is the same -> P uniform over the visible keys,
    so O_i is the plain mean of V over j (or over j <= i when causal)."""
    rng = np.random.default_rng(1)
    B, H, N, d = 2, 3, 19, 16
    q = rand(rng, B, H, N, d)
    k = np.broadcast_to(rand(rng, B, H, 1, d), (B, H, N, d)).copy()
    v = rand(rng, B, H, N, d)
    o, _ = oracle.fwd(q, k, v, causal, lib=lib)
    if causal:
        expect = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    else:
        expect = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
    np.testing.assert_allclose(o, expect, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_log_count(causal, lib=None):
    """Q = 0 -> all scores 0 -> LSE_i = ln(number of visible keys), O_i = mean of visible V."""
    rng = np.random.default_rng(2)
    B, Hq, Hkv, N, d = 1, 4, 2, 23, 32
    q = np.zeros((B, Hq, N, d))
    k, v = rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    o, lse = oracle.fwd(q, k, v, causal, lib=lib)
    counts = np.arange(1, N + 1) if causal else np.full(N, N)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(counts), lse.shape), rtol=0, atol=1e-13)
    vr = np.repeat(v, Hq // Hkv, axis=1)
    expect = (np.cumsum(vr, axis=2) / counts[None, None, :, None]) if causal else \
        np.broadcast_to(vr.mean(axis=2, keepdims=True), vr.shape)
    np.testing.assert_allclose(o, expect, rtol=0, atol=1e-13)


def test_causal_first_row_is_first_value(lib=None):
    """Causal row 0 sees only key 0: O_0 = V_0 exactly and LSE_0 = S_00 = sc * Q_0 . K_0."""
    rng = np.random.default_rng(3)
    B, Hq, Hkv, N, d = 2, 4, 2, 9, 16
    q, k, v = rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    sc = 0.37
    o, lse = oracle.fwd(q, k, v, True, scale=sc, lib=lib)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(o[b, h, 0], v[b, h // G, 0])
            assert lse[b, h, 0] == pytest.approx(sc * float(q[b, h, 0] @ k[b, h // G, 0]), abs=1e-14)


def test_default_scale_is_inverse_sqrt_head_dim(lib=None):
    rng = np.random.default_rng(4)
    q, k, v = rand(rng, 1, 2, 11, 48), rand(rng, 1, 2, 11, 48), rand(rng, 1, 2, 11, 48)
    o1, l1 = oracle.fwd(q, k, v, False, scale=None, lib=lib)
    o2, l2 = oracle.fwd(q, k, v, False, scale=1 / math.sqrt(48), lib=lib)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-15)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal, lib=None):
    rng = np.random.default_rng(5)
    q, k = rand(rng, 1, 2, 31, 16) * 3, rand(rng, 1, 1, 31, 16) * 3
    for h in range(2):
        P = oracle.probs(q, k, 0, h, causal, lib=lib)
        assert np.all(P >= 0)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        if causal:
            assert np.all(np.triu(P, 1) == 0.0)
            assert np.all(np.diag(P) > 0)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_repeated_kv_heads(causal, lib=None):
    """Hq/Hkv query heads per kv head, contiguous groups: identical, bit for bit, to running
    with every kv head repeated G times (repeat_interleave)."""
    rng = np.random.default_rng(6)
    B, Hq, Hkv, N, d = 2, 6, 2, 13, 16
    q, k, v = rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    dout = rand(rng, B, Hq, N, d)
    G = Hq // Hkv
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    o1, l1 = oracle.fwd(q, k, v, causal, lib=lib)
    o2, l2 = oracle.fwd(q, kr, vr, causal, lib=lib)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    dq1, dk1, dv1 = oracle.bwd(q, k, v, dout, causal, lib=lib)
    dq2, dk2, dv2 = oracle.bwd(q, kr, vr, dout, causal, lib=lib)
    assert np.array_equal(dq1, dq2)
    # the grouped dK/dV is the sum over the group of the repeated-head gradients
    np.testing.assert_allclose(dk1, dk2.reshape(B, Hkv, G, N, d).sum(2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv1, dv2.reshape(B, Hkv, G, N, d).sum(2), rtol=0, atol=1e-13)


def test_permuting_keys_and_values_leaves_output(lib=None):
    rng = np.random.default_rng(7)
    q, k, v = rand(rng, 1, 2, 17, 16), rand(rng, 1, 2, 17, 16), rand(rng, 1, 2, 17, 16)
    perm = rng.permutation(17)
    o1, l1 = oracle.fwd(q, k, v, False, lib=lib)
    o2, l2 = oracle.fwd(q, k[:, :, perm], v[:, :, perm], False, lib=lib)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-14)


def test_output_is_linear_in_values(lib=None):
    rng = np.random.default_rng(8)
    q, k = rand(rng, 1, 2, 15, 16), rand(rng, 1, 2, 15, 16)
    v1, v2 = rand(rng, 1, 2, 15, 16), rand(rng, 1, 2, 15, 16)
    o1, _ = oracle.fwd(q, k, v1, True, lib=lib)
    o2, _ = oracle.fwd(q, k, v2, True, lib=lib)
    o3, _ = oracle.fwd(q, k, 2.0 * v1 - 3.0 * v2, True, lib=lib)
    np.testing.assert_allclose(o3, 2.0 * o1 - 3.0 * o2, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal, lib=None):
    """Adding one vector c to every key row adds sc*Q_i.c to every score of row i: P, O, dQ,
    dK and dV are unchanged (sum_j dS_ij = 0 removes the c term from dQ)."""
    rng = np.random.default_rng(9)
    B, Hq, Hkv, N, d = 1, 4, 2, 14, 16
    q, k, v = rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    dout = rand(rng, B, Hq, N, d)
    c = rand(rng, 1, 1, 1, d)
    o1, _ = oracle.fwd(q, k, v, causal, lib=lib)
    o2, _ = oracle.fwd(q, k + c, v, causal, lib=lib)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    g1 = oracle.bwd(q, k, v, dout, causal, lib=lib)
    g2 = oracle.bwd(q, k + c, v, dout, causal, lib=lib)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_dk_rows_sum_to_zero_and_dv_sums_to_dout(causal, lib=None):
    """sum_j dS_ij = 0 for every row (D_i = sum_j P_ij dP_ij) gives sum_j dK_j = 0 per group;
    sum_j P_ij = 1 gives sum_j dV_j = sum over the group's heads and rows of dO."""
    rng = np.random.default_rng(10)
    B, Hq, Hkv, N, d = 2, 4, 2, 21, 16
    q, k, v = rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    dout = rand(rng, B, Hq, N, d)
    _, dk, dv = oracle.bwd(q, k, v, dout, causal, lib=lib)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    expect = dout.reshape(B, Hkv, Hq // Hkv, N, d).sum(axis=(2, 3))
    np.testing.assert_allclose(dv.sum(axis=2), expect, rtol=0, atol=1e-11)


# ---------------------------------------------------------------- library special case

def _torch_reference(q, k, v, dout, causal, sc):
    t = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v)]
    o = F.scaled_dot_product_attention(t[0], t[1], t[2], is_causal=causal, scale=sc,
                                       enable_gqa=True)
    o.backward(torch.tensor(dout))
    return o.detach().numpy(), [x.grad.numpy() for x in t]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 2, 1, 16), (2, 4, 2, 33, 32), (1, 8, 1, 20, 64)])
def test_matches_torch_sdpa_fp64(shape, causal, lib=None):
    """torch's CPU float64 scaled_dot_product_attention (math backend) with autograd."""
    B, Hq, Hkv, N, d = shape
    rng = np.random.default_rng(11 + N)
    q, k, v = rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    dout = rand(rng, B, Hq, N, d)
    sc = 0.21
    o_ref, (dq_ref, dk_ref, dv_ref) = _torch_reference(q, k, v, dout, causal, sc)
    o, lse = oracle.fwd(q, k, v, causal, scale=sc, lib=lib)
    dq, dk, dv = oracle.bwd(q, k, v, dout, causal, scale=sc, lib=lib)
    for a, b in ((o, o_ref), (dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    # LSE against torch.logsumexp of the masked scaled scores
    G = Hq // Hkv
    s = sc * torch.einsum("bhid,bhjd->bhij", torch.tensor(q), torch.tensor(np.repeat(k, G, axis=1)))
    if causal:
        s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 3, 17])
def test_gradients_match_central_differences(N, causal, lib=None):
    """dQ, dK, dV against central differences (h = 1e-6) of L = sum(O * dO)."""
    rng = np.random.default_rng(12 + N)
    B, Hq, Hkv, d = 1, 2, 1, 16
    q, k, v = rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    dout = rand(rng, B, Hq, N, d)
    grads = oracle.bwd(q, k, v, dout, causal, lib=lib)
    h = 1e-6

    def loss(qq, kk, vv):
        o, _ = oracle.fwd(qq, kk, vv, causal, lib=lib)
        return float((o * dout).sum())

    for which, (x, g) in enumerate(zip((q, k, v), grads)):
        fd = np.empty_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-300)
        assert err <= 1e-7, (which, err)


def test_delta_equals_dout_dot_output(lib=None):
    """D_i = sum_j P_ij dP_ij equals dO_i . O_i; checked through dQ of a one-key-shifted run:
    with a single visible key (causal row 0) P = 1, dS = 0 and dQ_0 = 0 exactly."""
    rng = np.random.default_rng(13)
    q, k, v = rand(rng, 1, 2, 6, 16), rand(rng, 1, 1, 6, 16), rand(rng, 1, 1, 6, 16)
    dout = rand(rng, 1, 2, 6, 16)
    dq, _, _ = oracle.bwd(q, k, v, dout, True, lib=lib)
    assert np.all(np.abs(dq[:, :, 0]) <= 1e-15)


# ---------------------------------------------------------------- varlen

def test_varlen_page_example_cu_seqlens(lib=None):
    """cu_seqlens [0, 5, 12]: two sequences, rows 0..4 and 5..11; each is its own problem."""
    ex = json.load(open(os.path.join(GOLDEN, "varlen_cu_seqlens_example.json")))
    cu = ex["cu_seqlens"]
    assert len(cu) - 1 == ex["batch_size"] and cu[-1] == ex["total_tokens"]
    rng = np.random.default_rng(14)
    H, d = 2, 16
    qkv = rand(rng, ex["total_tokens"], 3, H, d)
    for causal in (False, True):
        out, lse = oracle.fwd_varlen(qkv, cu, causal, lib=lib)
        for s, (a, b) in enumerate(ex["sequences"]):
            # perturbing every other sequence leaves this one's rows unchanged, bit for bit
            other = qkv.copy()
            mask = np.ones(ex["total_tokens"], bool)
            mask[a:b] = False
            other[mask] = rand(rng, int(mask.sum()), 3, H, d)
            out2, lse2 = oracle.fwd_varlen(other, cu, causal, lib=lib)
            assert np.array_equal(out[a:b], out2[a:b]) and np.array_equal(lse[:, a:b], lse2[:, a:b])


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_per_sequence_dense_runs(causal, lib=None):
    rng = np.random.default_rng(15)
    lengths = [7, 1, 20, 13]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    H, d = 3, 16
    qkv = rand(rng, int(cu[-1]), 3, H, d)
    out, lse = oracle.fwd_varlen(qkv, cu, causal, scale=0.3, lib=lib)
    for s in range(len(lengths)):
        a, b = cu[s], cu[s + 1]
        seq = qkv[a:b]  # [L,3,H,d] -> [1,H,L,d]
        q = seq[:, 0].transpose(1, 0, 2)[None]
        k = seq[:, 1].transpose(1, 0, 2)[None]
        v = seq[:, 2].transpose(1, 0, 2)[None]
        o, l = oracle.fwd(q, k, v, causal, scale=0.3, lib=lib)
        assert np.array_equal(out[a:b], o[0].transpose(1, 0, 2))
        assert np.array_equal(lse[:, a:b], l[0])


def test_varlen_rejects_bad_cu_seqlens(lib=None):
    qkv = np.zeros((5, 3, 1, 16))
    for cu in ([0, 3, 2, 5], [1, 5], [0, 4]):
        with pytest.raises(ValueError):
            oracle.fwd_varlen(qkv, cu, False, lib=lib)


# ---------------------------------------------------------------- sampled entry points

@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_and_keys_match_full(causal, lib=None):
    rng = np.random.default_rng(16)
    B, Hq, Hkv, N, d = 2, 4, 2, 29, 16
    q, k, v = rand(rng, B, Hq, N, d), rand(rng, B, Hkv, N, d), rand(rng, B, Hkv, N, d)
    dout = rand(rng, B, Hq, N, d)
    o, lse = oracle.fwd(q, k, v, causal, lib=lib)
    dq, dk, dv = oracle.bwd(q, k, v, dout, causal, lib=lib)
    rows = np.array([[0, 0, 0], [1, 3, 28], [0, 2, 13], [1, 1, 5]])
    keys = np.array([[0, 0, 0], [1, 1, 28], [0, 1, 17]])
    o_s, l_s = oracle.fwd_rows(q, k, v, rows, causal, lib=lib)
    dq_s, dk_s, dv_s = oracle.bwd_sampled(q, k, v, dout, rows, keys, causal, lib=lib)
    for t, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(o_s[t], o[b, h, i], rtol=0, atol=1e-14)
        np.testing.assert_allclose(l_s[t], lse[b, h, i], rtol=0, atol=1e-14)
        np.testing.assert_allclose(dq_s[t], dq[b, h, i], rtol=0, atol=1e-13)
    for t, (b, g, j) in enumerate(keys):
        np.testing.assert_allclose(dk_s[t], dk[b, g, j], rtol=0, atol=1e-13)
        np.testing.assert_allclose(dv_s[t], dv[b, g, j], rtol=0, atol=1e-13)


def test_flop_count_matches_page_example():
    """The page's worked count for one Q.K^T of one head at N=2048, d=64."""
    from exact_attention_50_gb300 import workloads
    ex = json.load(open(os.path.join(GOLDEN, "flop_count_example.json")))
    # the forward counts two such contractions per head: half of it is one contraction
    assert workloads.fwd_flops(1, 1, ex["N"], ex["d"], False) / 2 == ex["one_gemm_one_head_flops"]


# ---------------------------------------------------------------- KV cache / cross-attention

def _lower_right_counts(Nq, L, causal):
    """Visible keys per query row, from torch's own bottom-right causal mask (a library
    definition of the alignment, not the oracle's rule retyped)."""
    if L == 0:
        return np.zeros(Nq, dtype=np.int64)
    if not causal:
        return np.full(Nq, L, dtype=np.int64)
    import warnings
    from torch.nn.attention.bias import causal_lower_right
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        mask = causal_lower_right(Nq, L)._materialize(device="cpu")
    return mask.sum(dim=-1).numpy().astype(np.int64)


def _kv_inputs(seed, B=3, Hq=4, Hkv=2, Nq=5, Nk=11, d=16):
    rng = np.random.default_rng(seed)
    return rng, rand(rng, B, Hq, Nq, d), rand(rng, B, Hkv, Nk, d), rand(rng, B, Hkv, Nk, d)


@pytest.mark.parametrize("causal", [False, True])
def test_kvcache_zero_queries_give_log_count(causal, lib=None):
    """Q = 0 -> every visible score is 0 -> LSE_i = ln(visible keys) (-inf when none) and O_i
    is the mean of the visible V rows (0 when none).  Lengths 11, 4 (< Nq: under the causal
    mask the first row sees nothing) and 0 (an empty cache)."""
    rng, q, k, v = _kv_inputs(31)
    q[:] = 0.0
    lens = [11, 4, 0]
    B, Hq, Nq, d = q.shape
    G = Hq // k.shape[1]
    o, lse = oracle.fwd_kvcache(q, k, v, lens, causal, lib=lib)
    for b, L in enumerate(lens):
        cnt = _lower_right_counts(Nq, L, causal)
        for h in range(Hq):
            for i in range(Nq):
                c = int(cnt[i])
                if c == 0:
                    assert lse[b, h, i] == -np.inf
                    np.testing.assert_array_equal(o[b, h, i], 0.0)
                else:
                    np.testing.assert_allclose(lse[b, h, i], math.log(c), rtol=0, atol=1e-13)
                    np.testing.assert_allclose(o[b, h, i], v[b, h // G, :c].mean(axis=0), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_kvcache_matches_torch_lower_right_sdpa(causal, lib=None):
    """torch's float64 SDPA per batch on the cache cut to its length, with the library's
    bottom-right causal mask and GQA; rows that see no key are checked by the pin above."""
    _, q, k, v = _kv_inputs(32, B=3, Hq=6, Hkv=3, Nq=7, Nk=20, d=16)
    lens = [20, 9, 3]
    sc = 0.3
    o, lse = oracle.fwd_kvcache(q, k, v, lens, causal, scale=sc, lib=lib)
    from torch.nn.attention.bias import causal_lower_right
    import warnings
    for b, L in enumerate(lens):
        tq = torch.tensor(q[b:b + 1])
        tk, tv = torch.tensor(k[b:b + 1, :, :L]), torch.tensor(v[b:b + 1, :, :L])
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            mask = causal_lower_right(q.shape[2], L) if causal else None
            ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=sc, enable_gqa=True).numpy()
        cnt = _lower_right_counts(q.shape[2], L, causal)
        seen = cnt > 0
        np.testing.assert_allclose(o[b][:, seen], ref[0][:, seen], rtol=0, atol=1e-12)
        # LSE: torch.logsumexp of the scores of the visible keys
        s = sc * torch.einsum("hid,hjd->hij", torch.tensor(q[b]), torch.tensor(np.repeat(k[b, :, :L], q.shape[1] // k.shape[1], axis=0)))
        if causal:
            with warnings.catch_warnings():
                warnings.simplefilter("ignore")
                vis = causal_lower_right(q.shape[2], L)._materialize(device="cpu")
            s = s.masked_fill(~vis, float("-inf"))
        np.testing.assert_allclose(lse[b][:, seen], torch.logsumexp(s, dim=-1).numpy()[:, seen], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_kvcache_full_square_cache_is_self_attention(causal, lib=None):
    """Nq == Nk with every cache full: the dense (self-attention) oracle, mask included."""
    _, q, k, v = _kv_inputs(33, B=2, Hq=4, Hkv=2, Nq=9, Nk=9, d=16)
    o, lse = oracle.fwd_kvcache(q, k, v, None, causal, lib=lib)
    o2, lse2 = oracle.fwd(q, k, v, causal, lib=lib)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-14)


def test_kvcache_ignores_cache_rows_past_length(lib=None):
    """Cache rows at or past cache_seqlens[b] do not enter the result."""
    rng, q, k, v = _kv_inputs(34)
    lens = [6, 11, 1]
    o, lse = oracle.fwd_kvcache(q, k, v, lens, True, lib=lib)
    k2, v2 = k.copy(), v.copy()
    for b, L in enumerate(lens):
        k2[b, :, L:] = rand(rng, *k2[b, :, L:].shape) * 50
        v2[b, :, L:] = rand(rng, *v2[b, :, L:].shape) * 50
    o2, lse2 = oracle.fwd_kvcache(q, k2, v2, lens, True, lib=lib)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_kvcache_rejects_bad_lengths(lib=None):
    _, q, k, v = _kv_inputs(35)
    for lens in ([12, 1, 1], [-1, 2, 2]):
        with pytest.raises(ValueError):
            oracle.fwd_kvcache(q, k, v, lens, False, lib=lib)


# ---------------------------------------------------------------- cross-attention backward

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(3, 5), (5, 3)])
def test_cross_bwd_matches_central_differences(Nq, Nk, causal, lib=None):
    """dQ, dK, dV against central differences (h = 1e-6) of L = sum(O * dO), O from the
    KV-cache forward with full caches; with Nq > Nk under the causal mask the first rows see
    no key (O = 0 there, no gradient)."""
    rng = np.random.default_rng(40 + Nq)
    B, Hq, Hkv, d = 1, 2, 1, 8
    q, k, v = rand(rng, B, Hq, Nq, d), rand(rng, B, Hkv, Nk, d), rand(rng, B, Hkv, Nk, d)
    dout = rand(rng, B, Hq, Nq, d)
    grads = oracle.bwd_cross(q, k, v, dout, causal, lib=lib)
    h = 1e-6

    def loss(qq, kk, vv):
        o, _ = oracle.fwd_kvcache(qq, kk, vv, None, causal, lib=lib)
        return float((o * dout).sum())

    for which, (x, g) in enumerate(zip((q, k, v), grads)):
        fd = np.empty_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p, args_m = [q, k, v], [q, k, v]
            args_p[which], args_m[which] = xp, xm
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-300)
        assert err <= 1e-7, (which, err)


@pytest.mark.parametrize("causal", [False, True])
def test_cross_bwd_matches_torch_lower_right_sdpa(causal, lib=None):
    """torch's float64 SDPA with its bottom-right causal mask and autograd, GQA, Nq < Nk."""
    rng = np.random.default_rng(45)
    B, Hq, Hkv, Nq, Nk, d = 2, 4, 2, 6, 19, 16
    q, k, v = rand(rng, B, Hq, Nq, d), rand(rng, B, Hkv, Nk, d), rand(rng, B, Hkv, Nk, d)
    dout = rand(rng, B, Hq, Nq, d)
    sc = 0.27
    import warnings
    from torch.nn.attention.bias import causal_lower_right
    t = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v)]
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")
        mask = causal_lower_right(Nq, Nk)._materialize(device="cpu") if causal else None
    o = F.scaled_dot_product_attention(t[0], t[1], t[2], attn_mask=mask, scale=sc, enable_gqa=True)
    o.backward(torch.tensor(dout))
    got = oracle.bwd_cross(q, k, v, dout, causal, scale=sc, lib=lib)
    for g, x in zip(got, t):
        np.testing.assert_allclose(g, x.grad.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_cross_bwd_square_is_dense_backward(causal, lib=None):
    rng = np.random.default_rng(46)
    q, k, v, dout = rand(rng, 1, 4, 11, 16), rand(rng, 1, 2, 11, 16), rand(rng, 1, 2, 11, 16), rand(rng, 1, 4, 11, 16)
    for a, b in zip(oracle.bwd_cross(q, k, v, dout, causal, lib=lib), oracle.bwd(q, k, v, dout, causal, lib=lib)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
