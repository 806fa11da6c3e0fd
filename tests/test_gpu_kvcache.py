"""GPU parity of the KV-cache / cross-attention forward (attn_fwd_kvcache) through the C ABI:
against the fp64 oracle on ragged caches (empty caches, caches shorter than the query block
under the causal mask, partial key tiles), several row blocks per (batch, kv head), 1 / several
/ automatic key ranges; bitwise equality with the dense forward when the cache is the whole
square problem; invariance to the split count; device-side rejection of bad cache lengths."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_50_gb300 import _lib, build
from exact_attention_50_gb300 import attention as A
from exact_attention_50_gb300 import workloads as W
from tests.parity import assert_close_f32, assert_close_native, to_np

pytestmark = pytest.mark.gpu

LSE_TOL = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 2e-3}


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    _lib.load()
    return torch.device("cuda:0")


def run_case(dev, B, Hq, Hkv, Nq, Nk, d, dtype, lens, causal, splits, seed):
    q, k, v, cl = W.kvcache_inputs(B, Hq, Hkv, Nq, Nk, d, dtype, lens, seed=seed)
    tdt = W.DTYPES[dtype]
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    cld = cl.to(dev) if cl is not None else None
    o32, lse = A.fwd_kvcache(qd, kd, vd, cld, causal, num_splits=splits, out_f32=True)
    o, lse2 = A.fwd_kvcache(qd, kd, vd, cld, causal, num_splits=splits)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    o_ref, lse_ref = oracle.fwd_kvcache(to_np(q), to_np(k), to_np(v), None if cl is None else cl.numpy(), causal)
    what = f"kvcache {dtype} B{B} Hq{Hq} Hkv{Hkv} Nq{Nq} Nk{Nk} d{d} causal={causal} splits={splits}"
    assert_close_f32(o32, o_ref, tdt, what + " O (fp32)")
    assert_close_native(o, o_ref, tdt, what + " O")
    l, lr = to_np(lse), lse_ref
    empty = np.isneginf(lr)
    assert np.array_equal(np.isneginf(l), empty), what + ": rows without keys differ"
    assert np.abs(l[~empty] - lr[~empty]).max(initial=0.0) <= LSE_TOL[tdt], what + " LSE"
    assert torch.equal(lse, lse2)
    return o32, lse


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 64), ("bf16", 80)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_matches_oracle(dev, dtype, d, causal, splits):
    # Nq = 5 against caches of 700 (5.5 key tiles), 333, 3 (< Nq: under the causal mask the
    # first rows see nothing) and 0 keys
    run_case(dev, 4, 8, 2, 5, 700, d, dtype, [700, 333, 3, 0], causal, splits, seed=41)


@pytest.mark.parametrize("causal", [False, True])
def test_row_blocks_straddling_heads(dev, causal):
    """G * Nq = 400 rows per kv head: four 128-row blocks, three of them spanning two heads."""
    run_case(dev, 2, 4, 1, 100, 900, 128, "bf16", [900, 517], causal, 0, seed=42)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
def test_cross_attention_full_caches(dev, dtype, causal):
    """No cache lengths: every batch attends all Nk keys (cross-attention Nq != Nk)."""
    run_case(dev, 2, 6, 3, 300, 520, 64, dtype, None, causal, 0, seed=43)


@pytest.mark.parametrize("causal", [False, True])
def test_square_cache_equals_dense_forward_bitwise(dev, causal):
    """Nq = Nk = L, one key range: the rows, key tiles and arithmetic are those of attn_fwd."""
    q, k, v, _ = W.dense_inputs(2, 4, 2, 256, 128, "bf16", seed=44, with_dout=False)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = A.fwd(qd, kd, vd, causal)
    o2, l2 = A.fwd_kvcache(qd, kd, vd, None, causal, num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert A.get_device_status() == _lib.ATTN_OK


def test_split_count_changes_only_rounding(dev):
    """Each range rounds its P to bf16 against its own running max, so O moves by P's rounding
    (2^-9 relative per weight, twice: bound 2^-8 at |V| <= 1 scale) while the LSE, summed
    from the unrounded fp32 weights, moves only by fp32 summation order."""
    q, k, v, cl = W.kvcache_inputs(3, 16, 4, 2, 4000, 128, "bf16", [4000, 2500, 129], seed=45)
    qd, kd, vd, cld = q.to(dev), k.to(dev), v.to(dev), cl.to(dev)
    ref, lref = A.fwd_kvcache(qd, kd, vd, cld, True, num_splits=1, out_f32=True)
    for s in (2, 7, 32, 0):
        o, l = A.fwd_kvcache(qd, kd, vd, cld, True, num_splits=s, out_f32=True)
        assert (o - ref).abs().max().item() <= 2.0 ** -8, s
        assert (l - lref).abs().max().item() <= 1e-5, s
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK


def test_empty_cache_and_empty_queries(dev):
    q, k, v, _ = W.kvcache_inputs(2, 4, 2, 3, 0, 64, "bf16", None, seed=46)
    o, lse = A.fwd_kvcache(q.to(dev), k.to(dev), v.to(dev), None, False)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0 and bool(torch.isneginf(lse).all())
    q0 = torch.zeros(2, 4, 0, 64, dtype=torch.bfloat16, device=dev)
    o0, l0 = A.fwd_kvcache(q0, k.to(dev), v.to(dev), None, False)
    assert o0.shape == (2, 4, 0, 64) and l0.shape == (2, 4, 0)
    assert A.get_device_status() == _lib.ATTN_OK


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bad_cache_length_reported_by_device(dev, dtype):
    q, k, v, _ = W.kvcache_inputs(2, 4, 2, 1, 300, 64, dtype, None, seed=47)
    bad = torch.tensor([100, 301], dtype=torch.int32, device=dev)  # longer than the cache
    o, lse = A.fwd_kvcache(q.to(dev), k.to(dev), v.to(dev), bad, False)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_ERR_DEVICE_INPUT
    assert A.get_device_status() == _lib.ATTN_OK  # reading clears it
    assert bool(torch.isneginf(lse[1]).all())      # that batch is treated as empty


def test_decode_workload_sampled(dev):
    """The benchmark's decode workload at full size (B=8, Hq=32, Hkv=8, one query, caches of
    U[16384, 32768] keys, d=128 bf16) in its launch configuration (automatic split count):
    batches 0 and 5 against the oracle, every batch finite."""
    wl = W.WORKLOADS["decode_bf16"]
    q, k, v, cl = W.kvcache_inputs(wl.B, wl.Hq, wl.Hkv, wl.extra["Nq"], wl.N, wl.d, wl.dtype, wl.extra["lens"], seed=0)
    qd, kd, vd, cld = q.to(dev), k.to(dev), v.to(dev), cl.to(dev)
    o32, lse = A.fwd_kvcache(qd, kd, vd, cld, wl.causal, out_f32=True)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    assert bool(torch.isfinite(o32).all()) and bool(torch.isfinite(lse).all())
    for b in (0, 5):
        o_ref, l_ref = oracle.fwd_kvcache(to_np(q[b:b + 1]), to_np(k[b:b + 1]), to_np(v[b:b + 1]),
                                          cl[b:b + 1].numpy(), wl.causal)
        assert_close_f32(o32[b:b + 1], o_ref, torch.bfloat16, f"decode workload batch {b}")
        assert np.abs(to_np(lse[b:b + 1]) - l_ref).max() <= 2e-3
