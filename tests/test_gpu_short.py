"""The short-sequence forward (N <= 64): several (batch, kv head) problems packed into one
128-row tile with a block-diagonal mask, or, when a kv head's G * N query rows exceed 128, one
128-row block of them per work item.  Checked against the fp64 oracle element by element at
B * H in the thousands, N in {1, 17, 64}, with causal and non-causal masks, GQA and MHA, a packed
last tile that is only partly filled, and head dims below 64."""
import os

import numpy as np
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


def run_and_check(dev, B, Hq, Hkv, N, d, dtype, causal, seed):
    q, k, v, _ = W.dense_inputs(B, Hq, Hkv, N, d, dtype, seed=seed, with_dout=False)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o32, lse = A.fwd(qd, kd, vd, causal, None, out_f32=True)
    o, lse_n = A.fwd(qd, kd, vd, causal, None)
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    o_ref, lse_ref = oracle.fwd(to_np(q), to_np(k), to_np(v), causal)
    what = f"short {dtype} B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} causal={causal}"
    tdt = W.DTYPES[dtype]
    assert_close_f32(o32, o_ref, tdt, what + " O(fp32)")
    assert_close_native(o, o_ref, tdt, what + " O(native)")
    assert torch.equal(lse, lse_n)
    assert_close_f32(lse, lse_ref, torch.float16, what + " LSE")
    return o


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 64])
def test_short_mha_thousands_of_heads(dev, N, causal, dtype):
    # B * H = 2048 problems; N = 17 packs 7 per tile, leaving the last tile partly empty
    run_and_check(dev, 64, 32, 32, N, 128, dtype, causal, seed=N)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(128, 16, 4, 17, 64),    # G * N = 68: one unit per tile
                                   (64, 32, 8, 13, 64),     # G * N = 52: two units per tile
                                   (32, 32, 4, 64, 128),    # G * N = 256: two row blocks per unit
                                   (40, 16, 2, 17, 128),    # G * N = 136: a 128-row block and 8 rows
                                   (100, 8, 1, 64, 64)])    # MQA, G * N = 512
def test_short_gqa(dev, shape, causal):
    B, Hq, Hkv, N, d = shape
    run_and_check(dev, B, Hq, Hkv, N, d, "bf16", causal, seed=B + N)


@pytest.mark.parametrize("d", [16, 48, 80])
def test_short_head_dims_below_the_tile(dev, d):
    run_and_check(dev, 50, 12, 4, 33, d, "f16", True, seed=d)


def test_short_units_not_a_multiple_of_the_packing(dev):
    # N = 5: 25 units per tile; 1001 units leave a last tile with one unit
    run_and_check(dev, 7, 143, 143, 5, 64, "bf16", False, seed=5)


def test_short_kernel_agrees_with_the_general_kernel(dev):
    """Both kernels compute the same attention; the switch ATTN_SHORT_KERNEL=0 routes N <= 64
    to the general persistent kernel.  Their fp32 results agree to rounding."""
    q, k, v, _ = W.dense_inputs(32, 16, 4, 48, 128, "bf16", seed=9, with_dout=False)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    a, la = A.fwd(qd, kd, vd, True, None, out_f32=True)
    os.environ["ATTN_SHORT_KERNEL"] = "0"
    try:
        b, lb = A.fwd(qd, kd, vd, True, None, out_f32=True)
    finally:
        del os.environ["ATTN_SHORT_KERNEL"]
    torch.cuda.synchronize()
    assert A.get_device_status() == _lib.ATTN_OK
    assert float((a - b).abs().max()) < 1e-2
    assert float((la - lb).abs().max()) < 1e-4
