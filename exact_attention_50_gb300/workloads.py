"""Seeded synthetic inputs and the workload table.

This module only draws random numbers and describes shapes; it holds none of the attention
arithmetic, so both the CUDA path's tests/benchmark and the CPU oracle can take their inputs
from it without sharing any computation.

Drawing protocol (the pages give no recipe; this is the stated reading): a CPU
``torch.Generator`` seeded with ``seed``; values drawn as float32 standard normals in the
order Q, K, V, dO; then rounded to the compute dtype.  For the packed varlen workload the
sequence lengths are drawn first (uniform integers in [lo, hi]), then qkv.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    """One attention problem shape.  ``scale=None`` means 1/sqrt(d)."""
    name: str
    dtype: str
    B: int = 1
    Hq: int = 1
    Hkv: int = 1
    N: int = 0
    d: int = 64
    causal: bool = False
    scale: float | None = None
    backward: bool = False
    # varlen: number of sequences and the inclusive length range
    varlen: tuple | None = None
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


# The workloads the method is exercised on.  The second is shaped like the pages' A10 example
# (one batch, 32 heads, 2048 tokens, head_dim 64); the others are the GQA / varlen / long
# context training shapes.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32 B1 H2 N128 d64 fp32 fwd", "f32", B=1, Hq=2, Hkv=2, N=128, d=64,
                         causal=False, scale=1.0 / 8.0, backward=False),
    # the fp32 configuration's shape at B * H = 256: enough work for the CUDA-core kernel not to be
    # launch-bound
    "f32_bh256": Workload("f32_bh256 B128 H2 N128 d64 fp32 fwd", "f32", B=128, Hq=2, Hkv=2, N=128, d=64,
                          causal=False, scale=1.0 / 8.0, backward=False),
    "mha_f16": Workload("mha_f16 B1 H32 N2048 d64 fp16 fwd", "f16", B=1, Hq=32, Hkv=32, N=2048,
                        d=64, causal=False, scale=1.0 / 8.0, backward=False),
    "mha_f16_causal": Workload("mha_f16_causal B1 H32 N2048 d64 fp16 causal fwd", "f16", B=1,
                               Hq=32, Hkv=32, N=2048, d=64, causal=True, scale=1.0 / 8.0),
    "gqa_bf16": Workload("gqa_bf16 B4 Hq32 Hkv8 N2048 d128 bf16 causal fwd+bwd", "bf16", B=4,
                         Hq=32, Hkv=8, N=2048, d=128, causal=True, scale=None, backward=True),
    "varlen_bf16": Workload("varlen_bf16 16 seqs L~U[64,4096] H16 d128 bf16 causal fwd", "bf16",
                            Hq=16, Hkv=16, d=128, causal=True, scale=None, varlen=(16, 64, 4096)),
    "varlen_bf16_train": Workload("varlen_bf16_train 16 seqs L~U[64,4096] H16 d128 bf16 causal fwd+bwd", "bf16",
                                  Hq=16, Hkv=16, d=128, causal=True, scale=None, varlen=(16, 64, 4096),
                                  backward=True),
    "long_bf16": Workload("long_bf16 B1 Hq32 Hkv8 N32768 d128 bf16 causal fwd+bwd", "bf16", B=1,
                          Hq=32, Hkv=8, N=32768, d=128, causal=True, scale=None, backward=True),
    # many short sequences (the short-sequence kernel): 6144 problems of 64 tokens, head_dim 64,
    # the diffusion-model shape of the attention-operator article's section 2.3 (64 queries,
    # 768 = 12 x 64 channels) as self-attention
    "short_bf16": Workload("short_bf16 B512 H12 N64 d64 bf16 fwd", "bf16", B=512, Hq=12, Hkv=12, N=64, d=64,
                           causal=False, scale=None),
    # prefill against a cache (cross-attention forward and backward, Nq != Nk): a 2048-token chunk
    # whose queries are the last 2048 positions of a 16384-key sequence (bottom-right causal mask)
    "cross_bf16": Workload("cross_bf16 B2 Hq32 Hkv8 Nq2048 Nk16384 d128 bf16 causal fwd+bwd", "bf16", B=2, Hq=32,
                           Hkv=8, N=16384, d=128, causal=True, scale=None, backward=True,
                           extra={"Nq": 2048, "cross": True}),
    # decode against a KV cache: one new token per sequence, caches of U[16384, 32768] keys
    "decode_bf16": Workload("decode_bf16 B8 Hq32 Hkv8 Nq1 cache U[16384,32768] of 32768 d128 bf16", "bf16", B=8,
                            Hq=32, Hkv=8, N=32768, d=128, causal=True, scale=None,
                            extra={"Nq": 1, "lens": (16384, 32768)}),
}


def generator(seed: int) -> torch.Generator:
    return torch.Generator("cpu").manual_seed(int(seed))


def dense_inputs(B, Hq, Hkv, N, d, dtype: str, seed: int = 0, with_dout: bool = True):
    """Q [B,Hq,N,d], K and V [B,Hkv,N,d], dO [B,Hq,N,d] on the CPU, in ``dtype``."""
    g = generator(seed)
    tdt = DTYPES[dtype]
    q = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float32).to(tdt)
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32).to(tdt)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float32).to(tdt)
    dout = torch.randn(B, Hq, N, d, generator=g, dtype=torch.float32).to(tdt) if with_dout else None
    return q, k, v, dout


def varlen_lengths(nseq: int, lo: int, hi: int, seed: int = 0) -> list[int]:
    g = generator(seed)
    return torch.randint(lo, hi + 1, (nseq,), generator=g).tolist()


def cu_seqlens_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def varlen_inputs(lengths, H: int, d: int, dtype: str, seed: int = 0, with_dout: bool = False):
    """Packed qkv [T,3,H,d] (and dO [T,H,d]) for the given lengths, plus cu_seqlens int32.

    When ``lengths`` is an int triple (nseq, lo, hi) the lengths are drawn first from the
    same generator, then qkv."""
    g = generator(seed)
    if isinstance(lengths, tuple) and len(lengths) == 3 and not isinstance(lengths[0], list):
        nseq, lo, hi = lengths
        lengths = torch.randint(lo, hi + 1, (nseq,), generator=g).tolist()
    lengths = [int(x) for x in lengths]
    T = sum(lengths)
    tdt = DTYPES[dtype]
    qkv = torch.randn(T, 3, H, d, generator=g, dtype=torch.float32).to(tdt)
    dout = torch.randn(T, H, d, generator=g, dtype=torch.float32).to(tdt) if with_dout else None
    return qkv, cu_seqlens_from_lengths(lengths), lengths, dout


def kvcache_inputs(B, Hq, Hkv, Nq, Nk, d, dtype: str, lens=None, seed: int = 0):
    """Q [B,Hq,Nq,d], K and V caches [B,Hkv,Nk,d] on the CPU in ``dtype``, and the cache
    lengths as int32 [B] (None when ``lens`` is None).  ``lens`` is a list of lengths or an
    inclusive range (lo, hi) drawn first from the generator, then Q, K, V."""
    g = generator(seed)
    if isinstance(lens, tuple):
        lens = torch.randint(lens[0], lens[1] + 1, (B,), generator=g).tolist()
    tdt = DTYPES[dtype]
    q = torch.randn(B, Hq, Nq, d, generator=g, dtype=torch.float32).to(tdt)
    k = torch.randn(B, Hkv, Nk, d, generator=g, dtype=torch.float32).to(tdt)
    v = torch.randn(B, Hkv, Nk, d, generator=g, dtype=torch.float32).to(tdt)
    return q, k, v, None if lens is None else torch.tensor([int(x) for x in lens], dtype=torch.int32)


def kvcache_visible_pairs(lens, Nq: int, causal: bool) -> int:
    """(query, key) pairs that enter the KV-cache forward: Nq * L per batch, or under the
    bottom-right causal mask sum_i clamp(L - Nq + i + 1, 0, L)."""
    total = 0
    for L in lens:
        L = int(L)
        if causal:
            total += sum(min(L, max(0, L - Nq + i + 1)) for i in range(Nq))
        else:
            total += Nq * L
    return total


def kvcache_fwd_flops(lens, Hq, Nq, d, causal: bool) -> float:
    """Two contractions (Q.K^T and P.V) of 2 d FLOPs per visible pair per query head."""
    return 4.0 * Hq * d * kvcache_visible_pairs(lens, Nq, causal)


def fwd_flops(B, Hq, N, d, causal: bool) -> float:
    """Algorithmic forward FLOPs: two N x N x d contractions per head (4 B Hq N^2 d), halved
    when causal (the masked half is never computed)."""
    f = 4.0 * B * Hq * N * N * d
    return f / 2 if causal else f


def varlen_fwd_flops(lengths, H, d, causal: bool) -> float:
    return sum(fwd_flops(1, H, int(n), d, causal) for n in lengths)


def bwd_flops(B, Hq, N, d, causal: bool) -> float:
    """Backward: five N x N x d contractions against the forward's two (2.5x)."""
    return 2.5 * fwd_flops(B, Hq, N, d, causal)
