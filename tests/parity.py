"""Comparison helpers for the GPU-vs-oracle parity tests (no attention arithmetic here).

Tolerances (max absolute error, outputs and gradients alike): fp32 1e-5, fp16 2e-3,
bf16 1e-2.  They gate the kernel's fp32 result before the final rounding to the storage dtype
(ATTN_FLAG_OUT_F32).  The stored fp16/bf16 outputs are checked against
tol + half an ulp of the storage dtype at the value, since a correctly rounded bf16 value
of magnitude >= 4 can already sit 0.0156 away from the exact one."""
import numpy as np
import torch

TOL = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 1e-2}
EPS = {torch.float16: 2.0 ** -10, torch.bfloat16: 2.0 ** -7}


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def max_abs(a, b) -> float:
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)))


def assert_close_f32(gpu, ref, dtype, what=""):
    """gpu: the kernel's fp32 result; ref: the fp64 oracle."""
    g = to_np(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = max_abs(g, ref)
    assert err <= TOL[dtype], f"{what}: max abs error {err:.3e} > {TOL[dtype]:.1e}"
    return err


def half_ulp(x: np.ndarray, dtype) -> np.ndarray:
    if dtype == torch.float32:
        return np.zeros_like(x)
    _, e = np.frexp(np.abs(x))  # |x| = m 2^e, m in [0.5, 1)
    return 0.5 * EPS[dtype] * np.ldexp(1.0, (e - 1).astype(np.int64))


def assert_close_native(gpu, ref, dtype, what=""):
    """gpu: a stored fp16/bf16/fp32 tensor; ref: the fp64 oracle."""
    g = to_np(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    bound = TOL[dtype] + half_ulp(np.maximum(np.abs(ref), np.abs(g)), dtype)
    excess = np.abs(g - ref) - bound
    worst = float(np.max(excess)) if excess.size else -1.0
    assert worst <= 0, f"{what}: exceeds tol + half ulp by {worst:.3e}"
    return max_abs(g, ref)
