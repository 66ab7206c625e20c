"""Element-wise comparison of CUDA results with the CPU oracle.

Tolerances: per-token outputs |gpu - ref| <= 1e-6 + 1e-5 |ref|; gradients
|gpu - ref| <= 1e-6 + 1e-4 |ref|, plus half a unit in the last place of the
gradient dtype at |ref| when gradients are stored in bf16/fp16 (the rounding of
the store itself). Non-finite values must match in class (NaN, +inf, -inf);
zero-gradient rows must be exactly zero.
"""
from __future__ import annotations

import numpy as np
import torch

LOSS_RTOL, LOSS_ATOL = 1e-5, 1e-6
GRAD_RTOL, GRAD_ATOL = 1e-4, 1e-6

_MANT = {torch.bfloat16: (7, -126), torch.float16: (10, -14)}


def to64(x: torch.Tensor) -> np.ndarray:
    """Exact upcast of device values to host float64."""
    return x.detach().float().cpu().double().numpy()


def half_ulp(ref: np.ndarray, dtype) -> np.ndarray:
    if dtype not in _MANT:
        return np.zeros_like(ref)
    mant, emin = _MANT[dtype]
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.where(a > 0, np.ldexp(0.5, (e - mant).astype(np.int64)), np.ldexp(0.5, emin - mant))


def assert_close(got, ref, rtol, atol, what, grad_dtype=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    for name, fn in (("NaN", np.isnan), ("+inf", np.isposinf), ("-inf", np.isneginf)):
        bad = fn(got) != fn(ref)
        assert not bad.any(), f"{what}: {name} class differs at {np.argwhere(bad)[:5].tolist()}"
    fin = np.isfinite(ref)
    tol = atol + rtol * np.abs(ref)
    if grad_dtype is not None:
        tol = tol + half_ulp(ref, grad_dtype)
    err = np.where(fin, np.abs(np.where(fin, got, 0.0) - np.where(fin, ref, 0.0)), 0.0)
    over = fin & (err > tol)
    if over.any():
        i = tuple(np.argwhere(over)[0])
        raise AssertionError(f"{what}: {over.sum()} elements out of tolerance; first at {i}: "
                             f"gpu={got[i]!r} ref={ref[i]!r} tol={tol[i]!r}; max err {err[fin].max():.3e}")


def assert_loss(got, ref, what):
    assert_close(got, ref, LOSS_RTOL, LOSS_ATOL, what)


def assert_grad(got, ref, what, grad_dtype=None):
    assert_close(got, ref, GRAD_RTOL, GRAD_ATOL, what, grad_dtype)


def assert_zero_rows(grad: np.ndarray, rows, what):
    for r in rows:
        assert np.all(grad[r] == 0.0), f"{what}: row {r} gradient is not exactly zero"
