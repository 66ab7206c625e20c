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


def assert_close(got, ref, rtol, atol, what, grad_dtype=None, floor=None):
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
    if floor is not None:
        tol = tol + np.asarray(floor, dtype=np.float64)
    err = np.where(fin, np.abs(np.where(fin, got, 0.0) - np.where(fin, ref, 0.0)), 0.0)
    over = fin & (err > tol)
    if over.any():
        i = tuple(np.argwhere(over)[0])
        raise AssertionError(f"{what}: {over.sum()} elements out of tolerance; first at {i}: "
                             f"gpu={got[i]!r} ref={ref[i]!r} tol={tol[i]!r}; max err {err[fin].max():.3e}")


def assert_loss(got, ref, what):
    assert_close(got, ref, LOSS_RTOL, LOSS_ATOL, what)


def assert_grad(got, ref, what, grad_dtype=None, floor=None):
    """`floor`: an extra per-element allowance (kl_branch_floor), added to the
    stated tolerance only where the arithmetic cannot reach it."""
    assert_close(got, ref, GRAD_RTOL, GRAD_ATOL, what, grad_dtype, floor)


def kl_branch_floor(s64, t64, beta, g=None):
    """The fp32 rounding floor of the KL-branch gradients (reading R21): at beta
    = 1 the student gradient g p_j (D_j - KL), D = ln p - ln q, and at beta = 0
    the teacher gradient g q_j (D_j - KL), D = ln q - ln p, are small
    differences of log-ratios of tens of nats on a row whose target is nearly
    one-hot against a broad other side; the saved KL alone is rounded to fp32
    (half an ulp of |KL|) and every log-ratio carries its own rounding. The
    allowance is |g| tgt_j 2^-20 (|D_j| + |KL| + max_k tgt_k |D_k|), taken from
    the oracle's float64 statistics. Returns (floor for dS, floor for dT); zero
    where the branch does not apply or the row has no finite value."""
    from oracle import oracle as O

    s64 = np.asarray(s64, dtype=np.float64)
    t64 = np.asarray(t64, dtype=np.float64)
    zero = np.zeros_like(s64)
    if beta not in (0.0, 1.0):
        return zero, zero
    n = s64.shape[0]
    gg = np.ones(n) if g is None else np.abs(np.asarray(g, dtype=np.float64)).reshape(n)
    m_s, l_s, c_s = O.row_stats(s64)
    m_t, l_t, c_t = O.row_stats(t64)
    ok = (c_s == 0) & (c_t == 0)
    with np.errstate(invalid="ignore", over="ignore"):
        lp = np.where(np.isfinite(s64), s64 - m_s[:, None] - l_s[:, None], -np.inf)
        lq = np.where(np.isfinite(t64), t64 - m_t[:, None] - l_t[:, None], -np.inf)
        tgt_l, oth_l = (lp, lq) if beta == 1.0 else (lq, lp)
        tgt = np.exp(tgt_l)
        d = np.where(np.isfinite(tgt_l) & np.isfinite(oth_l), tgt_l - oth_l, 0.0)
        kl = np.sum(np.where(tgt > 0, tgt * d, 0.0), axis=1)
        fl = gg[:, None] * tgt * 2.0**-20 * (np.abs(d) + np.abs(kl)[:, None]
                                              + np.max(tgt * np.abs(d), axis=1)[:, None])
    fl = np.where(ok[:, None] & np.isfinite(kl)[:, None], fl, 0.0)
    return (fl, zero) if beta == 1.0 else (zero, fl)


def assert_zero_rows(grad: np.ndarray, rows, what):
    for r in rows:
        assert np.all(grad[r] == 0.0), f"{what}: row {r} gradient is not exactly zero"
