"""The fused-linear JSD (tensor-core logits tiles, never written to memory)
against the CPU oracle's composition: float64 logits from the same bf16 hidden
states and head weights, the JSD row oracle, and the chain rule through the
heads.

Tolerance, derived from the arithmetic (the stated per-element tolerances of
the logits ops apply to logits given as inputs; here the logits are formed in
fp32 from exact bf16 products):
  * logit j of a row is a sum of H exact products accumulated in fp32, so its
    error is at most delta_j = 2 H 2^-24 sum_k |h_k w_jk|;
  * the loss: the stated 1e-6 + 1e-5 |ref| plus the first-order effect of the
    logit errors, sum_j (|dS_j| delta_s_j + |dT_j| delta_t_j) at g = 1;
  * dh = dS w and dw = dS^T h: the stated gradient tolerance of each dS_j
    (1e-6 + 1e-4 |dS_j|) plus the effect of the logit errors on dS_j,
    4 (p_j + q_j + |dS_j|) max delta, carried through the sum with |w| (|h|),
    plus the split of dS into two bf16 parts (2^-16 relative) and the fp32
    accumulation of the sum (2 K 2^-24 relative), both against sum |dS w|.
Each element must be within that bound; and, so that a small systematic error
(a scale, a dropped term) cannot hide inside a loose bound, the median
relative error over the elements that are not tiny must stay below 1e-4."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity_util import to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from softmax_divergence_lm_gb300 import build
    build.build()
    from softmax_divergence_lm_gb300 import binding
    binding.load()
    return binding


def run(B, h_s, w_s, h_t, w_t, beta, g, student=True, teacher=True):
    heads = B.make_heads(h_s, w_s, h_t, w_t)
    n, v = h_s.shape[0], w_s.shape[0]
    fwd_b, bwd_b = B.vpd_jsd_linear_workspace(heads, student, teacher)
    ws = torch.empty(max(fwd_b, bwd_b, 16), dtype=torch.uint8, device="cuda")
    loss = torch.full((n,), 7.0, device="cuda")
    saved = torch.full((n, 6), 7.0, device="cuda")
    c0 = B.vpd_launch_count()
    B.vpd_jsd_linear_fwd(heads, beta, loss, saved, ws)
    dh_s = torch.full((n, h_s.shape[1]), 5.0, device="cuda") if student else None
    dw_s = torch.full((v, h_s.shape[1]), 5.0, device="cuda") if student else None
    dh_t = torch.full((n, h_t.shape[1]), 5.0, device="cuda") if teacher else None
    dw_t = torch.full((v, h_t.shape[1]), 5.0, device="cuda") if teacher else None
    B.vpd_jsd_linear_bwd(heads, beta, g, loss, saved, dh_s, dw_s, dh_t, dw_t, ws)
    torch.cuda.synchronize()
    B.vpd_device_status()
    launches = B.vpd_launch_count() - c0
    return loss, saved, dh_s, dw_s, dh_t, dw_t, launches


def _bounds(h, w, s64):
    """delta_j per row: 2 H 2^-24 sum_k |h_k w_jk|."""
    H = h.shape[1]
    return 2.0 * H * 2.0**-24 * (np.abs(h) @ np.abs(w).T)


def _check_tol(got, ref, tol, what):
    got, ref = np.asarray(got), np.asarray(ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    over = err > tol
    if over.any():
        i = tuple(np.argwhere(over)[0])
        raise AssertionError(f"{what}: {over.sum()} of {err.size} elements beyond the derived bound; first at {i}: "
                             f"gpu={got[i]!r} ref={ref[i]!r} bound={tol[i]!r}")
    big = np.abs(ref) > 1e-3 * np.max(np.abs(ref))
    med = float(np.median(err[big] / np.abs(ref[big]))) if big.any() else 0.0
    assert med <= 1e-4, f"{what}: median relative error {med:.3e} above 1e-4"


def check(B, h_s, w_s, h_t, w_t, beta, label, rows=None, vocab_rows=None, student=True, teacher=True):
    n = h_s.shape[0]
    gen = torch.Generator(device="cpu").manual_seed(3)
    g = torch.randn(n, generator=gen).cuda()
    loss, saved, dh_s, dw_s, dh_t, dw_t, launches = run(B, h_s, w_s, h_t, w_t, beta, g, student, teacher)
    assert launches >= 4
    hs, ws_, ht, wt = (to64(x) for x in (h_s, w_s, h_t, w_t))
    g64 = to64(g)
    rl, ra, rb, rdhs, rdws, rdht, rdwt = O.jsd_linear(hs, ws_, ht, wt, beta, g64, threads=8)
    # logits, statistics and the logits gradient at g = 1 for the bounds
    s64, t64 = hs @ ws_.T, ht @ wt.T
    _, _, _, ds1, dt1 = O.jsd(s64, t64, beta, None, threads=8)
    _, _, _, dsg, dtg = O.jsd(s64, t64, beta, g64, threads=8)
    ms, ls, _ = O.row_stats(s64)
    mt, lt, _ = O.row_stats(t64)
    p = np.exp(s64 - ms[:, None] - ls[:, None])
    q = np.exp(t64 - mt[:, None] - lt[:, None])
    d_s, d_t = _bounds(hs, ws_, s64), _bounds(ht, wt, t64)
    tag = f"{label} beta={beta}"
    # loss and saved statistics
    tol = 1e-6 + 1e-5 * np.abs(rl) + np.sum(np.abs(ds1) * d_s + np.abs(dt1) * d_t, axis=1)
    _check_tol(to64(loss), rl, tol, tag + " loss")
    sv = to64(saved)
    _check_tol(sv[:, 0], ms, 1e-6 + np.max(d_s, axis=1), tag + " saved m_s")
    _check_tol(sv[:, 2], mt, 1e-6 + np.max(d_t, axis=1), tag + " saved m_t")
    # gradients through the heads
    for want, name, dhx, dwx, rdh, rdw, hx, wx, dgx, dbx in (
            (student, "student", dh_s, dw_s, rdhs, rdws, hs, ws_, dsg, d_s),
            (teacher, "teacher", dh_t, dw_t, rdht, rdwt, ht, wt, dtg, d_t)):
        if not want:
            continue
        dmax = np.max(d_s) + np.max(d_t)
        e = 1e-6 * np.abs(g64)[:, None] + 1e-4 * np.abs(dgx) + 4.0 * (np.abs(g64)[:, None] * (p + q) + np.abs(dgx)) * dmax
        split = (2.0**-16 + 2.0 * dgx.shape[1] * 2.0**-24) * (np.abs(dgx) @ np.abs(wx))
        _check_tol(to64(dhx), rdh, 1e-6 + 1e-4 * np.abs(rdh) + e @ np.abs(wx) + split, f"{tag} dh {name}")
        split = (2.0**-16 + 2.0 * dgx.shape[0] * 2.0**-24) * (np.abs(dgx).T @ np.abs(hx))
        _check_tol(to64(dwx), rdw, 1e-6 + 1e-4 * np.abs(rdw) + e.T @ np.abs(hx) + split, f"{tag} dw {name}")
    return loss


@pytest.mark.parametrize("beta", [0.5, 0.0, 1.0, 0.2])
def test_linear_small_every_row(B, beta):
    """Three row tiles (the last ragged), eight vocabulary tiles (the last
    ragged), different hidden sizes for the two heads."""
    from softmax_divergence_lm_gb300 import synth
    h_s, w_s, h_t, w_t = synth.linear_heads(device="cuda", n=300, v=1000, hidden_s=128, hidden_t=192, seed=11)
    check(B, h_s, w_s, h_t, w_t, beta, "small")


def test_linear_detached_teacher_and_chunks(B):
    """More rows than one backward chunk (8192): two chunks, the second ragged
    (300 rows), dW accumulated over both; teacher gradients not wanted."""
    from softmax_divergence_lm_gb300 import synth
    h_s, w_s, h_t, w_t = synth.linear_heads(device="cuda", n=8192 + 300, v=504, hidden_s=64, hidden_t=128, seed=12)
    check(B, h_s, w_s, h_t, w_t, 0.5, "chunks", teacher=False)


def test_linear_teacher_gradients_only(B):
    """Only the teacher head's gradients wanted (the student's skipped in the
    gradient pass), a row count that leaves a partial warp block and whole
    warps past the rows in the last row tile, a ragged last vocabulary tile."""
    from softmax_divergence_lm_gb300 import synth
    h_s, w_s, h_t, w_t = synth.linear_heads(device="cuda", n=200, v=648, hidden_s=64, hidden_t=128, seed=15)
    check(B, h_s, w_s, h_t, w_t, 0.3, "teacher only", student=False)


def test_linear_identical_heads(B):
    """The same head and hidden states on both sides: JSD 0 up to the logit
    rounding, gradients 0 up to it."""
    from softmax_divergence_lm_gb300 import synth
    h, w, _, _ = synth.linear_heads(device="cuda", n=256, v=768, hidden_s=128, hidden_t=128, seed=13)
    g = torch.ones(256, device="cuda")
    loss, _, dh_s, _, _, _, _ = run(B, h, w, h, w, 0.5, g)
    assert np.all(np.abs(to64(loss)) < 1e-6)
    assert np.all(np.abs(to64(dh_s)) < 1e-5)


def test_linear_qwen_heads(B):
    """The pages' head shapes: Qwen2.5 vocabulary (151936), student hidden 896
    (Qwen2.5-0.5B), teacher hidden 1536 (Qwen2.5-1.5B), on 512 rows."""
    from softmax_divergence_lm_gb300 import synth
    h_s, w_s, h_t, w_t = synth.linear_heads(device="cuda", n=512, seed=14)
    check(B, h_s, w_s, h_t, w_t, 0.5, "qwen heads", teacher=False)
