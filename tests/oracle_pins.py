"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with a
fact fixed by the pages or by mathematics: hand-derived closed forms
(``tests/golden/two_token.json``), identities (JSD of a row with itself is 0,
disjoint supports give the binary entropy H(beta), 0 <= JSD_beta <= H(beta),
JSD_beta(s, t) = JSD_{1-beta}(t, s)), the second-order closed form for nearly
identical rows, shift invariance under a large offset and masked-vocabulary
equivalence to the reduced vocabulary ('Add
vocabulary-parallel logprobs, entropy and KL ops', section Tests), +inf KL when
the target has mass on a masked token (same section), the beta = 0 / 1 branches
against a library KL ('[VocabTP] Add vocabulary-parallel generalized JSD with
Triton kernels', section Changes), library log-softmax and entropy routines,
and brute-force central finite differences for every gradient.

The pins are plain functions so that the mutation test can run them against a
deliberately broken copy of the oracle.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy import special, stats

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "two_token.json")
INTERIOR = (0.1, 0.25, 0.5, 0.75, 0.9)
ALL_BETAS = (0.0,) + INTERIOR + (1.0,)


def binary_entropy(b: float) -> float:
    return -b * math.log(b) - (1.0 - b) * math.log(1.0 - b)


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    same_class = np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(np.isposinf(a), np.isposinf(b)) \
        and np.array_equal(np.isneginf(a), np.isneginf(b))
    assert same_class, f"{what}: non-finite classes differ\n{a}\n{b}"
    fa, fb = a[np.isfinite(a)], b[np.isfinite(b)]
    ok = np.all(np.abs(fa - fb) <= atol + rtol * np.abs(fb))
    assert ok, f"{what}: max abs diff {np.max(np.abs(fa - fb)) if fa.size else 0}"


def _value(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, {"log": math.log, "inf": math.inf}))
    return float(x)


def _logits(seq):
    return np.array([[float("-inf") if v == "-inf" else _value(v) for v in seq]])


# ---------------------------------------------------------------------------
def pin_golden_two_token():
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        expected = _value(c["value"])
        assert math.isclose(_value(c["expr"]), expected, rel_tol=1e-14) or expected == _value(c["expr"]), c["name"]
        if c["op"] == "jsd":
            got = O.jsd(_logits(c["student"]), _logits(c["teacher"]), c["beta"], grad=False)[0][0]
        elif c["op"] == "kl":
            got = O.kl(_logits(c["student"]), _logits(c["teacher"]), c["reverse"], grad=False)[0][0]
        elif c["op"] == "entropy":
            got = O.entropy(_logits(c["x"]), grad=False)[0][0]
        elif c["op"] == "logprobs":
            got = O.logprobs(_logits(c["x"]), [[c["index"]]], grad=False)[0][0, 0]
        else:
            raise AssertionError(c["op"])
        if math.isinf(expected):
            assert got == expected, (c["name"], got)
        else:
            assert math.isclose(got, expected, rel_tol=1e-13, abs_tol=1e-15), (c["name"], got, expected)


def pin_identical_inputs_zero():
    rng = np.random.default_rng(11)
    s = rng.normal(0, 3, (6, 37))
    s[1, :5] = -np.inf
    for beta in ALL_BETAS:
        loss, _, _, ds, dt = O.jsd(s, s.copy(), beta)
        assert np.all(np.abs(loss) < 1e-14), (beta, loss)
        assert np.all(np.abs(ds) < 1e-14) and np.all(np.abs(dt) < 1e-14), beta


def pin_disjoint_support_binary_entropy():
    rng = np.random.default_rng(12)
    v = 29
    s = rng.normal(0, 2, (5, v))
    t = rng.normal(0, 2, (5, v))
    for r in range(5):
        own = rng.random(v) < 0.5
        own[0], own[1] = True, False
        s[r, ~own] = -np.inf
        t[r, own] = -np.inf
    for beta in INTERIOR:
        loss, a, b, ds, dt = O.jsd(s, t, beta)
        _close(loss, np.full(5, binary_entropy(beta)), 1e-13, 1e-14, f"H({beta})")
        # each KL-to-mixture is -ln of the weight of its own side
        _close(a, np.full(5, -math.log(beta)), 1e-13, 1e-14, "KL(q||M)")
        _close(b, np.full(5, -math.log(1 - beta)), 1e-13, 1e-14, "KL(p||M)")
    for beta in (0.0, 1.0):
        loss, _, _, ds, dt = O.jsd(s, t, beta)
        assert np.all(np.isposinf(loss)), beta
        assert np.all(ds == 0) and np.all(dt == 0), beta


def pin_bounds():
    rng = np.random.default_rng(13)
    for scale in (0.1, 1.0, 4.0, 20.0):
        s = rng.normal(0, scale, (8, 41))
        t = rng.normal(0, scale, (8, 41))
        s[:, 3] += 15.0
        for beta in INTERIOR:
            loss = O.jsd(s, t, beta, grad=False)[0]
            assert np.all(loss >= -1e-15), (scale, beta, loss.min())
            assert np.all(loss <= binary_entropy(beta) + 1e-13), (scale, beta, loss.max())
        for reverse in (False, True):
            assert np.all(O.kl(s, t, reverse, grad=False)[0] >= -1e-15)


def pin_swap_symmetry():
    rng = np.random.default_rng(14)
    s = rng.normal(0, 2, (6, 23))
    t = rng.normal(0, 2, (6, 23))
    s[0, 2] = -np.inf
    t[1, 5] = -np.inf
    g = rng.normal(size=6)
    for beta in ALL_BETAS:
        l1, _, _, ds1, dt1 = O.jsd(s, t, beta, g)
        l2, _, _, ds2, dt2 = O.jsd(t, s, 1.0 - beta, g)
        _close(l1, l2, 1e-12, 1e-14, f"swap {beta}")
        _close(ds1, dt2, 1e-10, 1e-14, f"swap grad s {beta}")
        _close(dt1, ds2, 1e-10, 1e-14, f"swap grad t {beta}")


def pin_shift_invariance():
    rng = np.random.default_rng(15)
    # logits on a 2^-9 grid so that adding the offsets below is exact
    s = np.round(rng.normal(0, 3, (5, 31)) * 512) / 512
    t = np.round(rng.normal(0, 3, (5, 31)) * 512) / 512
    s[2, 4] = -np.inf
    t[3, 6] = -np.inf
    s2, t2 = s + 1.0e4, t - 3.0e3
    for beta in ALL_BETAS:
        a = O.jsd(s, t, beta)
        b = O.jsd(s2, t2, beta)
        for x, y in zip(a, b):
            _close(x, y, 1e-11, 1e-13, f"shift {beta}")
    for reverse in (False, True):
        for x, y in zip(O.kl(s, t, reverse), O.kl(s2, t2, reverse)):
            _close(x, y, 1e-11, 1e-13, "shift kl")
    for x, y in zip(O.entropy(s), O.entropy(s2)):
        _close(x, y, 1e-11, 1e-13, "shift entropy")
    idx = rng.integers(0, 31, (5, 3))
    a, b = O.logprobs(s, idx), O.logprobs(s2, idx)
    _close(a[0], b[0], 1e-11, 1e-13, "shift logprobs")
    _close(a[1], b[1], 1e-11, 1e-13, "shift logprobs grad")


def pin_masked_vocab_equivalence():
    rng = np.random.default_rng(16)
    v = 40
    s = rng.normal(0, 2, (4, v))
    t = rng.normal(0, 2, (4, v))
    masked = np.zeros(v, dtype=bool)
    masked[[0, 7, 8, 21, 39]] = True
    sm, tm = s.copy(), t.copy()
    sm[:, masked] = -np.inf
    tm[:, masked] = -np.inf
    sr, tr = s[:, ~masked], t[:, ~masked]
    for beta in ALL_BETAS:
        full = O.jsd(sm, tm, beta)
        red = O.jsd(sr, tr, beta)
        _close(full[0], red[0], 1e-13, 1e-14, "masked loss")
        _close(full[3][:, ~masked], red[3], 1e-12, 1e-14, "masked ds")
        _close(full[4][:, ~masked], red[4], 1e-12, 1e-14, "masked dt")
        assert np.all(full[3][:, masked] == 0) and np.all(full[4][:, masked] == 0)
    ef, er = O.entropy(sm), O.entropy(sr)
    _close(ef[0], er[0], 1e-13, 1e-14, "masked entropy")
    _close(ef[1][:, ~masked], er[1], 1e-12, 1e-14, "masked entropy grad")


def pin_kl_infinite_on_masked_target_mass():
    rng = np.random.default_rng(17)
    s = rng.normal(0, 1, (3, 16))
    t = rng.normal(0, 1, (3, 16))
    s[:, 5] = -np.inf
    t[0, 5] = 0.0
    t[1, 5] = t[1].max() - 120.0  # mass e^-120 relative to the top token: 0 in fp32
    t[2, 5] = -np.inf             # no mass there: finite
    loss, ds, dt = O.kl(s, t, reverse=False)
    assert np.isposinf(loss[0]) and np.isposinf(loss[1]) and np.isfinite(loss[2]), loss
    assert np.all(ds[:2] == 0) and np.all(dt[:2] == 0)
    j0 = O.jsd(s, t, 0.0)
    assert np.isposinf(j0[0][0]) and np.isposinf(j0[0][1]) and np.isfinite(j0[0][2])
    # reverse KL: the student is the target and has no mass on token 5
    assert np.all(np.isfinite(O.kl(s, t, reverse=True, grad=False)[0]))
    # the mirror image for reverse KL
    r = O.kl(t, s, reverse=True)
    assert np.isposinf(r[0][0]) and np.isposinf(r[0][1]) and np.all(r[1][:2] == 0)
    # interior JSD stays finite and within the bound
    for beta in INTERIOR:
        li = O.jsd(s, t, beta, grad=False)[0]
        assert np.all(np.isfinite(li)) and np.all(li <= binary_entropy(beta) + 1e-13)


def pin_endpoints_direct_kl():
    rng = np.random.default_rng(18)
    s = rng.normal(0, 2, (5, 19))
    t = rng.normal(0, 2, (5, 19))
    p = special.softmax(s, axis=1)
    q = special.softmax(t, axis=1)
    fwd = special.rel_entr(q, p).sum(axis=1)
    rev = special.rel_entr(p, q).sum(axis=1)
    _close(O.jsd(s, t, 0.0, grad=False)[0], fwd, 1e-12, 1e-14, "beta=0")
    _close(O.jsd(s, t, 1.0, grad=False)[0], rev, 1e-12, 1e-14, "beta=1")
    _close(O.kl(s, t, False, grad=False)[0], fwd, 1e-12, 1e-14, "kl fwd")
    _close(O.kl(s, t, True, grad=False)[0], rev, 1e-12, 1e-14, "kl rev")
    # the interior close to an endpoint is not that endpoint (branches, not limits):
    # it tends to 0 there, since both sides of the mixture become the same
    assert np.all(O.jsd(s, t, 1e-6, grad=False)[0] < 1e-4)


def _fd_check(fn, x, grad, label, h=1e-6, atol=1e-8):
    """Central differences of the scalar fn(x) against the analytic grad."""
    x = np.array(x, dtype=np.float64)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        if not np.isfinite(x[i]):
            assert grad[i] == 0.0, (label, i, grad[i])
            continue
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        num = (fn(xp) - fn(xm)) / (2 * h)
        assert abs(num - grad[i]) <= atol + 1e-6 * abs(num), (label, i, num, grad[i])


def pin_finite_differences():
    rng = np.random.default_rng(19)
    n, v = 3, 7
    s = rng.normal(0, 1.5, (n, v))
    t = rng.normal(0, 1.5, (n, v))
    g = rng.normal(0, 1, n)
    s_int, t_int = s.copy(), t.copy()
    s_int[0, 2] = -np.inf
    t_int[1, 4] = -np.inf
    for beta in (0.3, 0.5, 0.8):
        _, _, _, ds, dt = O.jsd(s_int, t_int, beta, g)
        _fd_check(lambda x: float(np.dot(g, O.jsd(x, t_int, beta, grad=False)[0])), s_int, ds, f"jsd ds {beta}")
        _fd_check(lambda x: float(np.dot(g, O.jsd(s_int, x, beta, grad=False)[0])), t_int, dt, f"jsd dt {beta}")
    # endpoints: mask only tokens the target does not cover, so KL stays finite
    s_fw, t_fw = s.copy(), t.copy()
    t_fw[0, 2] = -np.inf  # the teacher (forward-KL target) masks a token
    s_rv, t_rv = s.copy(), t.copy()
    s_rv[1, 4] = -np.inf  # the student (reverse-KL target) masks a token
    for beta, (sa, ta) in ((0.0, (s_fw, t_fw)), (1.0, (s_rv, t_rv))):
        _, _, _, ds, dt = O.jsd(sa, ta, beta, g)
        _fd_check(lambda x: float(np.dot(g, O.jsd(x, ta, beta, grad=False)[0])), sa, ds, f"jsd ds {beta}")
        _fd_check(lambda x: float(np.dot(g, O.jsd(sa, x, beta, grad=False)[0])), ta, dt, f"jsd dt {beta}")
    for reverse, (sa, ta) in ((False, (s_fw, t_fw)), (True, (s_rv, t_rv))):
        _, ds, dt = O.kl(sa, ta, reverse, g)
        _fd_check(lambda x: float(np.dot(g, O.kl(x, ta, reverse, grad=False)[0])), sa, ds, f"kl ds {reverse}")
        _fd_check(lambda x: float(np.dot(g, O.kl(sa, x, reverse, grad=False)[0])), ta, dt, f"kl dt {reverse}")
    _, dx = O.entropy(s_int, g)
    _fd_check(lambda x: float(np.dot(g, O.entropy(x, grad=False)[0])), s_int, dx, "entropy")
    idx = np.array([[1, 3, 3], [0, -100, 6], [5, 4, 1]])
    gk = rng.normal(0, 1, (n, 3))
    _, dx, _ = O.logprobs(s_int, idx, -100, gk)
    _fd_check(lambda x: float(np.sum(np.nan_to_num(O.logprobs(x, idx, -100, grad=False)[0]) * gk)), s_int, dx,
              "logprobs")


def jsd_second_order(s, t, beta):
    """The leading term of JSD_beta between softmax(s) and softmax(t) for
    t = s + eps * d: beta (1 - beta) / 2 * Var_p(t - s), p = softmax(s). It
    follows from KL(a || b) = 1/2 sum (a - b)^2 / b + O(|a - b|^3) with
    M = p (1 + beta eps u), q = p (1 + eps u), u = d - E_p d to first order; the
    relative remainder is O(eps). Computed by a library softmax."""
    p = special.softmax(s, axis=1)
    d = t - s
    mu = np.sum(p * d, axis=1)
    return 0.5 * beta * (1.0 - beta) * np.sum(p * (d - mu[:, None]) ** 2, axis=1)


def pin_jsd_second_order_near_identical_rows():
    # nearly identical rows: the divergence is a difference of O(eps) terms
    # that cancel to O(eps^2); the closed form above is exact to O(eps) relative
    rng = np.random.default_rng(27)
    s = rng.normal(0, 2, (4, 2048))
    d = rng.normal(0, 1, (4, 2048))
    for eps in (1e-3, 1e-4):
        t = s + eps * d
        for beta in (0.2, 0.5, 0.7):
            _close(O.jsd(s, t, beta, grad=False)[0], jsd_second_order(s, t, beta), eps, 0.0,
                   f"second order beta={beta} eps={eps}")


def pin_gradient_rows_sum_to_zero():
    rng = np.random.default_rng(20)
    s = rng.normal(0, 2, (6, 50))
    t = rng.normal(0, 2, (6, 50))
    s[0, :7] = -np.inf
    t[2, 10:20] = -np.inf
    g = rng.normal(size=6)
    for beta in INTERIOR:
        _, _, _, ds, dt = O.jsd(s, t, beta, g)
        assert np.all(np.abs(ds.sum(1)) < 1e-14) and np.all(np.abs(dt.sum(1)) < 1e-14), beta
    _, dx = O.entropy(s, g)
    assert np.all(np.abs(dx.sum(1)) < 1e-14)
    idx = rng.integers(0, 50, (6, 4))
    idx[:, 0] = 20  # always finite in every row
    _, dx, _ = O.logprobs(t, idx, -100, rng.normal(size=(6, 4)))
    assert np.all(np.abs(dx.sum(1)) < 1e-13)


def pin_entropy_closed_forms():
    v = 64
    for support in (1, 2, 5, 64):
        x = np.full((1, v), -np.inf)
        x[0, :support] = 3.25
        h, dx = O.entropy(x)
        assert abs(h[0] - math.log(support)) < 1e-14, support
        assert np.all(np.abs(dx) < 1e-15)
    rng = np.random.default_rng(21)
    x = rng.normal(0, 2, (4, 33))
    _close(O.entropy(x, grad=False)[0], stats.entropy(special.softmax(x, axis=1), axis=1), 1e-12, 1e-14, "entropy")


def pin_kl_uniform_student():
    rng = np.random.default_rng(22)
    v = 50
    t = rng.normal(0, 3, (4, v))
    s = np.zeros((4, v))
    hq = stats.entropy(special.softmax(t, axis=1), axis=1)
    _close(O.kl(s, t, reverse=False, grad=False)[0], math.log(v) - hq, 1e-12, 1e-14, "KL(q||uniform)")


def pin_logprobs_contract():
    rng = np.random.default_rng(23)
    x = rng.normal(0, 2, (3, 12))
    allids = np.tile(np.arange(12), (3, 1))
    out, _, err = O.logprobs(x, allids, grad=False)
    assert err == 0
    _close(np.exp(out).sum(1), np.ones(3), 1e-14, 1e-14, "sum of probs")
    _close(out, special.log_softmax(x, axis=1), 1e-12, 1e-14, "log_softmax")
    xm = x.copy()
    xm[0, 3] = -np.inf
    idx = np.array([[3, -100, 4], [12, 2, 2], [-1, 0, -100]])
    g = np.ones((3, 3))
    out, dx, err = O.logprobs(xm, idx, -100, g)
    assert err == 2, err
    assert out[0, 1] == 0.0 and out[2, 2] == 0.0
    assert np.isneginf(out[0, 0]) and np.isnan(out[1, 0]) and np.isnan(out[2, 0])
    # row 0: only position 2 (token 4) takes gradient
    p0 = special.softmax(np.where(np.isfinite(xm[0]), xm[0], -np.inf))
    want = -p0.copy()
    want[4] += 1.0
    _close(dx[0], want, 1e-12, 1e-14, "row 0 grad")
    # row 1: token 2 twice
    p1 = special.softmax(xm[1])
    want = -2 * p1
    want[2] += 2.0
    _close(dx[1], want, 1e-12, 1e-14, "row 1 grad")


def pin_fully_masked_rows():
    rng = np.random.default_rng(24)
    s = rng.normal(0, 2, (3, 10))
    t = rng.normal(0, 2, (3, 10))
    s[1] = -np.inf            # one input fully masked
    s[2], t[2] = -np.inf, -np.inf  # both fully masked
    g = np.ones(3)
    alone = O.jsd(s[:1], t[:1], 0.5, g[:1])
    for beta in ALL_BETAS:
        loss, _, _, ds, dt = O.jsd(s, t, beta, g)
        assert np.all(np.isnan(loss[1:])), beta
        assert np.all(ds[1:] == 0) and np.all(dt[1:] == 0)
    loss, _, _, ds, dt = O.jsd(s, t, 0.5, g)
    _close(loss[:1], alone[0], 0, 0, "valid row unaffected")
    _close(ds[:1], alone[3], 0, 0, "valid row grad unaffected")
    for reverse in (False, True):
        loss, ds, dt = O.kl(s, t, reverse, g)
        assert np.all(np.isnan(loss[1:])) and np.all(ds[1:] == 0) and np.all(dt[1:] == 0)
    h, dx = O.entropy(s, g)
    assert np.isnan(h[1]) and np.isfinite(h[0]) and np.all(dx[1] == 0)
    out, dx, _ = O.logprobs(s, np.array([[1], [1], [2]]), -100, np.ones((3, 1)))
    assert np.isnan(out[1, 0]) and np.all(dx[1] == 0) and np.all(dx[2] == 0)


def pin_nonfinite_inputs():
    rng = np.random.default_rng(25)
    s = rng.normal(0, 2, (3, 10))
    t = rng.normal(0, 2, (3, 10))
    s[1, 4] = np.nan
    t[2, 7] = np.inf
    for beta in ALL_BETAS:
        loss, _, _, ds, dt = O.jsd(s, t, beta)
        assert np.isfinite(loss[0]) and np.all(np.isnan(loss[1:])), beta
        assert np.all(ds[1:] == 0) and np.all(dt[1:] == 0)
    h, dx = O.entropy(s)
    assert np.isnan(h[1]) and np.all(dx[1] == 0)


def pin_segment_merge():
    rng = np.random.default_rng(26)
    v = 100
    x = rng.normal(0, 3, v) + 50.0
    x[40:55] = -np.inf  # a segment that is entirely masked
    m_ref, lse_ref, code = O.row_stats(x)
    assert code[0] == 0
    for widths in ([100], [0, 100, 0], [40, 15, 45], [10, 0, 30, 15, 0, 45], [1] * 100):
        m, z = O.segment_stats(x, widths)
        assert m == m_ref[0], widths
        assert abs(math.log(z) - lse_ref[0]) < 1e-14, widths
    # fully masked row: every segment contributes (-inf, 0)
    m, z = O.segment_stats(np.full(8, -np.inf), [3, 0, 5])
    assert m == -math.inf and z == 0.0


def pin_torch_fp64_autograd():
    """The pages' check against an independent FP64 dense PyTorch reference
    ('[VocabTP] ...', section Validation): log_softmax + kl_div with autograd."""
    import torch

    rng = np.random.default_rng(27)
    s = rng.normal(0, 2, (4, 21))
    t = rng.normal(0, 2, (4, 21))
    g = rng.normal(size=4)
    for beta in INTERIOR:
        st = torch.tensor(s, requires_grad=True)
        tt = torch.tensor(t, requires_grad=True)
        lp, lq = torch.log_softmax(st, 1), torch.log_softmax(tt, 1)
        lm = torch.logsumexp(torch.stack([lp + math.log(1 - beta), lq + math.log(beta)]), 0)
        kl_qm = torch.nn.functional.kl_div(lm, lq, reduction="none", log_target=True).sum(1)
        kl_pm = torch.nn.functional.kl_div(lm, lp, reduction="none", log_target=True).sum(1)
        loss = beta * kl_qm + (1 - beta) * kl_pm
        (loss * torch.tensor(g)).sum().backward()
        ol, _, _, ds, dt = O.jsd(s, t, beta, g)
        _close(ol, loss.detach().numpy(), 1e-12, 1e-14, f"torch loss {beta}")
        _close(ds, st.grad.numpy(), 1e-10, 1e-14, f"torch ds {beta}")
        _close(dt, tt.grad.numpy(), 1e-10, 1e-14, f"torch dt {beta}")


# ---------------------------------------------------------------------------
# Compositions: fused-linear JSD, cross-entropy, teacher top-k forward KL.
# ---------------------------------------------------------------------------
def pin_linear_logits_brute_force():
    """The logits step of the fused-linear oracle against explicit loops over
    the hidden dimension (pins which operand is transposed)."""
    rng = np.random.default_rng(31)
    n, v, hs, ht = 2, 5, 3, 4
    h_s, w_s = rng.normal(size=(n, hs)), rng.normal(size=(v, hs))
    h_t, w_t = rng.normal(size=(n, ht)), rng.normal(size=(v, ht))
    s = np.array([[sum(h_s[r, k] * w_s[j, k] for k in range(hs)) for j in range(v)] for r in range(n)])
    t = np.array([[sum(h_t[r, k] * w_t[j, k] for k in range(ht)) for j in range(v)] for r in range(n)])
    for beta in (0.0, 0.4, 1.0):
        lin = O.jsd_linear(h_s, w_s, h_t, w_t, beta, grad=False)[0]
        _close(lin, O.jsd(s, t, beta, grad=False)[0], 1e-13, 1e-15, f"linear logits beta={beta}")


def pin_linear_finite_differences():
    """Central differences of the fused-linear loss with respect to every entry
    of both hidden-state matrices and both head weights."""
    rng = np.random.default_rng(32)
    n, v, hs, ht = 3, 6, 4, 3
    h_s, w_s = rng.normal(size=(n, hs)), rng.normal(0, 0.8, (v, hs))
    h_t, w_t = rng.normal(size=(n, ht)), rng.normal(0, 0.8, (v, ht))
    g = rng.normal(size=n)
    for beta in (0.3, 0.0, 1.0):
        _, _, _, dhs, dws, dht, dwt = O.jsd_linear(h_s, w_s, h_t, w_t, beta, g)
        f = lambda a, b, c, d: float(np.dot(g, O.jsd_linear(a, b, c, d, beta, grad=False)[0]))  # noqa: E731
        _fd_check(lambda x: f(x, w_s, h_t, w_t), h_s, dhs, f"linear dh_s {beta}")
        _fd_check(lambda x: f(h_s, x, h_t, w_t), w_s, dws, f"linear dw_s {beta}")
        _fd_check(lambda x: f(h_s, w_s, x, w_t), h_t, dht, f"linear dh_t {beta}")
        _fd_check(lambda x: f(h_s, w_s, h_t, x), w_t, dwt, f"linear dw_t {beta}")


def pin_linear_identical_heads():
    """Identical student and teacher heads and hidden states: JSD 0 and every
    gradient 0 (the JSD of a distribution with itself)."""
    rng = np.random.default_rng(33)
    h, w = rng.normal(size=(4, 6)), rng.normal(size=(9, 6))
    loss, _, _, dhs, dws, dht, dwt = O.jsd_linear(h, w, h, w, 0.5, rng.normal(size=4))
    assert np.all(np.abs(loss) < 1e-15)
    for d in (dhs, dws, dht, dwt):
        assert np.all(np.abs(d) < 1e-14)


def pin_cross_entropy():
    """Cross-entropy: ln V on equal logits; -log_softmax(x / T) at the label
    from SciPy; 0 and no gradient at ignore_index; central differences."""
    rng = np.random.default_rng(34)
    x = rng.normal(0, 2, (5, 11))
    x[1, 3] = -np.inf
    labels = np.array([2, 4, -100, 10, 0])
    for temp in (1.0, 1.7):
        loss, dx, errs = O.cross_entropy(x, labels, -100, temp)
        assert errs == 0
        ref = -special.log_softmax(x / temp, axis=1)[np.arange(5), np.where(labels < 0, 0, labels)]
        ref[2] = 0.0
        _close(loss, ref, 1e-13, 1e-15, f"ce T={temp}")
        assert np.all(dx[2] == 0.0)
        g = rng.normal(size=5)
        _, dxg, _ = O.cross_entropy(x, labels, -100, temp, g)
        _fd_check(lambda y: float(np.dot(g, O.cross_entropy(y, labels, -100, temp, grad=False)[0])), x, dxg,
                  f"ce fd T={temp}")
    flat = np.zeros((2, 13))
    _close(O.cross_entropy(flat, [0, 12])[0], [math.log(13)] * 2, 1e-15, 0, "ce uniform")


def pin_topk_kl_full_vocabulary():
    """With every id selected (k = V) and the teacher's full log-softmax, the
    top-k forward KL is the full forward KL(P_t || P_s), value and student
    gradient, from the KL row oracle."""
    rng = np.random.default_rng(35)
    s = rng.normal(0, 2, (4, 9))
    t = rng.normal(0, 2, (4, 9))
    g = rng.normal(size=4)
    ids = np.tile(np.arange(9), (4, 1))
    tl = special.log_softmax(t, axis=1)
    kl, ds, errs = O.topk_forward_kl(s, ids, tl, -100, 1.0, g)
    assert errs == 0
    ref, rds, _ = O.kl(s, t, False, g)
    _close(kl, ref, 1e-12, 1e-14, "top-k = full KL")
    _close(ds, rds, 1e-11, 1e-14, "top-k = full KL, student gradient")


def pin_topk_kl_finite_differences_and_classes():
    """Central differences of the top-k forward KL (temperature 1.5, an ignored
    position, a duplicate id); +inf with zero gradient when the student masks
    an id the teacher gives mass."""
    rng = np.random.default_rng(36)
    s = rng.normal(0, 2, (3, 8))
    ids = np.array([[1, 5, 5], [0, -100, 7], [2, 3, 4]])
    tl = np.log(np.array([[0.5, 0.2, 0.1], [0.4, 0.3, 0.2], [0.6, 0.2, 0.1]]))
    g = rng.normal(size=3)
    _, ds, _ = O.topk_forward_kl(s, ids, tl, -100, 1.5, g)
    _fd_check(lambda y: float(np.dot(g, O.topk_forward_kl(y, ids, tl, -100, 1.5, grad=False)[0])), s, ds,
              "top-k kl fd")
    sm = s.copy()
    sm[2, 3] = -np.inf
    kl, dsm, _ = O.topk_forward_kl(sm, ids, tl, -100, 1.0, g)
    assert np.isposinf(kl[2]) and np.all(dsm[2] == 0.0) and np.all(np.isfinite(kl[:2]))


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
