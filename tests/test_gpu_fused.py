"""The single-read fused JSD forward+backward (thread-block clusters) against
the CPU oracle, on shapes that take the fused path (16-bit inputs, V a
multiple of 8, 16-byte aligned rows). Each call is checked to have issued
exactly one kernel launch, so a silent fallback to the streaming kernels
would fail the test."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity_util import assert_grad, assert_loss, assert_zero_rows, kl_branch_floor, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from softmax_divergence_lm_gb300 import build
    build.build()
    from softmax_divergence_lm_gb300 import binding
    binding.load()
    return binding


def make_rows(n, v, dtype, seed=1):
    g = torch.Generator(device="cpu").manual_seed(seed)
    s = torch.randn(n, v, generator=g) * 4
    s[6, v // 3] += 30.0                   # a peaked row (the teacher follows it, as in the workloads)
    t = s + torch.randn(n, v, generator=g) * 2
    s[0, 3:50] = -math.inf                 # student-masked tokens
    t[1, v - 40:] = -math.inf              # teacher-masked tail
    s[2], t[2] = -math.inf, -math.inf      # fully masked row
    t[3] = -math.inf                       # teacher fully masked
    s[4, 11] = math.nan                    # out of contract
    t[5, 0] = math.inf                     # out of contract
    t[7, :] = 0.5                          # uniform teacher
    s[8, :] = -math.inf                    # student with a single token
    s[8, v - 1] = 2.0
    return s.to(dtype).cuda(), t.to(dtype).cuda()


def off_grid(x):
    """The same rows with a row stride of V + 1 elements: rows that do not all
    start on a 16-byte boundary, which the single-read kernels do not take."""
    n, v = x.shape
    y = torch.empty(n, v + 1, dtype=x.dtype, device=x.device)
    y[:, :v].copy_(x)
    return y[:, :v]


def fused_call(B, s, t, beta, g, gdtype, want_s=True, want_t=True):
    n = s.shape[0] if s.dim() == 2 else s.shape[0] * s.shape[1]
    v = s.shape[-1]
    loss = torch.full((n,), 7.0, device="cuda")
    saved = torch.full((n, 6), 7.0, device="cuda")
    ds = torch.full((n, v), 3.0, dtype=gdtype, device="cuda") if want_s else None
    dt = torch.full((n, v), 3.0, dtype=gdtype, device="cuda") if want_t else None
    c0 = B.vpd_launch_count()
    B.vpd_jsd_fwdbwd(s, t, beta, None, g, loss, saved, ds, dt)
    torch.cuda.synchronize()
    B.vpd_device_status()  # raises if a bounded device-side wait gave up
    launches = B.vpd_launch_count() - c0
    return loss, saved, ds, dt, launches


def check(B, s, t, beta, gdtype, want_s=True, want_t=True, rows=None, label="", launches=(1,)):
    s2 = s if s.dim() == 2 else s.reshape(-1, s.shape[-1])
    t2 = t if t.dim() == 2 else t.reshape(-1, t.shape[-1])
    n = s2.shape[0]
    gen = torch.Generator(device="cpu").manual_seed(2)
    g = torch.randn(n, generator=gen).cuda()
    loss, saved, ds, dt, k = fused_call(B, s, t, beta, g, gdtype, want_s, want_t)
    assert k in launches, f"{label}: expected {launches} launches (the fused kernel), saw {k}"
    rows = np.arange(n) if rows is None else np.asarray(rows)
    r = torch.as_tensor(rows, device="cuda")
    s64, t64 = to64(s2[r]), to64(t2[r])
    rl, _, _, rds, rdt = O.jsd(s64, t64, beta, to64(g)[rows], threads=8)
    tag = f"{label} beta={beta} {s.dtype}->{gdtype}"
    assert_loss(to64(loss)[rows], rl, tag + " loss")
    gd = None if gdtype == torch.float32 else gdtype
    bad = np.nonzero(~np.isfinite(rl))[0]
    fs, ft = kl_branch_floor(s64, t64, beta, to64(g)[rows])
    if want_s:
        got = to64(ds[r])
        assert_grad(got, rds, tag + " dS", gd, floor=fs)
        assert_zero_rows(got, bad, tag + " dS")
    if want_t:
        got = to64(dt[r])
        assert_grad(got, rdt, tag + " dT", gd, floor=ft)
        assert_zero_rows(got, bad, tag + " dT")
    # saved statistics agree with the oracle's (m, ln Z) of each input
    sv = to64(saved)[rows]
    for col, x in ((0, s2), (2, t2)):
        m, lse, code = O.row_stats(to64(x[r]))
        ok = code == 0
        assert np.array_equal(sv[ok, col], m[ok]), f"{tag}: saved max differs"
        assert np.allclose(sv[ok, col + 1], lse[ok], rtol=1e-5, atol=5e-6), f"{tag}: saved log-sum-exp differs"
    return loss


# cluster sizes 1, 2, 4, 8 and 16 are all exercised by these vocabulary sizes
@pytest.mark.parametrize("v", [1024, 5008, 19208, 40000, 100000, 151936, 262144])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_fused_matches_oracle(B, v, dtype):
    n = 24 if v <= 40000 else 12
    s, t = make_rows(n, v, dtype, seed=v % 97)
    for beta in (0.5, 0.1, 0.0, 1.0):
        check(B, s, t, beta, dtype, label=f"V={v}")
    check(B, s, t, 0.7, torch.float32, label=f"V={v}")
    check(B, s, t, 0.5, dtype, want_t=False, label=f"V={v} detached")
    check(B, s, t, 0.5, dtype, want_s=False, label=f"V={v} teacher only")


# The forward-only kernel (no gradient wanted): statistics two rows ahead of
# pass C on three stages; same shapes as above, every beta branch.
@pytest.mark.parametrize("v", [1024, 5008, 19208, 40000, 100000, 151936, 262144])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_fused_forward_kernel_matches_oracle(B, v, dtype):
    n = 24 if v <= 40000 else 12
    s, t = make_rows(n, v, dtype, seed=v % 89 + 1)
    for beta in (0.5, 0.1, 0.0, 1.0):
        loss, saved, _, _, launches = fused_call(B, s, t, beta, None, dtype, want_s=False, want_t=False)
        assert launches == 1, f"V={v}: expected the single forward launch, saw {launches}"
        rl, ra, rb, _, _ = O.jsd(to64(s), to64(t), beta, grad=False, threads=8)
        tag = f"forward V={v} beta={beta} {dtype}"
        assert_loss(to64(loss), rl, tag + " loss")
        sv = to64(saved)
        for col, x in ((0, s), (2, t)):
            m, lse, code = O.row_stats(to64(x))
            ok = code == 0
            assert np.array_equal(sv[ok, col], m[ok]), f"{tag}: saved max differs"
            assert np.allclose(sv[ok, col + 1], lse[ok], rtol=1e-5, atol=5e-6), f"{tag}: saved log-sum-exp differs"
        if 0.0 < beta < 1.0:
            live = np.isfinite(rl)
            assert_loss(sv[live, 4], ra[live], tag + " saved KL(P_t||M)")
            assert_loss(sv[live, 5], rb[live], tag + " saved KL(P_s||M)")


def test_fused_forward_kernel_many_rows(B):
    """More rows than resident clusters through a [B, T-1, V] causal view: the
    three stages and the cluster slot rings wrap many times."""
    g = torch.Generator(device="cpu").manual_seed(6)
    base_s = (torch.randn(3, 401, 4096, generator=g) * 3).to(torch.bfloat16).cuda()
    base_t = (torch.randn(3, 401, 4096, generator=g) * 3).to(torch.bfloat16).cuda()
    s, t = base_s[:, :-1], base_t[:, :-1]
    loss, _, _, _, launches = fused_call(B, s, t, 0.3, None, torch.bfloat16, want_s=False, want_t=False)
    assert launches == 1
    rl = O.jsd(to64(s.reshape(-1, 4096)), to64(t.reshape(-1, 4096)), 0.3, grad=False, threads=8)[0]
    assert_loss(to64(loss), rl, "forward kernel, causal view")


def test_fused_forward_only_and_classes(B):
    s, t = make_rows(16, 8192, torch.bfloat16)
    loss, _, _, _, launches = fused_call(B, s, t, 0.5, None, torch.bfloat16, want_s=False, want_t=False)
    assert launches == 1
    lo = to64(loss)
    assert np.all(np.isnan(lo[2:6])) and np.all(np.isfinite(lo[[0, 1, 6, 7, 8]]))
    fwd = check(B, s, t, 0.0, torch.bfloat16, label="classes")
    assert np.isposinf(to64(fwd)[0]) and np.isposinf(to64(fwd)[8])


def test_fused_causal_view_and_many_rows(B):
    """More rows than resident clusters (every cluster loops over rows and
    reuses both shared-memory stages), through a [B, T-1, V] causal view."""
    g = torch.Generator(device="cpu").manual_seed(5)
    base_s = (torch.randn(3, 401, 4096, generator=g) * 3).to(torch.bfloat16).cuda()
    base_t = (torch.randn(3, 401, 4096, generator=g) * 3).to(torch.bfloat16).cuda()
    rows = np.unique(np.concatenate([np.arange(0, 1200, 7), [1199]]))
    check(B, base_s[:, :-1], base_t[:, :-1], 0.5, torch.bfloat16, rows=rows, label="causal")


def test_fused_many_rows_at_cluster_width(B):
    """Many rows per cluster at the Qwen vocabulary (clusters of 9 CTAs, 19
    workers x R = 4): every stage and cluster slot ring wraps many times.
    With this many rows the last ones go to the SMs the clusters leave idle
    (three streaming launches on a side stream), so the call makes one fused
    launch plus those three."""
    s, t = make_rows(240, 151936, torch.bfloat16, seed=13)
    rows = np.arange(0, 240, 7)
    check(B, s, t, 0.5, torch.bfloat16, rows=rows, label="240 rows", launches=(1, 4))


@pytest.mark.parametrize("gdtype", [torch.bfloat16, torch.float32])
def test_idle_sm_split_every_row(B, gdtype):
    """1000 rows at the Qwen vocabulary: the fused launch takes the first rows,
    the streaming kernels on the idle SMs the last ones; every row of both
    parts (and the boundary between them) against the oracle."""
    s, t = make_rows(1000, 151936, torch.bfloat16, seed=23)
    check(B, s, t, 0.5, gdtype, label="idle-SM split", launches=(4,))
    check(B, s, t, 0.0, gdtype, want_t=False, label="idle-SM split, forward KL, detached", launches=(4,))
    n = s.shape[0]
    loss = torch.empty(n, device="cuda")
    saved = torch.empty(n, 6, device="cuda")
    k = launches_of(B, lambda: B.vpd_jsd_fwd(s, t, 0.5, None, loss, saved))
    assert k == 3, f"forward with the idle-SM split: {k} launches"
    rl, ra, rb, _, _ = O.jsd(to64(s), to64(t), 0.5, grad=False, threads=8)
    assert_loss(to64(loss), rl, "idle-SM split forward loss")
    live = np.isfinite(rl)
    assert_loss(to64(saved)[live, 4], ra[live], "idle-SM split forward saved A")
    assert_loss(to64(saved)[live, 5], rb[live], "idle-SM split forward saved B")


def test_idle_sm_split_causal_view(B):
    """A [3, 401, V] causal-shift view at the Qwen vocabulary (1200 rows): the
    idle-SM split starts its side rows in the middle of a batch; every row of
    both parts against the oracle, forward+backward and forward only."""
    g = torch.Generator(device="cpu").manual_seed(29)
    base_s = (torch.randn(3, 401, 151936, generator=g) * 4).to(torch.bfloat16).cuda()
    base_t = (base_s.float().cpu() + torch.randn(3, 401, 151936, generator=g) * 2).to(torch.bfloat16).cuda()
    s, t = base_s[:, :-1], base_t[:, :-1]
    fused_rows, side_rows, _ = B.vpd_jsd_plan(s, t, None, torch.empty(1200, 151936, dtype=torch.bfloat16,
                                                                       device="cuda"), None)
    assert side_rows > 0 and fused_rows % 400 != 0, (fused_rows, side_rows)
    check(B, s, t, 0.5, torch.bfloat16, label="idle-SM split, causal view", launches=(4,))
    loss = torch.empty(1200, device="cuda")
    saved = torch.empty(1200, 6, device="cuda")
    k = launches_of(B, lambda: B.vpd_jsd_fwd(s, t, 0.5, None, loss, saved))
    assert k == 3, f"causal forward with the idle-SM split: {k} launches"
    rl = O.jsd(to64(s.reshape(-1, 151936)), to64(t.reshape(-1, 151936)), 0.5, grad=False, threads=8)[0]
    assert_loss(to64(loss), rl, "idle-SM split causal forward loss")


def test_forward_kernel_many_rows_at_cluster_width(B):
    """The forward-only kernel on 240 rows at the Qwen vocabulary (clusters of
    9 CTAs, 23 workers x R = 3): its stages and slot rings wrap many times."""
    s, t = make_rows(240, 151936, torch.bfloat16, seed=17)
    for beta in (0.5, 1.0):
        loss, saved, _, _, launches = fused_call(B, s, t, beta, None, torch.bfloat16, want_s=False, want_t=False)
        assert launches in (1, 3)  # plus the two streaming passes on the idle SMs
        rl, ra, rb, _, _ = O.jsd(to64(s), to64(t), beta, grad=False, threads=8)
        assert_loss(to64(loss), rl, f"forward 240 rows beta={beta}")
        if beta == 0.5:
            live = np.isfinite(rl)
            assert_loss(to64(saved)[live, 4], ra[live], "forward 240 rows saved KL(P_t||M)")


@pytest.mark.parametrize("beta", [0.5, 0.0, 1.0, 0.3])
def test_fp32_single_read(B, beta):
    """fp32 logits on the single-read kernels (32-byte vectors of 8 floats):
    every special row class, fwd+bwd in one launch, the forward-only kernel,
    and a segmented call (the same MAX / SUM merge over the CTA slices)."""
    s, t = make_rows(40, 8192, torch.float32, seed=31)
    check(B, s, t, beta, torch.float32, label="fp32 single-read", launches=(1,))
    n, v = s.shape
    rl, ra, rb, _, _ = O.jsd(to64(s), to64(t), beta, grad=False, threads=8)
    for seg in (None, [3000, 0, 5192]):
        loss = torch.full((n,), 7.0, device="cuda")
        saved = torch.full((n, 6), 7.0, device="cuda")
        k = launches_of(B, lambda: B.vpd_jsd_fwd(s, t, beta, seg, loss, saved))
        assert k == 1, f"fp32 forward, segments {seg}: {k} launches"
        assert_loss(to64(loss), rl, f"fp32 forward beta={beta} segments {seg}")
        live = np.isfinite(rl)
        sv = to64(saved)
        if beta not in (0.0, 1.0):
            assert_loss(sv[live, 4], ra[live], f"fp32 forward saved A, segments {seg}")
            assert_loss(sv[live, 5], rb[live], f"fp32 forward saved B, segments {seg}")


def test_fp32_single_read_wide_rows_and_split(B):
    """fp32 rows at V = 128256 in 8 uneven segments (the edge-case workload's
    shape) with a common offset of 1e4: clusters of 10 or more CTAs, the last
    rows on the idle SMs; every row against the oracle."""
    from softmax_divergence_lm_gb300 import synth
    v = 128256
    g = torch.Generator(device="cpu").manual_seed(37)
    s = torch.randn(600, v, generator=g) * 3 + 1.0e4
    t = torch.randn(600, v, generator=g) * 3 + 1.0e4
    s[torch.rand(600, v, generator=g) < 0.1] = -math.inf
    s, t = s.cuda(), t.cuda()
    seg = synth.segment_widths(37, v)
    n = s.shape[0]
    gr = torch.randn(n, generator=g).cuda()
    loss = torch.empty(n, device="cuda")
    saved = torch.empty(n, 6, device="cuda")
    ds = torch.empty(n, v, device="cuda")
    dt = torch.empty(n, v, device="cuda")
    fused_rows, side_rows, planned = B.vpd_jsd_plan(s, t, seg, ds, dt)
    assert fused_rows > 0 and planned in (1, 4)
    k = launches_of(B, lambda: B.vpd_jsd_fwdbwd(s, t, 0.5, seg, gr, loss, saved, ds, dt))
    assert k == planned, f"{k} launches, planned {planned}"
    B.vpd_device_status()
    rows = np.arange(0, n, 9)
    rows = np.unique(np.concatenate([rows, [n - 1, fused_rows - 1, min(fused_rows, n - 1)]]))
    r = torch.as_tensor(rows, device="cuda")
    rl, _, _, rds, rdt = O.jsd(to64(s[r]), to64(t[r]), 0.5, to64(gr)[rows], threads=8)
    assert_loss(to64(loss)[rows], rl, "fp32 wide rows loss")
    assert_grad(to64(ds[r]), rds, "fp32 wide rows dS")
    assert_grad(to64(dt[r]), rdt, "fp32 wide rows dT")


def test_fused_equals_streaming_path(B):
    """The fused single-read call and the two-pass forward + backward agree."""
    s, t = make_rows(32, 151936, torch.bfloat16, seed=7)
    n, v = s.shape
    g = torch.rand(n, device="cuda")
    f_loss, f_saved, f_ds, f_dt, _ = fused_call(B, s, t, 0.5, g, torch.float32)
    loss = torch.empty(n, device="cuda")
    saved = torch.empty(n, 6, device="cuda")
    ds = torch.empty(n, v, device="cuda")
    dt = torch.empty(n, v, device="cuda")
    B.vpd_jsd_fwd(s, t, 0.5, None, loss, saved)
    B.vpd_jsd_bwd(s, t, 0.5, None, g, saved, ds, dt)
    torch.cuda.synchronize()
    assert_loss(to64(f_loss), to64(loss), "fused vs streaming loss")
    assert_grad(to64(f_ds), to64(ds), "fused vs streaming dS")
    assert_grad(to64(f_dt), to64(dt), "fused vs streaming dT")


def test_one_hot_against_broad_fp32_floor_every_path(B):
    """A near one-hot student against a broad teacher at the KL branches: the
    gradient at the peak is a small difference of two log-ratios of tens of
    nats, so fp32 (the saved KL itself is an fp32 number) cannot resolve it to
    the stated absolute tolerance. Every path gets the same allowance, the
    rounding floor of `parity_util.kl_branch_floor`, on top of the stated
    tolerance: the single-read kernel (one and two segments), the streaming
    kernels (rows off the 16-byte grid), and the KL forward + backward in both
    directions; the loss and every other
    gradient meet the stated tolerance."""
    v = 1024
    g0 = torch.Generator(device="cpu").manual_seed(11)
    s = torch.randn(4, v, generator=g0) * 4
    t = s + torch.randn(4, v, generator=g0) * 2
    s[:, 341] += 30.0  # peaked student, broad teacher
    s, t = s.to(torch.bfloat16).cuda(), t.to(torch.bfloat16).cuda()
    g = torch.randn(4, generator=g0).cuda()
    s64, t64, g64 = to64(s), to64(t), to64(g)
    n = s.shape[0]
    for beta in (1.0, 0.0):
        rl, _, _, rds, rdt = O.jsd(s64, t64, beta, g64, threads=4)
        fs, ft = kl_branch_floor(s64, t64, beta, g64)
        runs = {}
        loss, _, ds, dt, launches = fused_call(B, s, t, beta, g, torch.float32)
        assert launches == 1
        runs["single-read"] = (loss, ds, dt)
        # rows off the 16-byte grid (a row stride of V + 1) take the streaming
        # kernels; a two-segment table keeps the single-read kernel
        for label, (xs, xt, seg, k_want) in (("streaming", (off_grid(s), off_grid(t), None, 3)),
                                             ("single-read, two segments", (s, t, [v // 2, v - v // 2], 1))):
            l2 = torch.empty(n, device="cuda")
            sv = torch.empty(n, 6, device="cuda")
            d1 = torch.empty(n, v, device="cuda")
            d2 = torch.empty(n, v, device="cuda")
            k = launches_of(B, lambda: B.vpd_jsd_fwdbwd(xs, xt, beta, seg, g, l2, sv, d1, d2))
            assert k == k_want, f"{label}: {k} launches"
            runs[label] = (l2, d1, d2)
        l3 = torch.empty(n, device="cuda")
        sv = torch.empty(n, 6, device="cuda")
        d1 = torch.empty(n, v, device="cuda")
        d2 = torch.empty(n, v, device="cuda")
        B.vpd_kl_fwd(s, t, beta == 1.0, None, l3, sv)
        B.vpd_kl_bwd(s, t, beta == 1.0, None, g, sv, d1, d2)
        runs["KL op"] = (l3, d1, d2)
        torch.cuda.synchronize()
        for label, (lo, d1, d2) in runs.items():
            tag = f"one-hot beta={beta} {label}"
            assert_loss(to64(lo), rl, tag + " loss")
            assert_grad(to64(d1), rds, tag + " dS", floor=fs)
            assert_grad(to64(d2), rdt, tag + " dT", floor=ft)


def launches_of(B, fn):
    c0 = B.vpd_launch_count()
    fn()
    torch.cuda.synchronize()
    B.vpd_device_status()
    return B.vpd_launch_count() - c0


@pytest.mark.parametrize("v", [8, 16, 24])
def test_fused_tiny_vocabularies(B, v):
    """A slice of one vector per CTA, most lanes of the single worker warp
    past the slice end."""
    g = torch.Generator(device="cpu").manual_seed(v)
    s = (torch.randn(40, v, generator=g) * 3).to(torch.bfloat16).cuda()
    t = (torch.randn(40, v, generator=g) * 3).to(torch.bfloat16).cuda()
    for beta in (0.5, 0.0, 1.0):
        check(B, s, t, beta, torch.bfloat16, label=f"V={v}")


def test_fused_size_limit(B):
    """The widest row the single-read kernel takes (16 CTAs x 19 warps x 32
    threads x 4 vectors x 8 = 311296 columns) runs as one launch; one vector
    more falls back to the two streaming passes and the backward."""
    for v, fused in ((311296, True), (311304, False)):
        g = torch.Generator(device="cpu").manual_seed(v % 1000)
        s0 = torch.randn(6, v, generator=g) * 4
        s = s0.to(torch.bfloat16).cuda()
        t = (s0 + torch.randn(6, v, generator=g) * 2).to(torch.bfloat16).cuda()
        n = s.shape[0]
        gr = torch.rand(n, device="cuda")
        loss = torch.empty(n, device="cuda")
        saved = torch.empty(n, 6, device="cuda")
        ds = torch.empty(n, v, dtype=torch.bfloat16, device="cuda")
        dt = torch.empty_like(ds)
        k = launches_of(B, lambda: B.vpd_jsd_fwdbwd(s, t, 0.5, None, gr, loss, saved, ds, dt))
        assert (k == 1) == fused, f"V={v}: {k} launches"
        rl, _, _, rds, rdt = O.jsd(to64(s), to64(t), 0.5, to64(gr), threads=8)
        assert_loss(to64(loss), rl, f"V={v} loss")
        assert_grad(to64(ds), rds, f"V={v} dS", torch.bfloat16)
        assert_grad(to64(dt), rdt, f"V={v} dT", torch.bfloat16)


@pytest.mark.parametrize("v", [8, 16, 24])
def test_forward_kernel_tiny_vocabularies(B, v):
    """The forward-only kernel with one vector per CTA slice: most lanes of
    its single worker warp are past the slice end."""
    g = torch.Generator(device="cpu").manual_seed(v + 100)
    s = (torch.randn(40, v, generator=g) * 3).to(torch.bfloat16).cuda()
    t = (torch.randn(40, v, generator=g) * 3).to(torch.bfloat16).cuda()
    for beta in (0.5, 0.0, 1.0):
        loss, _, _, _, launches = fused_call(B, s, t, beta, None, torch.bfloat16, want_s=False, want_t=False)
        assert launches == 1
        rl = O.jsd(to64(s), to64(t), beta, grad=False, threads=4)[0]
        assert_loss(to64(loss), rl, f"forward V={v} beta={beta}")


def test_forward_size_limit(B):
    """vpd_jsd_fwd: the widest row the forward-only kernel takes in clusters of
    at most 10 CTAs (three stages of 4 x 19104 bytes plus the tail fill the
    232448 bytes of shared memory a CTA can have) is one launch; one vector
    more takes the two streaming passes."""
    for v, fused in ((191040, True), (191048, False)):
        g = torch.Generator(device="cpu").manual_seed(v % 1000)
        s0 = torch.randn(6, v, generator=g) * 4
        s = s0.to(torch.bfloat16).cuda()
        t = (s0 + torch.randn(6, v, generator=g) * 2).to(torch.bfloat16).cuda()
        n = s.shape[0]
        loss = torch.empty(n, device="cuda")
        saved = torch.empty(n, 6, device="cuda")
        k = launches_of(B, lambda: B.vpd_jsd_fwd(s, t, 0.5, None, loss, saved))
        assert (k == 1) == fused, f"V={v}: {k} launches"
        rl = O.jsd(to64(s), to64(t), 0.5, grad=False, threads=8)[0]
        assert_loss(to64(loss), rl, f"V={v} forward loss")


@pytest.mark.parametrize("v", [16032, 151936])
def test_forward_calls_through_single_read(B, v):
    """vpd_jsd_fwd takes the single-read forward kernel (one launch) at both
    vocabularies and matches the oracle's loss and saved statistics;
    vpd_kl_fwd matches the oracle's KL on either of its paths."""
    s, t = make_rows(12, v, torch.bfloat16, seed=v % 89)
    n = s.shape[0]
    loss = torch.empty(n, device="cuda")
    saved = torch.empty(n, 6, device="cuda")
    k = launches_of(B, lambda: B.vpd_jsd_fwd(s, t, 0.5, None, loss, saved))
    assert k == 1, f"V={v}: the JSD forward took {k} launches"
    rl, _, _, _, _ = O.jsd(to64(s), to64(t), 0.5, None, grad=False, threads=8)
    assert_loss(to64(loss), rl, f"V={v} forward loss")
    sv = to64(saved)
    for col, x in ((0, s), (2, t)):
        m, lse, code = O.row_stats(to64(x))
        ok = code == 0
        assert np.array_equal(sv[ok, col], m[ok])
        assert np.allclose(sv[ok, col + 1], lse[ok], rtol=1e-5, atol=5e-6)
    for rev in (0, 1):
        kl = torch.empty(n, device="cuda")
        B.vpd_kl_fwd(s, t, rev, None, kl, None)
        torch.cuda.synchronize()
        rk, _, _, _, _ = O.jsd(to64(s), to64(t), float(rev), None, grad=False, threads=8)
        assert_loss(to64(kl), rk, f"V={v} KL reverse={rev}")


def test_bf16_row_max_above_2_126(B):
    """A bf16 row whose largest finite logit exceeds 2^126 is out of contract
    on the single-read kernels and the online KL kernel: NaN with zero
    gradients (the limit keeps every clamped log-difference finite). The streaming kernels, reached here through
    rows off the 16-byte grid, and the oracle give the finite value. At beta = 0 the
    teacher gradient of such a row is a difference of two log-ratios near
    2^127 that fp32 cannot resolve (the same floor as for near one-hot rows),
    so there only the loss and the student gradient of those rows are
    compared."""
    v = 4096
    g0 = torch.Generator(device="cpu").manual_seed(21)
    s = torch.randn(4, v, generator=g0) * 3
    t = s + torch.randn(4, v, generator=g0)
    s[0, 5] = 2.0**127
    t[1, 9] = 2.0**127
    s, t = s.to(torch.bfloat16).cuda(), t.to(torch.bfloat16).cuda()
    g = torch.ones(4, device="cuda")
    for beta in (0.5, 0.0):
        loss, _, ds, dt, launches = fused_call(B, s, t, beta, g, torch.float32)
        assert launches == 1
        lo = to64(loss)
        assert np.all(np.isnan(lo[:2])) and np.all(np.isfinite(lo[2:]))
        assert_zero_rows(to64(ds), [0, 1], "2^127 row dS")
        assert_zero_rows(to64(dt), [0, 1], "2^127 row dT")
        rl, _, _, rds, rdt = O.jsd(to64(s), to64(t), beta, to64(g), threads=4)
        assert_loss(lo[2:], rl[2:], f"beta={beta} in-contract rows")
        fwd = torch.empty(4, device="cuda")
        k = launches_of(B, lambda: B.vpd_jsd_fwd(s, t, beta, None, fwd, torch.empty(4, 6, device="cuda")))
        # beta = 0.5: the forward-only cluster kernel; beta = 0: the online KL
        # kernel, where such rows are out of contract too
        assert k == 1 and np.all(np.isnan(to64(fwd)[:2]))
        assert_loss(to64(fwd)[2:], rl[2:], f"beta={beta} forward in-contract rows")
        # rows off the 16-byte grid: the streaming kernels, finite and equal to the oracle
        ls = torch.empty(4, device="cuda")
        sv = torch.empty(4, 6, device="cuda")
        ds2 = torch.empty(4, v, device="cuda")
        dt2 = torch.empty(4, v, device="cuda")
        k = launches_of(B, lambda: B.vpd_jsd_fwdbwd(off_grid(s), off_grid(t), beta, None, g, ls, sv, ds2, dt2))
        assert k == 3, f"off-grid rows: {k} launches"
        assert_loss(to64(ls), rl, f"beta={beta} streaming loss")
        assert_grad(to64(ds2), rds, f"beta={beta} streaming dS")
        keep = slice(None) if beta > 0.0 else slice(2, None)
        assert_grad(to64(dt2)[keep], rdt[keep], f"beta={beta} streaming dT")


def test_forward_16_cta_clusters_with_idle_split(B):
    """At V = 262144 the forward-only kernel needs clusters of 16 CTAs (112
    SMs); with enough rows the 40 idle SMs take a share on the streaming passes
    and the call takes that path (one fused launch plus two streaming ones):
    every row against the oracle, and the plan query agrees."""
    v = 262144
    g = torch.Generator(device="cpu").manual_seed(41)
    s0 = torch.randn(400, v, generator=g) * 4
    s = s0.to(torch.bfloat16).cuda()
    t = (s0 + torch.randn(400, v, generator=g) * 1.5).to(torch.bfloat16).cuda()
    n = s.shape[0]
    fused_rows, side_rows, planned = B.vpd_jsd_plan(s, t)
    loss = torch.empty(n, device="cuda")
    saved = torch.empty(n, 6, device="cuda")
    k = launches_of(B, lambda: B.vpd_jsd_fwd(s, t, 0.5, None, loss, saved))
    assert k == planned
    if side_rows:
        assert k == 3 and fused_rows + side_rows == n
    rl, ra, rb, _, _ = O.jsd(to64(s), to64(t), 0.5, grad=False, threads=8)
    assert_loss(to64(loss), rl, "V=262144 forward loss")
    assert_loss(to64(saved)[:, 4], ra, "V=262144 forward saved A")
    assert_loss(to64(saved)[:, 5], rb, "V=262144 forward saved B")
