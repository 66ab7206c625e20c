"""CUDA kernels (through the C ABI) against the CPU oracle, element by element.

Small cases run every row through the oracle at sizes that span several
vector tiles per thread and a ragged tail; the five full-size workloads
compare sampled rows (all special rows included) with the oracle, in the same
launch configuration the benchmark uses.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity_util import assert_grad, assert_loss, assert_zero_rows, kl_branch_floor, to64

pytestmark = pytest.mark.gpu

BETAS = (0.5, 0.0, 1.0, 0.25, 0.9)


@pytest.fixture(scope="module")
def B():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from softmax_divergence_lm_gb300 import build
    build.build()
    from softmax_divergence_lm_gb300 import binding
    binding.load()
    return binding


def _rows2d(x: torch.Tensor) -> torch.Tensor:
    return x if x.dim() == 2 else x.reshape(-1, x.shape[-1])


# ---------------------------------------------------------------------------
# Runners
# ---------------------------------------------------------------------------
def gpu_pair(B, s, t, beta, *, op="jsd", segments=None, g=None, gdtype=torch.float32, want_s=True,
             want_t=True, fused=False):
    """Run a pair op (jsd / kl-fwd / kl-rev) forward + backward on the GPU."""
    n = _rows2d(s).shape[0]
    v = s.shape[-1]
    dev = s.device
    loss = torch.full((n,), 7.0, device=dev)
    saved = torch.full((n, 6), 7.0, device=dev)
    ds = torch.full((n, v), 3.0, dtype=gdtype, device=dev) if want_s else None
    dt = torch.full((n, v), 3.0, dtype=gdtype, device=dev) if want_t else None
    if op == "jsd" and fused:
        B.vpd_jsd_fwdbwd(s, t, beta, segments, g, loss, saved, ds, dt)
    elif op == "jsd":
        B.vpd_jsd_fwd(s, t, beta, segments, loss, saved)
        B.vpd_jsd_bwd(s, t, beta, segments, g, saved, ds, dt)
    else:
        rev = op == "kl-rev"
        B.vpd_kl_fwd(s, t, rev, segments, loss, saved)
        B.vpd_kl_bwd(s, t, rev, segments, g, saved, ds, dt)
    torch.cuda.synchronize()
    return loss, saved, ds, dt


def _host_rows(x, rows):
    if x is None:
        return None
    if rows is None:
        return to64(x)
    return to64(x[torch.as_tensor(rows, device=x.device)])


def oracle_pair(s64, t64, beta, op="jsd", g=None):
    if op == "jsd":
        loss, a, b, ds, dt = O.jsd(s64, t64, beta, g, threads=8)
        return loss, ds, dt
    return O.kl(s64, t64, op == "kl-rev", g, threads=8)


def check_pair(B, s, t, beta, *, op="jsd", segments=None, rows=None, gdtype=torch.float32, want_s=True,
               want_t=True, fused=False, label=""):
    n = _rows2d(s).shape[0]
    gen = torch.Generator(device="cpu").manual_seed(5)
    g = torch.randn(n, generator=gen).to(s.device)
    loss_d, saved_d, ds_d, dt_d = gpu_pair(B, s, t, beta, op=op, segments=segments, g=g, gdtype=gdtype,
                                           want_s=want_s, want_t=want_t, fused=fused)
    rows = np.arange(n) if rows is None else np.asarray(rows)
    loss, saved = to64(loss_d), to64(saved_d)
    ds, dt = _host_rows(ds_d, rows), _host_rows(dt_d, rows)
    del ds_d, dt_d
    s64 = _host_rows(_rows2d(s), rows)
    t64 = _host_rows(_rows2d(t), rows)
    rl, rds, rdt = oracle_pair(s64, t64, beta, op, to64(g)[rows])
    tag = f"{label} {op} beta={beta} {s.dtype}->{gdtype}"
    assert_loss(loss[rows], rl, tag + " loss")
    gd = None if gdtype == torch.float32 else gdtype
    branch = {"kl-fwd": 0.0, "kl-rev": 1.0}.get(op, beta)
    fs, ft = kl_branch_floor(s64, t64, branch, to64(g)[rows])
    if want_s:
        assert_grad(ds, rds, tag + " dS", gd, floor=fs)
    if want_t:
        assert_grad(dt, rdt, tag + " dT", gd, floor=ft)
    bad = np.nonzero(~np.isfinite(rl))[0]
    if want_s:
        assert_zero_rows(ds, bad, tag + " dS")
    if want_t:
        assert_zero_rows(dt, bad, tag + " dT")
    return loss, saved


def special_rows(n, v, seed=3, dtype=torch.float32, device="cuda"):
    """Random logits with masked tokens and every special row the contract names."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    s = torch.randn(n, v, generator=g) * 3
    t = 0.6 * s + torch.randn(n, v, generator=g) * 2
    s[0, 5:40] = -math.inf                  # masked tokens in the student
    t[1, 100:130] = -math.inf               # masked tokens in the teacher
    s[2], t[2] = -math.inf, -math.inf       # fully masked row (both)
    s[3] = -math.inf                        # fully masked student only
    t[4] = -math.inf                        # fully masked teacher only
    s[5, 7] = math.nan                      # outside the contract: NaN row
    t[6, 9] = math.inf                      # outside the contract: +inf row
    s[7, :] = -math.inf                     # student has one token, teacher many
    s[7, 3] = 1.0
    t[8, v // 2] = t[8].max() + 200.0       # a very peaked teacher
    s[9, v - 1] = -math.inf                 # masked last token (tail path)
    t[10, :] = t[10, 0]                     # uniform teacher
    s[11] = s[11] + 1.0e4                   # large common offset on one side
    return s.to(dtype).to(device), t.to(dtype).to(device)


# ---------------------------------------------------------------------------
# Small cases: every row through the oracle
# ---------------------------------------------------------------------------
def test_tiny_workload_all_ops(B):
    from softmax_divergence_lm_gb300 import synth
    s, t = synth.tiny(device="cuda")
    for beta in BETAS:
        check_pair(B, s, t, beta, label="tiny")
        check_pair(B, s, t, beta, fused=True, label="tiny fused")
    for op in ("kl-fwd", "kl-rev"):
        check_pair(B, s, t, None, op=op, label="tiny")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_ragged_special_rows(B, dtype):
    s, t = special_rows(67, 5003, dtype=dtype)
    for beta in (0.3, 0.0, 1.0):
        check_pair(B, s, t, beta, label="ragged")
        check_pair(B, s, t, beta, gdtype=dtype, label="ragged")
        check_pair(B, s, t, beta, fused=True, label="ragged")
    for op in ("kl-fwd", "kl-rev"):
        check_pair(B, s, t, None, op=op, label="ragged")
        check_pair(B, s, t, None, op=op, gdtype=dtype, label="ragged")


def test_special_row_classes(B):
    s, t = special_rows(67, 5003)
    loss, saved = check_pair(B, s, t, 0.5, label="classes")
    assert np.all(np.isnan(loss[2:7])), loss[:12]
    assert np.isfinite(loss[0]) and np.isfinite(loss[7]) and np.isfinite(loss[11])
    fwd, _ = check_pair(B, s, t, 0.0, label="classes")
    assert np.isposinf(fwd[0]) and np.isposinf(fwd[7])  # teacher mass on student-masked ids


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_segments(B, dtype):
    s, t = special_rows(40, 3001, seed=9, dtype=dtype)
    for widths in ([3001], [1000, 0, 2001], [7, 1, 0, 1500, 1493, 0], [0, 3001, 0]):
        for beta in (0.5, 0.0, 1.0):
            check_pair(B, s, t, beta, segments=widths, label=f"seg {widths}")
        check_pair(B, s, t, None, op="kl-fwd", segments=widths, label=f"seg {widths}")
    # a segment that is entirely -inf
    s2, t2 = s.clone(), t.clone()
    s2[:, 1000:2001] = -math.inf
    t2[:, 1000:2001] = -math.inf
    check_pair(B, s2, t2, 0.5, segments=[1000, 1001, 1000], label="masked segment")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_strided_and_causal_views(B, dtype):
    g = torch.Generator(device="cpu").manual_seed(4)
    v = 4099
    base_s = (torch.randn(3, 65, v + 5, generator=g) * 3).to(dtype).cuda()
    base_t = (torch.randn(3, 65, v + 5, generator=g) * 3).to(dtype).cuda()
    # row stride v + 5: every row starts at a different 16-byte phase
    s = base_s.view(-1, v + 5)[:, :v]
    t = base_t.view(-1, v + 5)[:, :v]
    check_pair(B, s, t, 0.5, label="strided")
    check_pair(B, s, t, 0.5, fused=True, label="strided")
    # causal-shift view [B, T-1, V] of a [B, T, V] buffer
    cs = base_s[:, :-1, :v]
    ct = base_t[:, :-1, :v]
    check_pair(B, cs, ct, 0.5, label="causal")
    check_pair(B, cs, ct, 1.0, gdtype=dtype, label="causal")
    # student and teacher at different 16-byte phases: element-wise path
    ct2 = base_t.view(-1, v + 5)[:, 1:v + 1]
    check_pair(B, s, ct2, 0.5, label="phase")
    check_pair(B, s, ct2, None, op="kl-rev", label="phase")


def test_entropy_and_logprobs_small(B):
    for dtype in (torch.float32, torch.bfloat16, torch.float16):
        x, _ = special_rows(67, 5003, seed=11, dtype=dtype)
        n, v = x.shape
        x64 = to64(x)
        gen = torch.Generator(device="cpu").manual_seed(6)
        g = torch.randn(n, generator=gen).cuda()
        out = torch.empty(n, device="cuda")
        saved = torch.empty(n, 3, device="cuda")
        for segs in (None, [2000, 0, 3003]):
            B.vpd_entropy_fwd(x, segs, out, saved)
            for gd in (torch.float32, dtype):
                dx = torch.full((n, v), 3.0, dtype=gd, device="cuda")
                B.vpd_entropy_bwd(x, segs, g, saved, dx)
                torch.cuda.synchronize()
                ro, rdx = O.entropy(x64, to64(g), threads=8)
                assert_loss(to64(out), ro, f"entropy {dtype}")
                assert_grad(to64(dx), rdx, f"entropy grad {dtype}->{gd}", None if gd == torch.float32 else gd)
        # logprobs: top-k ids with duplicates, ignore_index and masked tokens
        k = 5
        idx = torch.randint(0, v, (n, k), generator=gen)
        idx[:, 1] = idx[:, 0]
        idx[::3, 2] = -100
        idx[0, 3] = 7  # masked in row 0 of special_rows (s[0, 5:40])
        idx = idx.cuda()
        gk = torch.randn(n, k, generator=gen).cuda()
        out = torch.empty(n, k, device="cuda")
        saved = torch.empty(n, 2, device="cuda")
        err = torch.empty(1, dtype=torch.int32, device="cuda")
        B.vpd_logprobs_fwd(x, None, idx, k, -100, out, saved, err)
        dx = torch.full((n, v), 3.0, dtype=torch.float32, device="cuda")
        B.vpd_logprobs_bwd(x, None, idx, k, -100, gk, saved, dx)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ro, rdx, rerr = O.logprobs(x64, idx.cpu().numpy(), -100, to64(gk), threads=8)
        assert rerr == 0
        assert_loss(to64(out), ro, f"logprobs {dtype}")
        assert_grad(to64(dx), rdx, f"logprobs grad {dtype}")


def test_logprobs_out_of_range_sets_flag(B):
    x = torch.randn(4, 100, device="cuda")
    idx = torch.tensor([[1], [100], [-5], [-100]], device="cuda")
    out = torch.empty(4, 1, device="cuda")
    err = torch.empty(1, dtype=torch.int32, device="cuda")
    B.vpd_logprobs_fwd(x, None, idx, 1, -100, out, None, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    o = to64(out)
    assert np.isfinite(o[0, 0]) and np.isnan(o[1, 0]) and np.isnan(o[2, 0]) and o[3, 0] == 0.0


def test_logprobs_without_flag(B):
    """With no err_flag the indices are validated on the host: valid indices
    give the same outputs as the flagged call; a bad one is an error and
    nothing is written."""
    x = torch.randn(4, 100, device="cuda")
    idx = torch.tensor([[1, 7], [99, -100], [0, 5], [-100, 42]], device="cuda")
    out_f = torch.empty(4, 2, device="cuda")
    out_n = torch.empty(4, 2, device="cuda")
    err = torch.empty(1, dtype=torch.int32, device="cuda")
    B.vpd_logprobs_fwd(x, None, idx, 2, -100, out_f, None, err)
    B.vpd_logprobs_fwd(x, None, idx, 2, -100, out_n, None, None)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_f, out_n)
    bad = idx.clone()
    bad[2, 1] = 100
    out_b = torch.full((4, 2), 7.0, device="cuda")
    with pytest.raises(B.VpdError) as e:
        B.vpd_logprobs_fwd(x, None, bad, 2, -100, out_b, None, None)
    assert e.value.status == 4  # VPD_ERR_INDEX
    torch.cuda.synchronize()
    assert bool((out_b == 7.0).all()), "nothing is written when an index is rejected"


def test_degenerate_shapes(B):
    # N = 0: nothing to do, nothing written
    e = torch.empty(0, 10, device="cuda")
    B.vpd_jsd_fwd(e, e, 0.5, None, torch.empty(0, device="cuda"), torch.empty(0, 6, device="cuda"))
    # V = 0: no distribution, NaN rows
    z = torch.empty(3, 0, device="cuda")
    loss = torch.zeros(3, device="cuda")
    B.vpd_jsd_fwd(z, z, 0.5, None, loss, torch.empty(3, 6, device="cuda"))
    torch.cuda.synchronize()
    assert torch.isnan(loss).all()
    # V = 1: every divergence is 0, entropy 0, gradients 0
    one = torch.randn(5, 1, device="cuda")
    check_pair(B, one, one + 1.0, 0.5, label="V=1")
    out = torch.empty(5, device="cuda")
    B.vpd_entropy_fwd(one, None, out, None)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_row_partition_invariance(B):
    """A row's result does not depend on which rows share the launch."""
    s, t = special_rows(67, 5003, seed=13, dtype=torch.bfloat16)
    full = [None if x is None else to64(x) for x in gpu_pair(B, s, t, 0.5)]
    part = [None if x is None else to64(x) for x in gpu_pair(B, s[20:31], t[20:31], 0.5)]
    assert np.array_equal(full[0][20:31], part[0], equal_nan=True)
    assert np.array_equal(full[2][20:31], part[2])
    assert np.array_equal(full[3][20:31], part[3])


# ---------------------------------------------------------------------------
# The five workloads at full size: sampled rows against the oracle
# ---------------------------------------------------------------------------
def _sample(n, extra=(), count=24, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(n, size=min(count, n), replace=False).tolist())
    rows.update([0, n - 1], extra)
    return np.array(sorted(rows))


def test_page_shard_workload(B):
    from softmax_divergence_lm_gb300 import synth
    s, t, ids = synth.page_shard(device="cuda")
    n, v = s.shape
    rows = _sample(n)
    for beta in (0.1, 0.5, 0.9):
        check_pair(B, s, t, beta, rows=rows, gdtype=torch.bfloat16, label="page_shard")
        check_pair(B, s, t, beta, rows=rows, fused=True, label="page_shard fused")
    for op in ("kl-fwd", "kl-rev"):
        check_pair(B, s, t, None, op=op, rows=rows, label="page_shard")
    # entropy and top-8 log-probs of the student on the teacher's top ids
    out = torch.empty(n, device="cuda")
    saved = torch.empty(n, 3, device="cuda")
    dx = torch.empty(n, v, dtype=torch.float32, device="cuda")
    B.vpd_entropy_fwd(s, None, out, saved)
    B.vpd_entropy_bwd(s, None, None, saved, dx)
    lp = torch.empty(n, 8, device="cuda")
    lsaved = torch.empty(n, 2, device="cuda")
    err = torch.empty(1, dtype=torch.int32, device="cuda")
    dl = torch.empty(n, v, dtype=torch.float32, device="cuda")
    B.vpd_logprobs_fwd(s, None, ids, 8, -100, lp, lsaved, err)
    B.vpd_logprobs_bwd(s, None, ids, 8, -100, None, lsaved, dl)
    torch.cuda.synchronize()
    r = torch.as_tensor(rows, device="cuda")
    s64 = to64(s[r])
    ro, rdx = O.entropy(s64, threads=8)
    assert_loss(to64(out)[rows], ro, "page_shard entropy")
    assert_grad(to64(dx[r]), rdx, "page_shard entropy grad")
    lo, ldx, lerr = O.logprobs(s64, ids[r].cpu().numpy().astype(np.int64), -100, threads=8)
    assert lerr == 0 and int(err.item()) == 0
    assert_loss(to64(lp)[rows], lo, "page_shard top-8 logprobs")
    assert_grad(to64(dl[r]), ldx, "page_shard top-8 logprobs grad")


def test_qwen_vocab_workload(B):
    from softmax_divergence_lm_gb300 import synth
    s3, t3 = synth.qwen_vocab(device="cuda")
    bsz, seq, v = s3.shape
    n = bsz * seq
    flat_s, flat_t = s3.view(n, v), t3.view(n, v)
    # (i) rows 0..N-2 of the [N, V] buffer
    nf, _, _ = B.vpd_jsd_plan(flat_s[:-1], flat_t[:-1], None, torch.empty(n - 1, v, dtype=torch.bfloat16,
                                                                          device="cuda"), None)
    nf_fwd, _, _ = B.vpd_jsd_plan(flat_s[:-1], flat_t[:-1])
    rows = _sample(n - 1, extra=[r for r in (nf - 1, nf, nf_fwd - 1, nf_fwd) if 0 <= r < n - 1], count=16)
    check_pair(B, flat_s[:-1], flat_t[:-1], 0.5, rows=rows, gdtype=torch.bfloat16, fused=True,
               label="qwen rows")
    check_pair(B, flat_s[:-1], flat_t[:-1], 0.5, rows=rows, want_t=False, fused=True, label="qwen detached")
    # float32 gradients pin the on-chip gradient arithmetic at the stated
    # tolerance, without the rounding of a 16-bit store
    check_pair(B, flat_s[:-1], flat_t[:-1], 0.5, rows=rows, fused=True, label="qwen fp32 grads")
    check_pair(B, flat_s[:-1], flat_t[:-1], 0.5, rows=rows, label="qwen two-pass")
    # (ii) the causal-shift view [4, 2047, V]
    cs, ct = s3[:, :-1], t3[:, :-1]
    rows = _sample(bsz * (seq - 1), count=16, seed=1)
    check_pair(B, cs, ct, 0.5, rows=rows, gdtype=torch.bfloat16, fused=True, label="qwen causal")


def test_edge_case_workload(B):
    from softmax_divergence_lm_gb300 import synth
    s, t, info = synth.edge_cases(device="cuda")
    n = s.shape[0]
    special = info["disjoint_rows"][:8] + info["dead_rows"][:4]
    rows = _sample(n, extra=special, count=12)
    segs = info["segments"]
    for beta in (0.0, 0.25, 0.5, 0.75, 1.0):
        loss, _ = check_pair(B, s, t, beta, segments=segs, rows=rows, label="edge")
        dead = info["dead_rows"]
        assert np.all(np.isnan(loss[dead]))
        disjoint = info["disjoint_rows"]
        if 0.0 < beta < 1.0:
            h = -beta * math.log(beta) - (1 - beta) * math.log(1 - beta)
            assert np.allclose(loss[disjoint], h, rtol=1e-5, atol=1e-6)
        elif beta == 0.0:
            live = np.setdiff1d(np.arange(n), dead)
            assert np.all(np.isposinf(loss[live]))  # the teacher has mass on student-masked ids
        else:
            assert np.all(np.isposinf(loss[disjoint]))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_large_sweep_workload(B, dtype):
    from softmax_divergence_lm_gb300 import synth
    s, t = synth.large_sweep(device="cuda", dtype=dtype)
    n, v = s.shape
    # the first and last rows of the idle-SM share of the fwd+bwd and of the
    # forward-only calls, besides a random sample
    nf, _, _ = B.vpd_jsd_plan(s, t, None, torch.empty(n, v, dtype=dtype, device="cuda"), None)
    nf_fwd, _, _ = B.vpd_jsd_plan(s, t)
    rows = _sample(n, extra=[r for r in (nf - 1, nf, nf_fwd - 1, nf_fwd) if 0 <= r < n], count=12)
    check_pair(B, s, t, 0.5, rows=rows, gdtype=dtype, fused=True, label="sweep fused")
    check_pair(B, s, t, 0.5, rows=rows, fused=True, label="sweep fused fp32 grads")
    check_pair(B, s, t, 0.5, rows=rows, gdtype=dtype, label="sweep two-pass")
    check_pair(B, s, t, None, op="kl-fwd", rows=rows, gdtype=dtype, label="sweep")
    out = torch.empty(n, device="cuda")
    saved = torch.empty(n, 3, device="cuda")
    dx = torch.empty(n, v, dtype=dtype, device="cuda")
    gen = torch.Generator(device="cpu").manual_seed(9)
    g = torch.randn(n, generator=gen).cuda()
    B.vpd_entropy_fwd(s, None, out, saved)
    B.vpd_entropy_bwd(s, None, g, saved, dx)
    torch.cuda.synchronize()
    r = torch.as_tensor(rows, device="cuda")
    ro, rdx = O.entropy(to64(s[r]), to64(g)[rows], threads=8)
    assert_loss(to64(out)[rows], ro, "sweep entropy")
    assert_grad(to64(dx[r]), rdx, "sweep entropy grad", dtype)
    del dx
    del s, t
    torch.cuda.empty_cache()
