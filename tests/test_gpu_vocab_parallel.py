"""The vocabulary-parallel steps (vpd_jsd_shard_* and the shard backward) on
the GPU, with the processes of a vocabulary-parallel group emulated inside one
process: every shard's steps run the library's kernels, and each all-reduce is
done by reducing the shards' [N, 2] buffers with torch between the steps (what
NCCL would do). Uneven shards, an empty shard, bf16 and fp32 inputs and the
special rows; each shard's loss and the shards' gradient columns side by side
against the oracle on the full vocabulary."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity_util import assert_grad, assert_loss, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from softmax_divergence_lm_gb300 import build
    build.build()
    from softmax_divergence_lm_gb300 import binding
    binding.load()
    return binding


def emulated_group(B, s_shards, t_shards, beta, g):
    n = s_shards[0].shape[0]
    w = len(s_shards)
    loss = [torch.empty(n, device="cuda") for _ in range(w)]
    saved = [torch.empty(n, 6, device="cuda") for _ in range(w)]
    x = [torch.empty(n, 2, device="cuda") for _ in range(w)]

    def all_reduce(op):
        r = torch.stack(x).amax(0) if op == "max" else torch.stack(x).sum(0)
        for b in x:
            b.copy_(r)

    for k in range(w):
        B.vpd_jsd_shard_stats(s_shards[k], t_shards[k], saved[k], x[k])
    all_reduce("max")
    for k in range(w):
        B.vpd_jsd_shard_rescale(n, saved[k], x[k])
    all_reduce("sum")
    for k in range(w):
        B.vpd_jsd_shard_divergence(s_shards[k], t_shards[k], beta, loss[k], saved[k], x[k])
    all_reduce("sum")
    for k in range(w):
        B.vpd_jsd_shard_finish(n, beta, saved[k], x[k], loss[k])
    ds, dt = [], []
    for k in range(w):
        d1 = torch.full(s_shards[k].shape, 3.0, device="cuda")
        d2 = torch.full(t_shards[k].shape, 3.0, device="cuda")
        B.vpd_jsd_bwd(s_shards[k], t_shards[k], beta, None, g, saved[k], d1, d2)
        ds.append(d1)
        dt.append(d2)
    torch.cuda.synchronize()
    return loss, saved, torch.cat(ds, 1), torch.cat(dt, 1)


def special(n, v, dtype, seed):
    gen = torch.Generator(device="cpu").manual_seed(seed)
    s = torch.randn(n, v, generator=gen) * 3
    t = 0.6 * s + torch.randn(n, v, generator=gen) * 2
    s[1, 2:40] = -math.inf
    t[2, v - 30:] = -math.inf
    s[3], t[3] = -math.inf, -math.inf
    s[4, v - 1] = math.nan
    t[5, 7] = math.inf
    s[6, 0] = -math.inf              # forward KL: +inf (teacher mass on it)
    t[7, v // 2] = -math.inf         # reverse KL: +inf
    s[8, : v // 2] = -math.inf       # the student lives on the later shards only
    return s.to(dtype).cuda(), t.to(dtype).cuda()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("widths", [(700, 0, 1349, 1), (2050,), (1024, 1026)], ids=["uneven+empty", "one", "two"])
def test_emulated_shards_match_oracle(B, dtype, widths):
    n, v = 16, sum(widths)
    s, t = special(n, v, dtype, seed=len(widths))
    offs = np.concatenate([[0], np.cumsum(widths)])
    s_sh = [s[:, offs[k]:offs[k + 1]] for k in range(len(widths))]
    t_sh = [t[:, offs[k]:offs[k + 1]] for k in range(len(widths))]
    gen = torch.Generator(device="cpu").manual_seed(9)
    g = torch.randn(n, generator=gen).cuda()
    for beta in (0.5, 0.0, 1.0, 0.2):
        loss, saved, ds, dt = emulated_group(B, s_sh, t_sh, beta, g)
        rl, ra, rb, rds, rdt = O.jsd(to64(s), to64(t), beta, to64(g), threads=4)
        for k, lk in enumerate(loss):
            assert_loss(to64(lk), rl, f"shard {k} loss beta={beta} {widths}")
        assert_grad(to64(ds), rds, f"dS beta={beta} {widths}")
        assert_grad(to64(dt), rdt, f"dT beta={beta} {widths}")
        # every shard holds the same saved statistics, equal to the oracle's
        for k in range(1, len(widths)):
            assert torch.equal(torch.nan_to_num(saved[k], 1.0), torch.nan_to_num(saved[0], 1.0))


def test_emulated_tp2_qwen_vocab(B):
    """Two shards of the Qwen2.5 vocabulary (75968 columns each, as in the
    pages' TP2 runs) on sampled rows of the Qwen-vocabulary workload."""
    from softmax_divergence_lm_gb300 import synth
    s3, t3 = synth.qwen_vocab(device="cuda", batch=1, seq=256)
    s, t = s3[0], t3[0]
    n, v = s.shape
    h = v // 2
    g = torch.full((n,), 1.0 / n, device="cuda")
    loss, _, ds, dt = emulated_group(B, [s[:, :h], s[:, h:]], [t[:, :h], t[:, h:]], 0.3, g)
    rows = np.arange(0, n, 9)
    r = torch.as_tensor(rows, device="cuda")
    rl, _, _, rds, rdt = O.jsd(to64(s[r]), to64(t[r]), 0.3, to64(g)[rows], threads=8)
    assert_loss(to64(loss[0])[rows], rl, "TP2 loss rank 0")
    assert_loss(to64(loss[1])[rows], rl, "TP2 loss rank 1")
    assert_grad(to64(ds[r]), rds, "TP2 dS")
    assert_grad(to64(dt[r]), rdt, "TP2 dT")
