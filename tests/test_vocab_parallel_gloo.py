"""The vocabulary-parallel exchange protocol (softmax_divergence_lm_gb300.
vocab_parallel: one MAX and two SUM all-reduces of [N, 2] per-token buffers,
'Add vocabulary-parallel logprobs, entropy and KL ops', section How) with real
gloo ranks on CPU. Each rank holds an uneven vocabulary shard (one case gives a
rank an empty shard); the per-shard steps run in a float64 CPU stand-in for
the library's kernels. Every rank's loss and the ranks' gradient columns put
side by side must equal the single-process oracle on the full vocabulary."""
from __future__ import annotations

import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(n=9, v=23):
    rng = np.random.default_rng(4)
    s = rng.normal(0, 3, (n, v))
    t = 0.6 * s + rng.normal(0, 2, (n, v))
    s[1, 2:6] = -np.inf           # masked student tokens (on rank 0's shard)
    t[2, v - 3:] = -np.inf        # masked teacher tail (on the last shard)
    s[3], t[3] = -np.inf, -np.inf  # no distribution: NaN, zero gradient
    s[4, v - 1] = np.nan          # outside the contract, on the last shard only
    t[5, 1] = -np.inf             # the teacher masks a token the student keeps
    s[6, 0] = -np.inf             # the student masks a token the teacher keeps
    return s, t


def _worker(rank, world, port, widths, betas, queue):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, TESTS)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from softmax_divergence_lm_gb300 import vocab_parallel as VP
        from vocab_parallel_double import NumpyShardKernels

        s, t = _inputs()
        off = int(np.sum(widths[:rank]))
        sl = slice(off, off + widths[rank])
        s_loc = torch.from_numpy(np.ascontiguousarray(s[:, sl]))
        t_loc = torch.from_numpy(np.ascontiguousarray(t[:, sl]))
        g = torch.from_numpy(np.linspace(-1.0, 1.5, s.shape[0]))
        out = []
        k = NumpyShardKernels()
        for beta in betas:
            loss, saved = VP.jsd_forward(s_loc.double(), t_loc.double(), beta, kernels=k)
            ds, dt = torch.empty_like(s_loc), torch.empty_like(t_loc)
            VP.jsd_backward(s_loc, t_loc, beta, g, saved, ds, dt, kernels=k)
            out.append((beta, loss.numpy().copy(), ds.numpy().copy(), dt.numpy().copy()))
        queue.put((rank, out))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("widths", [(9, 14), (0, 23), (23, 0)], ids=["uneven", "empty-first", "empty-last"])
def test_two_gloo_ranks_vocab_shards_match_oracle(widths):
    # the exchange buffers are float32, as on the GPU, so the comparison uses
    # the stated tolerances
    sys.path.insert(0, ROOT)
    from oracle import oracle as O

    O.build()
    betas = (0.5, 0.0, 1.0, 0.3)
    world = 2
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, widths, betas, queue)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(queue.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    s, t = _inputs()
    g = np.linspace(-1.0, 1.5, s.shape[0])
    for i, beta in enumerate(betas):
        rl, _, _, rds, rdt = O.jsd(s, t, beta, g)
        for r in range(world):
            got = results[r][i][1]
            assert np.array_equal(np.isnan(got), np.isnan(rl)) and np.array_equal(np.isposinf(got), np.isposinf(rl))
            fin = np.isfinite(rl)
            # float32 buffers between the steps: the stated loss tolerance
            assert np.all(np.abs(got[fin] - rl[fin]) <= 1e-6 + 1e-5 * np.abs(rl[fin])), (beta, r)
        ds = np.concatenate([results[r][i][2] for r in range(world)], axis=1)
        dt = np.concatenate([results[r][i][3] for r in range(world)], axis=1)
        assert np.all(np.abs(ds - rds) <= 1e-6 + 1e-4 * np.abs(rds)), beta
        assert np.all(np.abs(dt - rdt) <= 1e-6 + 1e-4 * np.abs(rdt)), beta
        assert math.isnan(rl[3]) and math.isnan(rl[4])
