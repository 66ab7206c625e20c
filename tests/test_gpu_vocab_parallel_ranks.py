"""The vocabulary-parallel JSD through its torch.distributed driver with two
real processes: two gloo ranks share the one GPU, each runs the library's
shard kernels on its own vocabulary shard, and the all-reduces of the [N, 2]
exchange buffers go through gloo on the host (the kernels of the two ranks
never wait on each other). The autograd op `vocab_parallel_jsd` is used, so
the backward is exercised too. Each rank's loss and the ranks' gradient
columns side by side must match the oracle on the full vocabulary."""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(n=48, v=3000):
    g = torch.Generator(device="cpu").manual_seed(31)
    s = torch.randn(n, v, generator=g) * 3
    t = 0.6 * s + torch.randn(n, v, generator=g) * 2
    s[1, 5:40] = -float("inf")
    s[3], t[3] = -float("inf"), -float("inf")
    return s.to(torch.bfloat16), t.to(torch.bfloat16)


def _worker(rank, world, port, widths, queue):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from softmax_divergence_lm_gb300 import build
        from softmax_divergence_lm_gb300 import vocab_parallel as VP

        build.build()
        torch.cuda.set_device(0)
        s, t = _inputs()
        off = int(np.sum(widths[:rank]))
        s_loc = s[:, off:off + widths[rank]].contiguous().cuda().requires_grad_(True)
        t_loc = t[:, off:off + widths[rank]].contiguous().cuda().requires_grad_(True)
        g = torch.linspace(-1.0, 1.0, s.shape[0], device="cuda")
        out = []
        for beta in (0.5, 0.0):
            s_loc.grad = t_loc.grad = None
            loss = VP.vocab_parallel_jsd(s_loc, t_loc, beta)
            loss.backward(g)
            torch.cuda.synchronize()
            out.append((beta, loss.detach().double().cpu().numpy(), s_loc.grad.double().cpu().numpy(),
                        t_loc.grad.double().cpu().numpy()))
        queue.put((rank, out))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("widths", [(1100, 1900), (0, 3000)], ids=["uneven", "empty"])
def test_two_ranks_on_one_gpu_match_oracle(widths):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, TESTS)
    from oracle import oracle as O
    from parity_util import assert_grad, assert_loss

    assert torch.cuda.is_available()
    world = 2
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, widths, queue)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(queue.get(timeout=600) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    s, t = _inputs()
    s64, t64 = s.double().numpy(), t.double().numpy()
    g = np.linspace(-1.0, 1.0, s.shape[0])
    for i, beta in enumerate((0.5, 0.0)):
        rl, _, _, rds, rdt = O.jsd(s64, t64, beta, g)
        for r in range(world):
            assert_loss(results[r][i][1], rl, f"rank {r} loss beta={beta}")
        ds = np.concatenate([results[r][i][2] for r in range(world)], axis=1)
        dt = np.concatenate([results[r][i][3] for r in range(world)], axis=1)
        assert_grad(ds, rds, f"dS beta={beta}", torch.bfloat16)
        assert_grad(dt, rdt, f"dT beta={beta}", torch.bfloat16)
