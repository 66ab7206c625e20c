"""Multi-rank logic on CPU with two gloo ranks: each rank computes its own
contiguous share of the token rows (no data exchange: rows are independent),
the slowest rank's time is what the benchmark reports, and the per-rank
results assemble into the single-process result exactly."""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from oracle import oracle as O

        rng = np.random.default_rng(0)
        n, v = 37, 64
        s = rng.normal(0, 3, (n, v))
        t = s + rng.normal(0, 1, (n, v))
        r0, r1 = bench.row_shard(n, world, rank)
        loss, _, _, ds, _ = O.jsd(s[r0:r1], t[r0:r1], 0.5)
        slowest = bench.max_over_ranks(float(rank + 1), world, device="cpu")
        bench.barrier(world)
        queue.put((rank, r0, r1, loss, ds, slowest))
    finally:
        dist.destroy_process_group()


def test_row_shards_cover_the_batch():
    import bench
    for n in (0, 1, 7, 8191):
        for world in (1, 2, 3, 8):
            spans = [bench.row_shard(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_two_gloo_ranks_match_single_process():
    sys.path.insert(0, ROOT)
    from oracle import oracle as O

    O.build()
    world = 2
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, queue)) for r in range(world)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    rng = np.random.default_rng(0)
    s = rng.normal(0, 3, (37, 64))
    t = s + rng.normal(0, 1, (37, 64))
    loss, _, _, ds, _ = O.jsd(s, t, 0.5)
    got_loss = np.concatenate([r[3] for r in results])
    got_ds = np.concatenate([r[4] for r in results])
    assert np.array_equal(got_loss, loss) and np.array_equal(got_ds, ds)
    assert all(r[5] == float(world) for r in results)  # every rank sees the slowest time
