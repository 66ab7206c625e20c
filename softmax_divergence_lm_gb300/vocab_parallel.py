"""Vocabulary-parallel generalized JSD / KL across processes.

Each process holds one ordered vocabulary shard [N, V_k] of the student and
teacher logits (V_k may differ between processes and may be 0). The forward
exchanges only [N]-sized per-token statistics: one MAX all-reduce of the maxima
and two SUM all-reduces (the rescaled sum-exps, then the two KL-to-mixture
partial sums), as in 'Add vocabulary-parallel logprobs, entropy and KL ops',
section How, and '[VocabTP] Add vocabulary-parallel generalized JSD with
Triton kernels', section Changes. The backward is local: each process gets the
gradient of its own vocabulary columns, and every process back-propagates the
same replicated per-token loss.

All per-row work runs in the library's kernels (``vpd_jsd_shard_*`` and
``vpd_jsd_bwd``); this module only orders the steps and runs the
``torch.distributed`` all-reduces between them on the [N, 2] exchange buffer.
The step functions are reached through a ``kernels`` object so that the
protocol can be exercised by multi-process tests on hosts without a GPU.
"""
from __future__ import annotations

import torch
import torch.distributed as dist
from torch.autograd.function import once_differentiable

from . import binding as B


class ShardKernels:
    """The library's per-shard steps on device tensors (the product path)."""

    def stats(self, s, t, saved, xbuf):
        B.vpd_jsd_shard_stats(s, t, saved, xbuf)

    def rescale(self, rows, saved, xbuf):
        B.vpd_jsd_shard_rescale(rows, saved, xbuf)

    def divergence(self, s, t, beta, loss, saved, xbuf):
        B.vpd_jsd_shard_divergence(s, t, beta, loss, saved, xbuf)

    def finish(self, rows, beta, saved, xbuf, loss):
        B.vpd_jsd_shard_finish(rows, beta, saved, xbuf, loss)

    def backward(self, s, t, beta, grad, saved, ds, dt):
        B.vpd_jsd_bwd(s, t, beta, None, grad, saved, ds, dt)


def _all_reduce(x: torch.Tensor, op, group):
    """All-reduce of the [N, 2] exchange buffer. NCCL reduces it in device
    memory; a gloo group gets a host copy (the buffer is 8 bytes per row)."""
    if x.is_cuda and dist.get_backend(group) == "gloo":
        h = x.cpu()
        dist.all_reduce(h, op=op, group=group)
        x.copy_(h)
    else:
        dist.all_reduce(x, op=op, group=group)


def _rows(x: torch.Tensor) -> int:
    return x.shape[0] if x.dim() == 2 else x.shape[0] * x.shape[1]


def jsd_forward(s_local: torch.Tensor, t_local: torch.Tensor, beta: float, group=None, kernels=None):
    """Per-token JSD_beta (beta = 0 / 1: forward / reverse KL) of the full
    vocabulary from this process's shard. Returns (loss [N], saved [N, 6]),
    identical on every process of `group`."""
    k = kernels or ShardKernels()
    n = _rows(s_local)
    dev = s_local.device
    loss = torch.empty(n, dtype=torch.float32, device=dev)
    saved = torch.empty(n, B.SAVED_PAIR, dtype=torch.float32, device=dev)
    xbuf = torch.empty(n, 2, dtype=torch.float32, device=dev)
    k.stats(s_local, t_local, saved, xbuf)
    _all_reduce(xbuf, dist.ReduceOp.MAX, group)   # global maxima
    k.rescale(n, saved, xbuf)
    _all_reduce(xbuf, dist.ReduceOp.SUM, group)   # global sum-exps
    k.divergence(s_local, t_local, float(beta), loss, saved, xbuf)
    _all_reduce(xbuf, dist.ReduceOp.SUM, group)   # global KL-to-mixture sums
    k.finish(n, float(beta), saved, xbuf, loss)
    return loss, saved


def jsd_backward(s_local, t_local, beta, grad, saved, ds=None, dt=None, kernels=None):
    """This process's vocabulary columns of dS and dT; no communication."""
    k = kernels or ShardKernels()
    k.backward(s_local, t_local, float(beta), grad, saved, ds, dt)
    return ds, dt


class _VocabParallelJSD(torch.autograd.Function):
    @staticmethod
    def forward(ctx, s, t, beta, group):
        loss, saved = jsd_forward(s, t, beta, group)
        ctx.save_for_backward(s, t, saved)
        ctx.beta = beta
        return loss.view(s.shape[:-1])

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        s, t, saved = ctx.saved_tensors
        ds = torch.empty_like(s) if ctx.needs_input_grad[0] else None
        dt = torch.empty_like(t) if ctx.needs_input_grad[1] else None
        jsd_backward(s, t, ctx.beta, g.reshape(-1).to(torch.float32).contiguous(), saved, ds, dt)
        return ds, dt, None, None


def vocab_parallel_jsd(student_shard: torch.Tensor, teacher_shard: torch.Tensor, beta: float = 0.5,
                       group=None) -> torch.Tensor:
    """Autograd op: the per-token JSD_beta over the full vocabulary, each process
    passing its own ordered shard of the student and teacher logits."""
    return _VocabParallelJSD.apply(student_shard, teacher_shard, float(beta), group)
