"""The autograd layer (softmax_divergence_lm_gb300.ops) against the CPU oracle:
forward values and the gradients autograd delivers to both inputs, the
input-dtype gradient default, the refusal of a second backward ('Add
vocabulary-parallel logprobs, entropy and KL ops', section Limitations: only
first-order gradients), and the index check of the log-prob op."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity_util import assert_grad, assert_loss, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from softmax_divergence_lm_gb300 import build
    build.build()
    from softmax_divergence_lm_gb300 import ops as ops_mod
    return ops_mod


def _inputs(n, v, dtype, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    s = torch.randn(n, v, generator=g) * 3
    t = s + torch.randn(n, v, generator=g) * 2
    s[1, 10:60] = -math.inf
    s[2], t[2] = -math.inf, -math.inf  # no distribution: NaN, zero gradient
    return s.to(dtype).cuda(), t.to(dtype).cuda()


def _upstream(n, seed=4):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(n, generator=g).cuda()


def _gd(dtype):
    return None if dtype == torch.float32 else dtype


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("beta", [0.5, 0.0, 1.0])
def test_jsd_autograd(ops, dtype, beta):
    s, t = _inputs(16, 4104, dtype, seed=1)
    s.requires_grad_(True)
    t.requires_grad_(True)
    loss = ops.jsd(s, t, beta)
    g = _upstream(16)
    # the NaN row's upstream gradient is nonzero on purpose: its input gradient stays 0
    loss.backward(g)
    assert s.grad.dtype == dtype and t.grad.dtype == dtype  # gradients in the input dtype by default
    rl, _, _, rds, rdt = O.jsd(to64(s), to64(t), beta, to64(g), threads=4)
    assert_loss(to64(loss), rl, f"ops.jsd beta={beta} {dtype}")
    assert_grad(to64(s.grad), rds, f"ops.jsd dS beta={beta}", _gd(dtype))
    assert_grad(to64(t.grad), rdt, f"ops.jsd dT beta={beta}", _gd(dtype))
    assert np.all(to64(s.grad)[2] == 0) and np.all(to64(t.grad)[2] == 0)


def test_jsd_detached_teacher(ops):
    s, t = _inputs(8, 2048, torch.bfloat16, seed=2)
    s.requires_grad_(True)
    loss = ops.jsd(s, t.detach(), 0.3)
    g = _upstream(8)
    loss.backward(g)
    _, _, _, rds, _ = O.jsd(to64(s), to64(t), 0.3, to64(g), threads=4)
    assert_grad(to64(s.grad), rds, "ops.jsd detached dS", torch.bfloat16)
    assert t.grad is None


@pytest.mark.parametrize("reverse", [False, True])
def test_kl_autograd(ops, reverse):
    s, t = _inputs(12, 3000, torch.float32, seed=3)
    s.requires_grad_(True)
    t.requires_grad_(True)
    loss = ops.kl_div(s, t, reverse=reverse)
    g = _upstream(12)
    loss.backward(g)
    rl, rds, rdt = O.kl(to64(s), to64(t), reverse, to64(g), threads=4)
    assert_loss(to64(loss), rl, f"ops.kl_div reverse={reverse}")
    assert_grad(to64(s.grad), rds, "ops.kl_div dS")
    assert_grad(to64(t.grad), rdt, "ops.kl_div dT")


def test_entropy_autograd_3d(ops):
    s, _ = _inputs(12, 1500, torch.bfloat16, seed=5)
    x = s.view(3, 4, 1500).clone().requires_grad_(True)
    h = ops.entropy(x)
    assert h.shape == (3, 4)
    g = _upstream(12).view(3, 4)
    h.backward(g)
    ro, rdx = O.entropy(to64(s), to64(g).reshape(-1), threads=4)
    assert_loss(to64(h).reshape(-1), ro, "ops.entropy")
    assert_grad(to64(x.grad).reshape(12, 1500), rdx, "ops.entropy dX", torch.bfloat16)


def test_logprobs_autograd(ops):
    s, _ = _inputs(10, 777, torch.float32, seed=6)
    x = s.clone().requires_grad_(True)
    idx = torch.randint(0, 777, (10, 3), generator=torch.Generator().manual_seed(1)).cuda()
    idx[0, 1] = -100          # ignored position
    idx[3, 2] = idx[3, 0]     # duplicate id
    out = ops.logprobs(x, idx)
    gk = torch.randn(10, 3, generator=torch.Generator().manual_seed(2)).cuda()
    out.backward(gk)
    ro, rdx, errs = O.logprobs(to64(s), idx.cpu().numpy(), -100, to64(gk), threads=4)
    assert errs == 0
    assert_loss(to64(out), ro, "ops.logprobs")
    assert_grad(to64(x.grad), rdx, "ops.logprobs dX")
    one = ops.logprobs(s, idx[:, 0])  # one id per token: [N] output
    assert one.shape == (10,)


def test_logprobs_out_of_range_raises_index_error(ops):
    s, _ = _inputs(4, 100, torch.float32, seed=7)
    idx = torch.tensor([[1], [2], [100], [3]], device="cuda")
    with pytest.raises(IndexError):
        ops.logprobs(s, idx)


@pytest.mark.parametrize("op", ["jsd", "kl", "entropy", "logprobs"])
def test_double_backward_raises(ops, op):
    s, t = _inputs(4, 512, torch.float32, seed=8)
    s.requires_grad_(True)
    t.requires_grad_(True)
    if op == "jsd":
        y = ops.jsd(s, t, 0.5)
    elif op == "kl":
        y = ops.kl_div(s, t)
    elif op == "entropy":
        y = ops.entropy(s)
    else:
        y = ops.logprobs(s, torch.zeros(4, 1, dtype=torch.int64, device="cuda"))
    y = torch.nan_to_num(y).sum()
    (gs,) = torch.autograd.grad(y, s, create_graph=True)
    with pytest.raises(RuntimeError):
        torch.autograd.grad(gs.sum(), s)


def test_jsd_fwdbwd_wrapper(ops):
    s, t = _inputs(6, 8192, torch.bfloat16, seed=9)
    g = _upstream(6)
    loss, saved, ds, dt = ops.jsd_fwdbwd(s, t, 0.5, grad_loss=g, grad_dtype=torch.float32)
    rl, _, _, rds, rdt = O.jsd(to64(s), to64(t), 0.5, to64(g), threads=4)
    assert_loss(to64(loss), rl, "jsd_fwdbwd loss")
    assert_grad(to64(ds), rds, "jsd_fwdbwd dS")
    assert_grad(to64(dt), rdt, "jsd_fwdbwd dT")
    assert saved.shape == (6, 6)
