"""Cross-entropy and the teacher top-k forward KL ('Add vocabulary-parallel
logprobs, entropy and KL ops', sections What and How), with and without a
temperature, through the C ABI against the oracle's compositions, element by
element at the stated tolerances; plus their autograd wrappers."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity_util import assert_grad, assert_loss, assert_zero_rows, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from softmax_divergence_lm_gb300 import build
    build.build()
    from softmax_divergence_lm_gb300 import binding
    binding.load()
    return binding


def rows(n, v, dtype, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(n, v, generator=g) * 3
    x[1, 5:60] = -math.inf     # masked tokens
    x[2] = -math.inf           # no distribution
    x[3, 11] = math.nan        # out of contract
    x[4, v - 1] = x[4].max() + 40.0  # peaked
    return x.to(dtype).cuda()


def teacher_topk(n, v, k, seed):
    """Teacher top-k ids and log-probs, made on the host in float64 (inputs to
    both sides)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    t = torch.randn(n, v, generator=g, dtype=torch.float64) * 3
    lp = torch.log_softmax(t, dim=1)
    val, ids = torch.topk(lp, k, dim=1)
    return ids.contiguous(), val.to(torch.float32).contiguous()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("temp", [1.0, 0.7])
def test_cross_entropy(B, dtype, temp):
    n, v = 24, 3001
    x = rows(n, v, dtype, seed=1)
    gen = torch.Generator(device="cpu").manual_seed(2)
    labels = torch.randint(0, v, (n,), generator=gen)
    labels[5] = -100            # ignored
    labels[1] = 20              # a masked label: +inf, no gradient
    labels = labels.cuda()
    g = torch.randn(n, generator=gen).cuda()
    loss = torch.full((n,), 7.0, device="cuda")
    saved = torch.empty(n, 2, device="cuda")
    err = torch.empty(1, dtype=torch.int32, device="cuda")
    dx = torch.full((n, v), 3.0, device="cuda")
    B.vpd_cross_entropy_fwd(x, None, labels, -100, temp, loss, saved, err)
    B.vpd_cross_entropy_bwd(x, None, labels, -100, temp, g, saved, dx)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rl, rdx, errs = O.cross_entropy(to64(x), labels.cpu().numpy(), -100, temp, to64(g), threads=4)
    assert errs == 0
    assert_loss(to64(loss), rl, f"CE T={temp} {dtype}")
    assert np.isposinf(to64(loss)[1]) and to64(loss)[5] == 0.0
    assert_grad(to64(dx), rdx, f"CE grad T={temp} {dtype}")
    assert_zero_rows(to64(dx), [1, 2, 3, 5], "CE grad")


def test_cross_entropy_out_of_range(B):
    x = rows(6, 100, torch.float32, seed=3)[[0, 4, 5, 4]].contiguous()
    labels = torch.tensor([1, 2, 100, 3], device="cuda")
    loss = torch.empty(4, device="cuda")
    err = torch.empty(1, dtype=torch.int32, device="cuda")
    B.vpd_cross_entropy_fwd(x, None, labels, -100, 1.0, loss, None, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1 and math.isnan(float(loss[2]))
    with pytest.raises(B.VpdError) as info:
        B.vpd_cross_entropy_fwd(x, None, labels, -100, 1.0, loss, None, None)
    assert info.value.status == B.VPD_ERR_INDEX


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("temp", [1.0, 1.5])
def test_topk_forward_kl(B, dtype, temp):
    n, v, k = 24, 4104, 8
    s = rows(n, v, dtype, seed=4)
    ids, tl = teacher_topk(n, v, k, seed=5)
    ids[6, 3] = -100                    # ignored position
    ids[7, 2] = ids[7, 1]               # duplicate id
    tl[8, 5] = -math.inf                # no teacher mass at one position
    ids[9, 0] = 30                      # the student masks id 30 in row 1 only...
    ids[1, 0] = 30                      # ...so row 1 is +inf (teacher mass on a masked id)
    ids, tl = ids.cuda(), tl.cuda()
    gen = torch.Generator(device="cpu").manual_seed(6)
    g = torch.randn(n, generator=gen).cuda()
    kl = torch.full((n,), 7.0, device="cuda")
    saved = torch.empty(n, 2, device="cuda")
    err = torch.empty(1, dtype=torch.int32, device="cuda")
    ds = torch.full((n, v), 3.0, device="cuda")
    B.vpd_topk_kl_fwd(s, None, ids, k, -100, tl, temp, kl, saved, err)
    B.vpd_topk_kl_bwd(s, None, ids, k, -100, tl, temp, g, saved, ds)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rk, rds, errs = O.topk_forward_kl(to64(s), ids.cpu().numpy(), to64(tl), -100, temp, to64(g), threads=4)
    assert errs == 0
    assert_loss(to64(kl), rk, f"top-k KL T={temp} {dtype}")
    assert np.isposinf(to64(kl)[1])
    assert_grad(to64(ds), rds, f"top-k KL grad T={temp} {dtype}")
    assert_zero_rows(to64(ds), [1, 2, 3], "top-k KL grad")


def test_page_shard_cross_entropy_and_topk_kl(B):
    """The shard workload: cross-entropy at the teacher's argmax and the
    top-8 forward KL with the teacher's log-probs, on sampled rows."""
    from softmax_divergence_lm_gb300 import synth
    s, t, ids = synth.page_shard(device="cuda")
    n, v = s.shape
    rng = np.random.default_rng(0)
    r = np.unique(np.concatenate([rng.choice(n, 24, replace=False), [0, n - 1]]))
    rt = torch.as_tensor(r, device="cuda")
    # teacher log-probs at its top-8 ids, made on the host in float64
    tl = torch.log_softmax(t[rt].double().cpu(), dim=1).gather(1, ids[rt].cpu()).float()
    tl_all = torch.zeros(n, 8)
    tl_all[torch.as_tensor(r)] = tl
    tl_all = tl_all.cuda()
    g = torch.ones(n, device="cuda")
    loss = torch.empty(n, device="cuda")
    saved = torch.empty(n, 2, device="cuda")
    err = torch.empty(1, dtype=torch.int32, device="cuda")
    dx = torch.empty(n, v, dtype=torch.bfloat16, device="cuda")
    labels = ids[:, 0].contiguous()
    B.vpd_cross_entropy_fwd(s, None, labels, -100, 1.0, loss, saved, err)
    B.vpd_cross_entropy_bwd(s, None, labels, -100, 1.0, g, saved, dx)
    torch.cuda.synchronize()
    rl, rdx, _ = O.cross_entropy(to64(s[rt]), labels[rt].cpu().numpy(), -100, 1.0, np.ones(len(r)), threads=8)
    assert_loss(to64(loss)[r], rl, "page_shard CE")
    assert_grad(to64(dx[rt]), rdx, "page_shard CE grad", torch.bfloat16)
    kl = torch.empty(n, device="cuda")
    B.vpd_topk_kl_fwd(s, None, ids, 8, -100, tl_all, 1.0, kl, saved, err)
    B.vpd_topk_kl_bwd(s, None, ids, 8, -100, tl_all, 1.0, g, saved, dx)
    torch.cuda.synchronize()
    rk, rds, _ = O.topk_forward_kl(to64(s[rt]), ids[rt].cpu().numpy(), tl.double().numpy(), -100, 1.0,
                                   np.ones(len(r)), threads=8)
    assert_loss(to64(kl)[r], rk, "page_shard top-8 KL")
    assert_grad(to64(dx[rt]), rds, "page_shard top-8 KL grad", torch.bfloat16)


def test_autograd_wrappers(B):
    from softmax_divergence_lm_gb300 import ops
    n, v, k = 10, 999, 4
    x = rows(n, v, torch.float32, seed=7)[5:].clone().requires_grad_(True)  # rows without special classes
    m = x.shape[0]
    labels = torch.randint(0, v, (m,), generator=torch.Generator().manual_seed(1)).cuda()
    ce = ops.cross_entropy(x, labels, temperature=2.0)
    g = torch.randn(m, generator=torch.Generator().manual_seed(2)).cuda()
    ce.backward(g)
    rl, rdx, _ = O.cross_entropy(to64(x), labels.cpu().numpy(), -100, 2.0, to64(g), threads=4)
    assert_loss(to64(ce), rl, "ops.cross_entropy")
    assert_grad(to64(x.grad), rdx, "ops.cross_entropy grad")
    ids, tl = teacher_topk(m, v, k, seed=8)
    x.grad = None
    kl = ops.topk_forward_kl(x, ids.cuda(), tl.cuda())
    kl.backward(g)
    rk, rds, _ = O.topk_forward_kl(to64(x), ids.numpy(), tl.double().numpy(), -100, 1.0, to64(g), threads=4)
    assert_loss(to64(kl), rk, "ops.topk_forward_kl")
    assert_grad(to64(x.grad), rds, "ops.topk_forward_kl grad")
    with pytest.raises(IndexError):
        ops.cross_entropy(x.detach(), torch.full((m,), v, device="cuda"))
