"""JSD forward+backward with the teacher logits in a pinned host cache
('Add an opt-in vocabulary-parallel KL route to OPSD', section "Update: copy
teacher-cache chunks from pinned memory"): the library's chunk pipeline (copy
stream, staging ring, events) against the oracle and against the same call with
the teacher already on the device."""
from __future__ import annotations

import ctypes

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


@pytest.mark.parametrize("dtype,gdtype", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32)])
@pytest.mark.parametrize("chunk,nstage", [(128, 2), (96, 4), (1000, 2)])
def test_teacher_cache_stream(B, dtype, gdtype, chunk, nstage):
    from softmax_divergence_lm_gb300 import synth
    s_all, t_all, _ = synth.page_shard(device="cuda", n=1000, topk=0)
    s = s_all.to(dtype)
    t_dev = t_all.to(dtype)
    t_host = t_dev.cpu().pin_memory()
    n, v = s.shape
    g = torch.randn(n, generator=torch.Generator().manual_seed(3)).cuda()
    staging = torch.empty(nstage * chunk * v * s.element_size(), dtype=torch.uint8, device="cuda")
    copy = torch.cuda.Stream()
    loss = torch.full((n,), 7.0, device="cuda")
    saved = torch.empty(n, 6, device="cuda")
    ds = torch.full((n, v), 3.0, dtype=gdtype, device="cuda")
    B.vpd_jsd_fwdbwd_teacher_stream(s, t_host, 0.5, g, loss, saved, ds, None, staging, chunk, copy_stream=copy)
    # the same call with the teacher on the device
    loss2 = torch.empty(n, device="cuda")
    saved2 = torch.empty(n, 6, device="cuda")
    ds2 = torch.empty(n, v, dtype=gdtype, device="cuda")
    B.vpd_jsd_fwdbwd(s, t_dev, 0.5, None, g, loss2, saved2, ds2, None)
    torch.cuda.synchronize()
    B.vpd_device_status()
    gd = None if gdtype == torch.float32 else gdtype
    assert_loss(to64(loss), to64(loss2), "streamed vs device-resident loss")
    assert_grad(to64(ds), to64(ds2), "streamed vs device-resident dS", gd)
    rows = np.unique(np.concatenate([np.arange(0, n, 37), [n - 1, chunk - 1, min(chunk, n - 1)]]))
    r = torch.as_tensor(rows, device="cuda")
    rl, _, _, rds, _ = O.jsd(to64(s[r]), to64(t_dev[r]), 0.5, to64(g)[rows], threads=8)
    assert_loss(to64(loss)[rows], rl, "streamed loss")
    assert_grad(to64(ds[r]), rds, "streamed dS", gd)


def test_pageable_cache_is_refused(B):
    n, v = 4, 64
    s = torch.randn(n, v, device="cuda")
    host = np.random.default_rng(0).normal(size=(n, v)).astype(np.float32)  # pageable
    loss = torch.empty(n, device="cuda")
    saved = torch.empty(n, 6, device="cuda")
    staging = torch.empty(2 * n * v * 4, dtype=torch.uint8, device="cuda")
    copy = torch.cuda.Stream()
    vs = B.make_view(s)
    st = B.load().vpd_jsd_fwdbwd_teacher_stream(
        ctypes.byref(vs), host.ctypes.data, B.VPD_F32, v, 0.5, None, loss.data_ptr(), saved.data_ptr(), None,
        None, staging.data_ptr(), staging.numel(), n, torch.cuda.current_stream().cuda_stream, copy.cuda_stream)
    assert st == B.VPD_ERR_ARG
