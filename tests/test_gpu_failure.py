"""Failure detection without a GPU fault: a bounded device-side wait is made
to run out (a copy that is never issued, set up by the library's test hook),
the kernel leaves its row loop instead of hanging, the host reads
VPD_ERR_TIMEOUT from vpd_device_status, and the device stays usable: the next
call on the same context matches the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import oracle as O
from parity_util import assert_loss, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from softmax_divergence_lm_gb300 import build
    build.build()
    from softmax_divergence_lm_gb300 import binding
    binding.load()
    return binding


def _call(B, s, t, grads=True):
    n, v = s.shape
    loss = torch.empty(n, device="cuda")
    saved = torch.empty(n, 6, device="cuda")
    ds = torch.empty(n, v, dtype=s.dtype, device="cuda") if grads else None
    dt = torch.empty(n, v, dtype=s.dtype, device="cuda") if grads else None
    c0 = B.vpd_launch_count()
    B.vpd_jsd_fwdbwd(s, t, 0.5, None, None, loss, saved, ds, dt)
    torch.cuda.synchronize()
    assert B.vpd_launch_count() - c0 == 1, "the single-read kernel must run"
    return loss


@pytest.mark.parametrize("grads", [True, False])  # the forward+backward and the forward-only kernel
@pytest.mark.parametrize("v", [8192, 151936])  # one CTA per row, and a cluster of CTAs per row
def test_bounded_wait_reports_timeout_and_device_recovers(B, v, grads):
    g = torch.Generator(device="cpu").manual_seed(3)
    s = (torch.randn(24, v, generator=g) * 3).to(torch.bfloat16).cuda()
    t = (torch.randn(24, v, generator=g) * 3).to(torch.bfloat16).cuda()
    _call(B, s, t, grads)
    B.vpd_device_status()  # clean before the injected failure
    B.vpd_test_withhold_copy(5)
    _call(B, s, t, grads)
    with pytest.raises(B.VpdError) as err:
        B.vpd_device_status()
    assert err.value.status == B.VPD_ERR_TIMEOUT
    B.vpd_device_status()  # the error word was cleared by the read
    loss = _call(B, s, t, grads)  # the context is still usable and the result is right
    B.vpd_device_status()
    rl = O.jsd(to64(s), to64(t), 0.5, grad=False, threads=8)[0]
    assert_loss(to64(loss), rl, "after recovery")
