"""The workspace-free fused-linear forward, vpd_jsd_linear_fwd_noalloc.

Some callers cannot allocate device memory for an op: an engine that owns all
device memory and hands each op only its inputs and outputs, or a
latency-critical loop where cudaMalloc / cudaFree would stall the device. For
them this entry point keeps its scratch in an array built into the library.
The test calls it through the C ABI twice in a row (the second call finds the
first call's contents in the array) and compares both results with the
workspace entry point, vpd_jsd_linear_fwd, within the tolerances the other
tests use (per-token loss 1e-6 + 1e-5 |ref|). It sits in a file of its own,
collected last."""
from __future__ import annotations

import numpy as np
import pytest
import torch

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


def _forward_with_workspace(B, heads, n, beta):
    fwd_b, _ = B.vpd_jsd_linear_workspace(heads, False, False)
    ws = torch.empty(fwd_b, dtype=torch.uint8, device="cuda")
    loss = torch.empty(n, device="cuda")
    saved = torch.empty(n, 6, device="cuda")
    B.vpd_jsd_linear_fwd(heads, beta, loss, saved, ws)
    torch.cuda.synchronize()
    return loss, saved


def test_no_alloc_forward_matches_workspace_forward_twice(B):
    from softmax_divergence_lm_gb300 import synth
    cases = []
    for seed, (n, v, hs, ht) in ((21, (700, 2000, 128, 192)), (22, (300, 1000, 64, 128))):
        h_s, w_s, h_t, w_t = synth.linear_heads(device="cuda", n=n, v=v, hidden_s=hs, hidden_t=ht, seed=seed)
        cases.append((B.make_heads(h_s, w_s, h_t, w_t), n, (h_s, w_s, h_t, w_t)))
    # two calls in a row on different problems: the second reads nothing stale
    for (heads, n, keep), beta in zip(cases, (0.5, 0.0)):
        ref_loss, ref_saved = _forward_with_workspace(B, heads, n, beta)
        loss = torch.full((n,), 7.0, device="cuda")
        saved = torch.full((n, 6), 7.0, device="cuda")
        B.vpd_jsd_linear_fwd_noalloc(heads, beta, loss, saved)
        torch.cuda.synchronize()
        B.vpd_device_status()
        assert_loss(to64(loss), to64(ref_loss), f"no-alloc forward beta={beta} loss")
        sv, rsv = to64(saved), to64(ref_saved)
        for col in range(6):
            assert_loss(sv[:, col], rsv[:, col], f"no-alloc forward beta={beta} saved[:, {col}]")
        assert np.all(np.isfinite(sv[:, :4]))


def test_no_alloc_forward_fewer_chunks_at_qwen_heads(B):
    """16384 rows of the Qwen heads: the fastest plan's partials exceed the
    built-in array, so the no-alloc forward runs with fewer, longer vocabulary
    chunks; same results as the workspace forward within the loss tolerance."""
    from softmax_divergence_lm_gb300 import synth
    n = 16384
    h_s, w_s, h_t, w_t = synth.linear_heads(device="cuda", n=n, seed=23)
    heads = B.make_heads(h_s, w_s, h_t, w_t)
    fwd_b, _ = B.vpd_jsd_linear_workspace(heads, False, False)
    assert fwd_b > 4 << 20 >= 32 * n
    ref_loss, ref_saved = _forward_with_workspace(B, heads, n, 0.5)
    loss = torch.full((n,), 7.0, device="cuda")
    saved = torch.full((n, 6), 7.0, device="cuda")
    B.vpd_jsd_linear_fwd_noalloc(heads, 0.5, loss, saved)
    torch.cuda.synchronize()
    B.vpd_device_status()
    assert_loss(to64(loss), to64(ref_loss), "no-alloc forward, 16384 rows, loss")
    sv, rsv = to64(saved), to64(ref_saved)
    for col in range(6):
        assert_loss(sv[:, col], rsv[:, col], f"no-alloc forward, 16384 rows, saved[:, {col}]")


def test_no_alloc_forward_rejects_oversized_problem(B):
    """A problem whose scratch would not fit the built-in array even with the
    vocabulary in one chunk (more than 131072 rows) is refused on the host with
    VPD_ERR_SHAPE (nothing is launched, nothing is read)."""
    heads = B.vpd_linear_heads(0x10000, 0x10000, 0x10000, 0x10000, 1 << 20, 151936, 896, 1536, 896, 896, 1536, 1536)
    fwd_b, _ = B.vpd_jsd_linear_workspace(heads, False, False)
    assert fwd_b > 4 << 20
    with pytest.raises(B.VpdError) as info:
        B.vpd_jsd_linear_fwd_noalloc(heads, 0.5, torch.empty(1 << 20, device="cuda"),
                                     torch.empty(1 << 20, 6, device="cuda"))
    assert info.value.status == B.VPD_ERR_SHAPE
