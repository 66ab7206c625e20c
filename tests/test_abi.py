"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every
symbol ``include/vpd.h`` declares, and rejects bad arguments on the host before
any CUDA call (no compute call is made here)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from softmax_divergence_lm_gb300 import binding as B
from softmax_divergence_lm_gb300 import build

HEADER = os.path.join(build.ROOT, "include", "vpd.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vpd_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(B.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.vpd_abi_version() == 1
    assert lib.vpd_status_string(B.VPD_ERR_SHAPE) == b"VPD_ERR_SHAPE"


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "library_path", lambda: "/nonexistent/libvpd.so")
    with pytest.raises(ImportError):
        B.load()


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def view(rows=4, vocab=16, dtype=B.VPD_F32, stride=None, data=FAKE, rpb=0, bstride=0):
    return B.vpd_view(data, dtype, rows, vocab, vocab if stride is None else stride, rpb, bstride)


def jsd_fwd(lib, s, t, beta=0.5, seg=None, loss=FAKE, saved=FAKE):
    return lib.vpd_jsd_fwd(ctypes.byref(s), ctypes.byref(t), beta, None if seg is None else ctypes.byref(seg),
                           loss, saved, None)


def segs(widths):
    arr = (ctypes.c_int64 * len(widths))(*widths)
    return B.vpd_segments(len(widths), arr), arr


@pytest.mark.parametrize("case,expect", [
    ("rows differ", B.VPD_ERR_SHAPE),
    ("vocab differ", B.VPD_ERR_SHAPE),
    ("dtypes differ", B.VPD_ERR_DTYPE),
    ("unknown dtype", B.VPD_ERR_DTYPE),
    ("beta above 1", B.VPD_ERR_ARG),
    ("beta negative", B.VPD_ERR_ARG),
    ("beta nan", B.VPD_ERR_ARG),
    ("stride below vocab", B.VPD_ERR_SHAPE),
    ("misaligned bf16", B.VPD_ERR_ARG),
    ("null data", B.VPD_ERR_ARG),
    ("null loss", B.VPD_ERR_ARG),
    ("null saved", B.VPD_ERR_ARG),
    ("negative rows", B.VPD_ERR_SHAPE),
])
def test_jsd_fwd_validation(lib, case, expect):
    s, t, beta, kw = view(), view(), 0.5, {}
    if case == "rows differ":
        t = view(rows=5)
    elif case == "vocab differ":
        t = view(vocab=17)
    elif case == "dtypes differ":
        t = view(dtype=B.VPD_BF16)
    elif case == "unknown dtype":
        s = t = view(dtype=9)
    elif case == "beta above 1":
        beta = 1.5
    elif case == "beta negative":
        beta = -0.1
    elif case == "beta nan":
        beta = float("nan")
    elif case == "stride below vocab":
        s = view(stride=8)
    elif case == "misaligned bf16":
        s, t = view(dtype=B.VPD_BF16, data=FAKE + 1), view(dtype=B.VPD_BF16)
    elif case == "null data":
        s = view(data=None)
    elif case == "null loss":
        kw = {"loss": None}
    elif case == "null saved":
        kw = {"saved": None}
    elif case == "negative rows":
        s = t = view(rows=-1)
    st = jsd_fwd(lib, s, t, beta, **kw)
    assert st == expect, (case, st, lib.vpd_last_error())
    assert lib.vpd_last_error()


@pytest.mark.parametrize("widths,expect", [
    ([8, 9], B.VPD_ERR_SHAPE),      # sums to 17, vocab is 16
    ([20, -4], B.VPD_ERR_SHAPE),    # negative width
    ([0] * 257, B.VPD_ERR_ARG),     # too many segments
])
def test_segment_validation(lib, widths, expect):
    sg, _keep = segs(widths)
    assert jsd_fwd(lib, view(), view(), seg=sg) == expect


def test_null_widths_rejected(lib):
    sg = B.vpd_segments(3, None)
    assert jsd_fwd(lib, view(), view(), seg=sg) == B.VPD_ERR_ARG


def test_empty_batch_is_a_noop_without_device_work(lib):
    # N = 0 returns before any CUDA call, so it succeeds even without a GPU
    assert jsd_fwd(lib, view(rows=0), view(rows=0), loss=None, saved=None) == B.VPD_OK


def test_gradient_validation(lib):
    s = view()
    saved = FAKE
    bad_stride = B.vpd_grad(FAKE, B.VPD_F32, 8)
    st = lib.vpd_jsd_bwd(ctypes.byref(s), ctypes.byref(s), 0.5, None, None, saved, ctypes.byref(bad_stride),
                         None, None)
    assert st == B.VPD_ERR_SHAPE
    mixed_a = B.vpd_grad(FAKE, B.VPD_F32, 16)
    mixed_b = B.vpd_grad(FAKE, B.VPD_BF16, 16)
    st = lib.vpd_jsd_bwd(ctypes.byref(s), ctypes.byref(s), 0.5, None, None, saved, ctypes.byref(mixed_a),
                         ctypes.byref(mixed_b), None)
    assert st == B.VPD_ERR_DTYPE
    st = lib.vpd_jsd_bwd(ctypes.byref(s), ctypes.byref(s), 0.5, None, None, None, ctypes.byref(mixed_a), None,
                         None)
    assert st == B.VPD_ERR_ARG  # saved is required


def test_logprobs_validation(lib):
    x = view()
    assert lib.vpd_logprobs_fwd(ctypes.byref(x), None, FAKE, 0, -100, FAKE, None, FAKE, None) == B.VPD_ERR_ARG
    # err_flag may be NULL (the indices are then checked on the host); a
    # missing index array is still an argument error, before any CUDA call
    assert lib.vpd_logprobs_fwd(ctypes.byref(x), None, None, 2, -100, FAKE, None, None, None) == B.VPD_ERR_ARG
