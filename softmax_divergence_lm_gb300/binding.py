"""Thin ctypes binding of libvpd (``include/vpd.h``), with the C names.

Every function here only marshals arguments: torch tensors become ``vpd_view``
/ ``vpd_grad`` descriptors holding device pointers, shapes and strides, and
the call runs on the current CUDA stream. All computation happens in the CUDA
kernels of ``libvpd.so``; there is no fallback. Loading fails loudly when the
library is missing (build it with ``python -m softmax_divergence_lm_gb300.build``).

Logits tensors may be 2-D ``[N, V]`` with unit stride along V (any row stride)
or 3-D ``[B, T, V]`` with unit stride along V (any batch and row strides, e.g.
the causal-shift view ``logits[:, :-1, :]``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

VPD_OK, VPD_ERR_ARG, VPD_ERR_DTYPE, VPD_ERR_SHAPE, VPD_ERR_INDEX, VPD_ERR_CUDA, VPD_ERR_TIMEOUT, \
    VPD_ERR_UNSUPPORTED = range(8)
VPD_F32, VPD_BF16, VPD_F16 = 0, 1, 2
VPD_MAX_SEGMENTS = 256
SAVED_PAIR, SAVED_ENTROPY, SAVED_LOGPROBS = 6, 3, 2

_DTYPES = {torch.float32: VPD_F32, torch.bfloat16: VPD_BF16, torch.float16: VPD_F16}

# every symbol declared in include/vpd.h
SYMBOLS = ("vpd_jsd_fwd", "vpd_jsd_bwd", "vpd_jsd_fwdbwd", "vpd_kl_fwd", "vpd_kl_bwd",
           "vpd_entropy_fwd", "vpd_entropy_bwd", "vpd_logprobs_fwd", "vpd_logprobs_bwd",
           "vpd_status_string", "vpd_last_error", "vpd_abi_version", "vpd_device_status",
           "vpd_launch_count", "vpd_test_withhold_copy", "vpd_jsd_linear_workspace", "vpd_jsd_linear_fwd",
           "vpd_jsd_linear_bwd", "vpd_jsd_linear_fwd_noalloc", "vpd_cross_entropy_fwd", "vpd_cross_entropy_bwd",
           "vpd_topk_kl_fwd", "vpd_topk_kl_bwd", "vpd_jsd_shard_stats", "vpd_jsd_shard_rescale",
           "vpd_jsd_shard_divergence", "vpd_jsd_shard_finish", "vpd_jsd_fwdbwd_teacher_stream", "vpd_jsd_plan")


class VpdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


class vpd_view(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("vocab", ctypes.c_int64), ("row_stride", ctypes.c_int64),
                ("rows_per_batch", ctypes.c_int64), ("batch_stride", ctypes.c_int64)]


class vpd_segments(ctypes.Structure):
    _fields_ = [("count", ctypes.c_int32), ("widths", ctypes.POINTER(ctypes.c_int64))]


class vpd_grad(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("row_stride", ctypes.c_int64)]


class vpd_linear_heads(ctypes.Structure):
    _fields_ = [("h_s", ctypes.c_void_p), ("w_s", ctypes.c_void_p), ("h_t", ctypes.c_void_p),
                ("w_t", ctypes.c_void_p), ("rows", ctypes.c_int64), ("vocab", ctypes.c_int64),
                ("hidden_s", ctypes.c_int64), ("hidden_t", ctypes.c_int64), ("ld_hs", ctypes.c_int64),
                ("ld_ws", ctypes.c_int64), ("ld_ht", ctypes.c_int64), ("ld_wt", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIBRARY


def load():
    """Load libvpd.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise ImportError(f"libvpd.so is not built ({path}); run "
                                  "`python -m softmax_divergence_lm_gb300.build`")
            _lib = _declare(ctypes.CDLL(path))
    return _lib


def _declare(lib):
    P = ctypes.POINTER
    V, S, G = P(vpd_view), P(vpd_segments), P(vpd_grad)
    f, vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    sig = {
        "vpd_jsd_fwd": [V, V, dbl, S, f, f, vp],
        "vpd_jsd_bwd": [V, V, dbl, S, f, f, G, G, vp],
        "vpd_jsd_fwdbwd": [V, V, dbl, S, f, f, f, G, G, vp],
        "vpd_kl_fwd": [V, V, i32, S, f, f, vp],
        "vpd_kl_bwd": [V, V, i32, S, f, f, G, G, vp],
        "vpd_entropy_fwd": [V, S, f, f, vp],
        "vpd_entropy_bwd": [V, S, f, f, G, vp],
        "vpd_logprobs_fwd": [V, S, f, i32, i64, f, f, f, vp],
        "vpd_logprobs_bwd": [V, S, f, i32, i64, f, f, G, vp],
        "vpd_device_status": [vp],
        "vpd_jsd_linear_workspace": [P(vpd_linear_heads), i32, i32, P(ctypes.c_size_t), P(ctypes.c_size_t)],
        "vpd_jsd_linear_fwd": [P(vpd_linear_heads), dbl, f, f, vp, ctypes.c_size_t, vp],
        "vpd_jsd_linear_bwd": [P(vpd_linear_heads), dbl, f, f, f, f, f, f, f, vp, ctypes.c_size_t, vp],
        "vpd_jsd_linear_fwd_noalloc": [P(vpd_linear_heads), dbl, f, f, vp],
        "vpd_cross_entropy_fwd": [V, S, f, i64, dbl, f, f, f, vp],
        "vpd_cross_entropy_bwd": [V, S, f, i64, dbl, f, f, G, vp],
        "vpd_topk_kl_fwd": [V, S, f, i32, i64, f, dbl, f, f, f, vp],
        "vpd_topk_kl_bwd": [V, S, f, i32, i64, f, dbl, f, f, G, vp],
        "vpd_jsd_shard_stats": [V, V, f, f, vp],
        "vpd_jsd_plan": [V, V, S, G, G, P(i64), P(i64), P(i32)],
        "vpd_jsd_fwdbwd_teacher_stream": [V, vp, i32, i64, dbl, f, f, f, G, G, vp, ctypes.c_size_t, i64, vp, vp],
        "vpd_jsd_shard_rescale": [i64, f, f, vp],
        "vpd_jsd_shard_divergence": [V, V, dbl, f, f, f, vp],
        "vpd_jsd_shard_finish": [i64, dbl, f, f, f, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.vpd_status_string.argtypes = [ctypes.c_int]
    lib.vpd_status_string.restype = ctypes.c_char_p
    lib.vpd_last_error.argtypes = []
    lib.vpd_last_error.restype = ctypes.c_char_p
    lib.vpd_abi_version.argtypes = []
    lib.vpd_abi_version.restype = ctypes.c_int32
    lib.vpd_launch_count.argtypes = []
    lib.vpd_launch_count.restype = ctypes.c_uint64
    lib.vpd_test_withhold_copy.argtypes = [ctypes.c_int64]
    lib.vpd_test_withhold_copy.restype = ctypes.c_int
    return lib


def _status_name(status: int) -> str:
    try:
        return load().vpd_status_string(status).decode()
    except Exception:  # noqa: BLE001 - naming only
        return f"status {status}"


def _check(status: int):
    if status != VPD_OK:
        raise VpdError(status, load().vpd_last_error().decode())


# ---------------------------------------------------------------------------
# Marshalling.
# ---------------------------------------------------------------------------
def _on_current_device(x: torch.Tensor, what: str):
    """The library launches on the current CUDA device: every tensor it is
    given must live there (a pointer into another GPU's memory would be read
    by kernels of this one)."""
    if not x.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if x.device.index != torch.cuda.current_device():
        raise ValueError(f"{what} is on {x.device}, the current device is cuda:{torch.cuda.current_device()}")


def _rows_vocab(view: vpd_view) -> tuple[int, int]:
    return int(view.rows), int(view.vocab)


def make_view(x: torch.Tensor) -> vpd_view:
    if x.dtype not in _DTYPES:
        raise TypeError(f"logits dtype {x.dtype} is not float32/bfloat16/float16")
    _on_current_device(x, "logits")
    if x.dim() == 2:
        n, v = x.shape
        if v > 1 and x.stride(1) != 1:
            raise ValueError("the vocabulary dimension must have unit stride")
        return vpd_view(x.data_ptr(), _DTYPES[x.dtype], n, v, x.stride(0) if n > 1 else v, 0, 0)
    if x.dim() == 3:
        b, t, v = x.shape
        if v > 1 and x.stride(2) != 1:
            raise ValueError("the vocabulary dimension must have unit stride")
        return vpd_view(x.data_ptr(), _DTYPES[x.dtype], b * t, v, x.stride(1) if t > 1 else v,
                        t, x.stride(0))
    raise ValueError("logits must be [N, V] or [B, T, V]")


def make_grad(g: torch.Tensor | None, rows: int | None = None, vocab: int | None = None) -> vpd_grad | None:
    """Gradient descriptor; with rows / vocab given, the tensor must be exactly
    [rows, vocab] (after flattening [B, T, V]), so that no row the kernels
    write lies past its allocation."""
    if g is None:
        return None
    if g.dtype not in _DTYPES:
        raise TypeError(f"gradient dtype {g.dtype} is not float32/bfloat16/float16")
    _on_current_device(g, "gradient")
    if g.dim() == 3:
        g = g.view(-1, g.shape[-1])
    if g.dim() != 2 or (g.shape[1] > 1 and g.stride(1) != 1):
        raise ValueError("gradient must be a dense [N, V] (or [B, T, V]) tensor with unit vocab stride")
    if rows is not None and (g.shape[0] != rows or g.shape[1] != vocab):
        raise ValueError(f"gradient shape {tuple(g.shape)} does not match the logits [{rows}, {vocab}]")
    return vpd_grad(g.data_ptr(), _DTYPES[g.dtype], g.stride(0) if g.shape[0] > 1 else g.shape[1])


def make_segments(widths) -> tuple[vpd_segments | None, object]:
    if widths is None:
        return None, None
    arr = (ctypes.c_int64 * len(widths))(*[int(w) for w in widths])
    return vpd_segments(len(widths), arr), arr  # keep arr alive alongside


def _fptr(t: torch.Tensor | None, numel: int | None = None, what: str = "per-row buffer"):
    """Device pointer of a contiguous float32 buffer of exactly `numel`
    elements (when given)."""
    if t is None:
        return None
    if t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous float32 CUDA tensor")
    _on_current_device(t, what)
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{what} has {t.numel()} elements, {numel} expected")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    dev = getattr(stream, "device", None)
    if dev is not None and getattr(dev, "index", None) is not None and dev.index != torch.cuda.current_device():
        raise ValueError(f"stream is on {dev}, the current device is cuda:{torch.cuda.current_device()}")
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _ref(x):
    return None if x is None else ctypes.byref(x)


# ---------------------------------------------------------------------------
# Entry points (same names and argument order as include/vpd.h). Each checks,
# before the call, that every buffer lives on the current device and has the
# size the kernels will read or write for the view's N, V (and k).
# ---------------------------------------------------------------------------
def _pair(s, t):
    vs, vt = make_view(s), make_view(t)
    n, v = _rows_vocab(vs)
    if _rows_vocab(vt) != (n, v):
        raise ValueError(f"student [{n}, {v}] and teacher {tuple(_rows_vocab(vt))} differ")
    return vs, vt, n, v


def vpd_jsd_fwd(s, t, beta, segments, loss, saved, stream=None):
    vs, vt, n, _ = _pair(s, t)
    seg, _keep = make_segments(segments)
    _check(load().vpd_jsd_fwd(ctypes.byref(vs), ctypes.byref(vt), float(beta), _ref(seg),
                              _fptr(loss, n, "loss"), _fptr(saved, n * SAVED_PAIR, "saved"), _stream(stream)))


def vpd_jsd_bwd(s, t, beta, segments, grad_loss, saved, ds, dt, stream=None):
    vs, vt, n, v = _pair(s, t)
    seg, _keep = make_segments(segments)
    gs, gt = make_grad(ds, n, v), make_grad(dt, n, v)
    _check(load().vpd_jsd_bwd(ctypes.byref(vs), ctypes.byref(vt), float(beta), _ref(seg),
                              _fptr(grad_loss, n, "grad_loss"), _fptr(saved, n * SAVED_PAIR, "saved"),
                              _ref(gs), _ref(gt), _stream(stream)))


def vpd_jsd_fwdbwd(s, t, beta, segments, grad_loss, loss, saved, ds, dt, stream=None):
    vs, vt, n, v = _pair(s, t)
    seg, _keep = make_segments(segments)
    gs, gt = make_grad(ds, n, v), make_grad(dt, n, v)
    _check(load().vpd_jsd_fwdbwd(ctypes.byref(vs), ctypes.byref(vt), float(beta), _ref(seg),
                                 _fptr(grad_loss, n, "grad_loss"), _fptr(loss, n, "loss"),
                                 _fptr(saved, n * SAVED_PAIR, "saved"), _ref(gs), _ref(gt), _stream(stream)))


def vpd_kl_fwd(s, t, reverse, segments, loss, saved, stream=None):
    vs, vt, n, _ = _pair(s, t)
    seg, _keep = make_segments(segments)
    _check(load().vpd_kl_fwd(ctypes.byref(vs), ctypes.byref(vt), int(bool(reverse)), _ref(seg),
                             _fptr(loss, n, "loss"), _fptr(saved, n * SAVED_PAIR, "saved"), _stream(stream)))


def vpd_kl_bwd(s, t, reverse, segments, grad_loss, saved, ds, dt, stream=None):
    vs, vt, n, v = _pair(s, t)
    seg, _keep = make_segments(segments)
    gs, gt = make_grad(ds, n, v), make_grad(dt, n, v)
    _check(load().vpd_kl_bwd(ctypes.byref(vs), ctypes.byref(vt), int(bool(reverse)), _ref(seg),
                             _fptr(grad_loss, n, "grad_loss"), _fptr(saved, n * SAVED_PAIR, "saved"),
                             _ref(gs), _ref(gt), _stream(stream)))


def vpd_entropy_fwd(x, segments, out, saved, stream=None):
    vx = make_view(x)
    n, _ = _rows_vocab(vx)
    seg, _keep = make_segments(segments)
    _check(load().vpd_entropy_fwd(ctypes.byref(vx), _ref(seg), _fptr(out, n, "out"),
                                  _fptr(saved, n * SAVED_ENTROPY, "saved"), _stream(stream)))


def vpd_entropy_bwd(x, segments, grad_out, saved, dx, stream=None):
    vx = make_view(x)
    n, v = _rows_vocab(vx)
    seg, _keep = make_segments(segments)
    gx = make_grad(dx, n, v)
    _check(load().vpd_entropy_bwd(ctypes.byref(vx), _ref(seg), _fptr(grad_out, n, "grad_out"),
                                  _fptr(saved, n * SAVED_ENTROPY, "saved"), _ref(gx), _stream(stream)))


def _index_ptr(index: torch.Tensor, numel: int):
    if index.dtype != torch.int64 or not index.is_contiguous():
        raise ValueError("index must be a contiguous int64 CUDA tensor")
    _on_current_device(index, "index")
    if index.numel() != numel:
        raise ValueError(f"index has {index.numel()} elements, {numel} expected")
    return index.data_ptr()


def vpd_logprobs_fwd(x, segments, index, k, ignore_index, out, saved, err_flag, stream=None):
    """err_flag: int32 CUDA tensor, or None (the library then checks the
    indices on the host and raises VPD_ERR_INDEX before launching)."""
    vx = make_view(x)
    n, _ = _rows_vocab(vx)
    seg, _keep = make_segments(segments)
    if err_flag is not None:
        if err_flag.dtype != torch.int32 or err_flag.numel() < 1:
            raise ValueError("err_flag must be an int32 CUDA tensor of at least one element, or None")
        _on_current_device(err_flag, "err_flag")
    _check(load().vpd_logprobs_fwd(ctypes.byref(vx), _ref(seg), _index_ptr(index, n * int(k)), int(k),
                                   int(ignore_index), _fptr(out, n * int(k), "out"),
                                   _fptr(saved, n * SAVED_LOGPROBS, "saved"),
                                   err_flag.data_ptr() if err_flag is not None else None, _stream(stream)))


def vpd_logprobs_bwd(x, segments, index, k, ignore_index, grad_out, saved, dx, stream=None):
    vx = make_view(x)
    n, v = _rows_vocab(vx)
    seg, _keep = make_segments(segments)
    gx = make_grad(dx, n, v)
    _check(load().vpd_logprobs_bwd(ctypes.byref(vx), _ref(seg), _index_ptr(index, n * int(k)), int(k),
                                   int(ignore_index), _fptr(grad_out, n * int(k), "grad_out"),
                                   _fptr(saved, n * SAVED_LOGPROBS, "saved"), _ref(gx), _stream(stream)))


def make_heads(h_s, w_s, h_t, w_t) -> vpd_linear_heads:
    """Descriptor of two bf16 linear heads: hidden states [N, H] and head
    weights [V, H] with unit stride along H, all on the current device."""
    for x, what in ((h_s, "h_s"), (w_s, "w_s"), (h_t, "h_t"), (w_t, "w_t")):
        if x.dtype != torch.bfloat16 or x.dim() != 2 or (x.shape[1] > 1 and x.stride(1) != 1):
            raise ValueError(f"{what} must be a bf16 [rows, hidden] tensor with unit stride along hidden")
        _on_current_device(x, what)
    if h_s.shape[1] != w_s.shape[1] or h_t.shape[1] != w_t.shape[1]:
        raise ValueError("hidden sizes of the hidden states and their head differ")
    if h_s.shape[0] != h_t.shape[0] or w_s.shape[0] != w_t.shape[0]:
        raise ValueError("student and teacher must share rows and vocabulary")
    ld = lambda x: x.stride(0) if x.shape[0] > 1 else x.shape[1]  # noqa: E731
    return vpd_linear_heads(h_s.data_ptr(), w_s.data_ptr(), h_t.data_ptr(), w_t.data_ptr(), h_s.shape[0],
                            w_s.shape[0], h_s.shape[1], h_t.shape[1], ld(h_s), ld(w_s), ld(h_t), ld(w_t))


def vpd_jsd_linear_workspace(heads: vpd_linear_heads, student_grads=True, teacher_grads=False) -> tuple[int, int]:
    f, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().vpd_jsd_linear_workspace(ctypes.byref(heads), int(bool(student_grads)), int(bool(teacher_grads)),
                                           ctypes.byref(f), ctypes.byref(b)))
    return int(f.value), int(b.value)


def _workspace(ws: torch.Tensor | None, need: int):
    if ws is None:
        raise ValueError("a workspace tensor is required")
    _on_current_device(ws, "workspace")
    nbytes = ws.numel() * ws.element_size()
    if not ws.is_contiguous() or nbytes < need:
        raise ValueError(f"workspace must be a contiguous tensor of at least {need} bytes")
    return ws.data_ptr(), nbytes


def vpd_jsd_linear_fwd(heads: vpd_linear_heads, beta, loss, saved, workspace, stream=None):
    n = int(heads.rows)
    need, _ = vpd_jsd_linear_workspace(heads, False, False)
    wp, wn = _workspace(workspace, need)
    _check(load().vpd_jsd_linear_fwd(ctypes.byref(heads), float(beta), _fptr(loss, n, "loss"),
                                     _fptr(saved, n * SAVED_PAIR, "saved"), wp, wn, _stream(stream)))


def vpd_jsd_linear_fwd_noalloc(heads: vpd_linear_heads, beta, loss, saved, stream=None):
    """vpd_jsd_linear_fwd without a workspace argument, for callers that may not
    allocate device memory (the library's built-in scratch array is used; calls
    that overlap on the GPU must not share it)."""
    n = int(heads.rows)
    _check(load().vpd_jsd_linear_fwd_noalloc(ctypes.byref(heads), float(beta), _fptr(loss, n, "loss"),
                                             _fptr(saved, n * SAVED_PAIR, "saved"), _stream(stream)))


def vpd_jsd_linear_bwd(heads: vpd_linear_heads, beta, grad_loss, loss, saved, dh_s, dw_s, dh_t, dw_t, workspace,
                       stream=None):
    n, v = int(heads.rows), int(heads.vocab)
    hs, ht = int(heads.hidden_s), int(heads.hidden_t)
    _, need = vpd_jsd_linear_workspace(heads, dh_s is not None or dw_s is not None,
                                       dh_t is not None or dw_t is not None)
    wp, wn = _workspace(workspace, need)
    _check(load().vpd_jsd_linear_bwd(ctypes.byref(heads), float(beta), _fptr(grad_loss, n, "grad_loss"),
                                     _fptr(loss, n, "loss"), _fptr(saved, n * SAVED_PAIR, "saved"),
                                     _fptr(dh_s, n * hs, "dh_s"), _fptr(dw_s, v * hs, "dw_s"),
                                     _fptr(dh_t, n * ht, "dh_t"), _fptr(dw_t, v * ht, "dw_t"), wp, wn,
                                     _stream(stream)))


def _flag_ptr(err_flag):
    if err_flag is None:
        return None
    if err_flag.dtype != torch.int32 or err_flag.numel() < 1:
        raise ValueError("err_flag must be an int32 CUDA tensor of at least one element, or None")
    _on_current_device(err_flag, "err_flag")
    return err_flag.data_ptr()


def vpd_cross_entropy_fwd(x, segments, labels, ignore_index, temperature, loss, saved, err_flag, stream=None):
    vx = make_view(x)
    n, _ = _rows_vocab(vx)
    seg, _keep = make_segments(segments)
    _check(load().vpd_cross_entropy_fwd(ctypes.byref(vx), _ref(seg), _index_ptr(labels, n), int(ignore_index),
                                        float(temperature), _fptr(loss, n, "loss"),
                                        _fptr(saved, n * SAVED_LOGPROBS, "saved"), _flag_ptr(err_flag),
                                        _stream(stream)))


def vpd_cross_entropy_bwd(x, segments, labels, ignore_index, temperature, grad_loss, saved, dx, stream=None):
    vx = make_view(x)
    n, v = _rows_vocab(vx)
    seg, _keep = make_segments(segments)
    gx = make_grad(dx, n, v)
    _check(load().vpd_cross_entropy_bwd(ctypes.byref(vx), _ref(seg), _index_ptr(labels, n), int(ignore_index),
                                        float(temperature), _fptr(grad_loss, n, "grad_loss"),
                                        _fptr(saved, n * SAVED_LOGPROBS, "saved"), _ref(gx), _stream(stream)))


def vpd_topk_kl_fwd(s, segments, index, k, ignore_index, teacher_logp, temperature, kl, saved, err_flag,
                    stream=None):
    vs = make_view(s)
    n, _ = _rows_vocab(vs)
    seg, _keep = make_segments(segments)
    _check(load().vpd_topk_kl_fwd(ctypes.byref(vs), _ref(seg), _index_ptr(index, n * int(k)), int(k),
                                  int(ignore_index), _fptr(teacher_logp, n * int(k), "teacher_logp"),
                                  float(temperature), _fptr(kl, n, "kl"), _fptr(saved, n * SAVED_LOGPROBS, "saved"),
                                  _flag_ptr(err_flag), _stream(stream)))


def vpd_topk_kl_bwd(s, segments, index, k, ignore_index, teacher_logp, temperature, grad_kl, saved, ds,
                    stream=None):
    vs = make_view(s)
    n, v = _rows_vocab(vs)
    seg, _keep = make_segments(segments)
    gs = make_grad(ds, n, v)
    _check(load().vpd_topk_kl_bwd(ctypes.byref(vs), _ref(seg), _index_ptr(index, n * int(k)), int(k),
                                  int(ignore_index), _fptr(teacher_logp, n * int(k), "teacher_logp"),
                                  float(temperature), _fptr(grad_kl, n, "grad_kl"),
                                  _fptr(saved, n * SAVED_LOGPROBS, "saved"), _ref(gs), _stream(stream)))


def vpd_jsd_shard_stats(s, t, saved, xbuf, stream=None):
    vs, vt, n, _ = _pair(s, t)
    _check(load().vpd_jsd_shard_stats(ctypes.byref(vs), ctypes.byref(vt), _fptr(saved, n * SAVED_PAIR, "saved"),
                                      _fptr(xbuf, n * 2, "xbuf"), _stream(stream)))


def vpd_jsd_shard_rescale(rows, saved, xbuf, stream=None):
    n = int(rows)
    _check(load().vpd_jsd_shard_rescale(n, _fptr(saved, n * SAVED_PAIR, "saved"), _fptr(xbuf, n * 2, "xbuf"),
                                        _stream(stream)))


def vpd_jsd_shard_divergence(s, t, beta, loss, saved, xbuf, stream=None):
    vs, vt, n, _ = _pair(s, t)
    _check(load().vpd_jsd_shard_divergence(ctypes.byref(vs), ctypes.byref(vt), float(beta), _fptr(loss, n, "loss"),
                                           _fptr(saved, n * SAVED_PAIR, "saved"), _fptr(xbuf, n * 2, "xbuf"),
                                           _stream(stream)))


def vpd_jsd_shard_finish(rows, beta, saved, xbuf, loss, stream=None):
    n = int(rows)
    _check(load().vpd_jsd_shard_finish(n, float(beta), _fptr(saved, n * SAVED_PAIR, "saved"),
                                       _fptr(xbuf, n * 2, "xbuf"), _fptr(loss, n, "loss"), _stream(stream)))


def vpd_jsd_fwdbwd_teacher_stream(s, t_host, beta, grad_loss, loss, saved, ds, dt, staging, chunk_rows,
                                  stream=None, copy_stream=None):
    """t_host: a pinned CPU tensor [N, V] (unit stride along V) of the
    student's dtype; staging: a device tensor of at least two chunks."""
    vs = make_view(s)
    n, v = _rows_vocab(vs)
    if vs.rows_per_batch:
        raise ValueError("the student must be a plain 2-D [N, V] view")
    if t_host.is_cuda or t_host.dtype != s.dtype or t_host.dim() != 2 or tuple(t_host.shape) != (n, v):
        raise ValueError("t_host must be a CPU tensor of the student's dtype and shape")
    if v > 1 and t_host.stride(1) != 1:
        raise ValueError("t_host must have unit stride along the vocabulary")
    if not t_host.is_pinned():
        raise ValueError("t_host must be pinned host memory")
    gs, gt = make_grad(ds, n, v), make_grad(dt, n, v)
    if copy_stream is None:
        raise ValueError("a copy stream distinct from the compute stream is required")
    _on_current_device(staging, "staging")
    _check(load().vpd_jsd_fwdbwd_teacher_stream(
        ctypes.byref(vs), t_host.data_ptr(), _DTYPES[t_host.dtype], t_host.stride(0) if n > 1 else v, float(beta),
        _fptr(grad_loss, n, "grad_loss"), _fptr(loss, n, "loss"), _fptr(saved, n * SAVED_PAIR, "saved"),
        _ref(gs), _ref(gt), staging.data_ptr(), staging.numel() * staging.element_size(), int(chunk_rows),
        _stream(stream), _stream(copy_stream)))


def vpd_jsd_plan(s, t, segments=None, ds=None, dt=None) -> tuple[int, int, int]:
    """(rows on the single-read kernel, rows on the idle SMs, launches) of a
    vpd_jsd_fwd (no gradients given) or vpd_jsd_fwdbwd call with these
    arguments; nothing is launched."""
    vs, vt, n, v = _pair(s, t)
    seg, _keep = make_segments(segments)
    gs, gt = make_grad(ds, n, v), make_grad(dt, n, v)
    fr, side, k = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    _check(load().vpd_jsd_plan(ctypes.byref(vs), ctypes.byref(vt), _ref(seg), _ref(gs), _ref(gt), ctypes.byref(fr),
                               ctypes.byref(side), ctypes.byref(k)))
    return int(fr.value), int(side.value), int(k.value)


def vpd_device_status(stream=None):
    _check(load().vpd_device_status(_stream(stream)))


def vpd_abi_version() -> int:
    return int(load().vpd_abi_version())


def vpd_launch_count() -> int:
    return int(load().vpd_launch_count())


def vpd_test_withhold_copy(row: int):
    _check(load().vpd_test_withhold_copy(int(row)))
