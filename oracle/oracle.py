"""Python access to the CPU oracle in ``vpd_oracle.c``, in double precision
or, on request, in the host's long double.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers allowed. The product path never imports
this module, and this module imports nothing from the product package.

The C source is compiled with the host compiler (``gcc -O2``, no fast-math) into
``oracle/_build/``; :func:`build` does it explicitly, and the first call to any
function does it on demand. Inputs are any array-likes convertible exactly to
float64 (fp32/bf16/fp16 values upcast exactly); outputs are float64 numpy
arrays. Every function runs one token row at a time over the full vocabulary;
``threads > 1`` only splits the rows over host threads (the C calls release
the interpreter lock).

The same source builds twice: ``libvpd_oracle.so`` works in double, and
``libvpd_oracle_ld.so`` (the source compiled with ``VPD_ORACLE_LONG_DOUBLE``)
carries every intermediate in long double (x86-64: 64-bit significand; AArch64:
113-bit), rounding once to float64 at the output. The row functions take
``precision="double"`` (default) or ``"long double"``; the second is a check on
the first's rounding, not a different definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "vpd_oracle.c")
LIBRARY = os.path.join(_HERE, "_build", "libvpd_oracle.so")
LIBRARY_LONG_DOUBLE = os.path.join(_HERE, "_build", "libvpd_oracle_ld.so")
PRECISIONS = ("double", "long double")

_lock = threading.Lock()
_lib = None
_lib_ld = None

_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def _check_precision(precision: str) -> None:
    if precision not in PRECISIONS:
        raise ValueError(f"precision must be one of {PRECISIONS}, not {precision!r}")


def compile_command(source: str = SOURCE, output: str = LIBRARY, precision: str = "double") -> list[str]:
    """The host-compiler command that builds the oracle library."""
    _check_precision(precision)
    defines = ["-DVPD_ORACLE_LONG_DOUBLE"] if precision == "long double" else []
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", *defines, "-o", output, source, "-lm"]


def build(force: bool = False, source: str = SOURCE, output: str | None = None,
          precision: str = "double") -> str:
    """Compile the oracle if the library is missing or older than its source."""
    _check_precision(precision)
    if output is None:
        output = LIBRARY_LONG_DOUBLE if precision == "long double" else LIBRARY
    os.makedirs(os.path.dirname(output), exist_ok=True)
    stale = (not os.path.exists(output)) or os.path.getmtime(output) < os.path.getmtime(source)
    if force or stale:
        tmp = output + f".tmp{os.getpid()}"
        subprocess.run(compile_command(source, tmp, precision), check=True)
        os.replace(tmp, output)
    return output


def load(path: str | None = None, precision: str = "double"):
    """Load (building first if needed) and return the ctypes handle."""
    global _lib, _lib_ld
    _check_precision(precision)
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if precision == "long double":
            if _lib_ld is None:
                _lib_ld = _declare(ctypes.CDLL(build(precision=precision)))
            return _lib_ld
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(lib):
    lib.vpd_oracle_row_stats.argtypes = [ctypes.c_int64, _f64p, _f64p, _f64p]
    lib.vpd_oracle_row_stats.restype = ctypes.c_int
    lib.vpd_oracle_segment_stats.argtypes = [ctypes.c_int64, _f64p, ctypes.c_int, _i64p, _f64p, _f64p]
    lib.vpd_oracle_segment_stats.restype = ctypes.c_int
    lib.vpd_oracle_jsd.argtypes = [ctypes.c_int64, ctypes.c_int64, _f64p, _f64p, ctypes.c_double,
                                   _f64p, _f64p, _f64p, _f64p, _f64p, _f64p]
    lib.vpd_oracle_jsd.restype = None
    lib.vpd_oracle_kl.argtypes = [ctypes.c_int64, ctypes.c_int64, _f64p, _f64p, ctypes.c_int,
                                  _f64p, _f64p, _f64p, _f64p]
    lib.vpd_oracle_kl.restype = None
    lib.vpd_oracle_entropy.argtypes = [ctypes.c_int64, ctypes.c_int64, _f64p, _f64p, _f64p, _f64p]
    lib.vpd_oracle_entropy.restype = None
    lib.vpd_oracle_logprobs.argtypes = [ctypes.c_int64, ctypes.c_int64, _f64p, ctypes.c_int64, _i64p,
                                        ctypes.c_int64, _f64p, _f64p, _f64p]
    lib.vpd_oracle_logprobs.restype = ctypes.c_int64
    return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    if a.dtype == np.int64:
        return a.ctypes.data_as(_i64p)
    return a.ctypes.data_as(_f64p)


def _rows2d(x) -> np.ndarray:
    x = _f64(x)
    if x.ndim == 1:
        x = x[None, :]
    if x.ndim != 2:
        raise ValueError("oracle inputs are [N, V]")
    return x


def _split(n: int, threads: int):
    threads = max(1, min(threads, n))
    step = (n + threads - 1) // threads if n else 0
    return [(a, min(a + step, n)) for a in range(0, n, step)] if n else []


def _run(n: int, threads: int, fn):
    parts = _split(n, threads)
    if len(parts) <= 1:
        for a, b in parts:
            fn(a, b)
        return
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        list(ex.map(lambda ab: fn(*ab), parts))


def row_stats(x, precision: str = "double"):
    """(m, lse, code) per row: max over the finite support, log of the sum-exp
    relative to it, and 0 / 1 (NaN or +inf present) / 2 (fully -inf)."""
    lib = load(precision=precision)
    x = _rows2d(x)
    n, v = x.shape
    m = np.empty(n)
    lse = np.empty(n)
    code = np.empty(n, dtype=np.int64)
    for r in range(n):
        mr = ctypes.c_double()
        lr = ctypes.c_double()
        code[r] = lib.vpd_oracle_row_stats(v, _ptr(x[r]), ctypes.byref(mr), ctypes.byref(lr))
        m[r], lse[r] = mr.value, lr.value
    return m, lse, code


def segment_stats(x, widths, precision: str = "double"):
    """Statistics (m, Z) of one row merged over ordered segments."""
    lib = load(precision=precision)
    x = _f64(x).reshape(-1)
    w = np.ascontiguousarray(np.asarray(widths, dtype=np.int64))
    m = ctypes.c_double()
    z = ctypes.c_double()
    rc = lib.vpd_oracle_segment_stats(x.size, _ptr(x), int(w.size), _ptr(w), ctypes.byref(m), ctypes.byref(z))
    if rc:
        raise ValueError("segment widths must be >= 0 and sum to the vocabulary size")
    return m.value, z.value


def jsd(s, t, beta: float, g=None, grad: bool = True, threads: int = 1, precision: str = "double"):
    """Generalized JSD per row. Returns (loss, kl_tm, kl_sm, ds, dt); kl_tm and
    kl_sm are KL(P_t||M) and KL(P_s||M) (NaN on the beta = 0 / 1 branches);
    ds, dt are None when grad is False."""
    lib = load(precision=precision)
    s = _rows2d(s)
    t = _rows2d(t)
    if s.shape != t.shape:
        raise ValueError("student and teacher must have the same [N, V] shape")
    n, v = s.shape
    g = None if g is None else _f64(g).reshape(n)
    loss, a, b = np.empty(n), np.empty(n), np.empty(n)
    ds = np.empty((n, v)) if grad else None
    dt = np.empty((n, v)) if grad else None

    def part(r0, r1):
        sl = slice(r0, r1)
        lib.vpd_oracle_jsd(r1 - r0, v, _ptr(s[sl]), _ptr(t[sl]), float(beta),
                           None if g is None else _ptr(g[sl]), _ptr(loss[sl]), _ptr(a[sl]),
                           _ptr(b[sl]), None if ds is None else _ptr(ds[sl]),
                           None if dt is None else _ptr(dt[sl]))

    _run(n, threads, part)
    return loss, a, b, ds, dt


def kl(s, t, reverse: bool, g=None, grad: bool = True, threads: int = 1, precision: str = "double"):
    """KL(P_t||P_s) (reverse False) or KL(P_s||P_t) (reverse True) per row.
    Returns (loss, ds, dt)."""
    lib = load(precision=precision)
    s = _rows2d(s)
    t = _rows2d(t)
    if s.shape != t.shape:
        raise ValueError("student and teacher must have the same [N, V] shape")
    n, v = s.shape
    g = None if g is None else _f64(g).reshape(n)
    loss = np.empty(n)
    ds = np.empty((n, v)) if grad else None
    dt = np.empty((n, v)) if grad else None

    def part(r0, r1):
        sl = slice(r0, r1)
        lib.vpd_oracle_kl(r1 - r0, v, _ptr(s[sl]), _ptr(t[sl]), int(bool(reverse)),
                          None if g is None else _ptr(g[sl]), _ptr(loss[sl]),
                          None if ds is None else _ptr(ds[sl]), None if dt is None else _ptr(dt[sl]))

    _run(n, threads, part)
    return loss, ds, dt


def entropy(x, g=None, grad: bool = True, threads: int = 1, precision: str = "double"):
    """Entropy per row. Returns (out, dx)."""
    lib = load(precision=precision)
    x = _rows2d(x)
    n, v = x.shape
    g = None if g is None else _f64(g).reshape(n)
    out = np.empty(n)
    dx = np.empty((n, v)) if grad else None

    def part(r0, r1):
        sl = slice(r0, r1)
        lib.vpd_oracle_entropy(r1 - r0, v, _ptr(x[sl]), None if g is None else _ptr(g[sl]),
                               _ptr(out[sl]), None if dx is None else _ptr(dx[sl]))

    _run(n, threads, part)
    return out, dx


def logprobs(x, index, ignore_index: int = -100, g=None, grad: bool = True, threads: int = 1,
             precision: str = "double"):
    """Selected log-probs. index is [N] or [N, K]; returns (out [N, K], dx, errors)."""
    lib = load(precision=precision)
    x = _rows2d(x)
    n, v = x.shape
    idx = np.ascontiguousarray(np.asarray(index, dtype=np.int64)).reshape(n, -1)
    k = idx.shape[1]
    g = None if g is None else _f64(g).reshape(n, k)
    out = np.empty((n, k))
    dx = np.empty((n, v)) if grad else None
    errors = [0]
    err_lock = threading.Lock()

    def part(r0, r1):
        sl = slice(r0, r1)
        e = lib.vpd_oracle_logprobs(r1 - r0, v, _ptr(x[sl]), k, _ptr(idx[sl]), int(ignore_index),
                                    None if g is None else _ptr(g[sl]), _ptr(out[sl]),
                                    None if dx is None else _ptr(dx[sl]))
        with err_lock:
            errors[0] += int(e)

    _run(n, threads, part)
    return out, dx, errors[0]


# ---------------------------------------------------------------------------
# Compositions on the row oracles above. Each is the plain definition written
# out step by step in float64: a library matmul or an elementwise numpy step
# where the definition has one, then the row oracles for everything softmax.
# ---------------------------------------------------------------------------
def jsd_linear(h_s, w_s, h_t, w_t, beta: float, g=None, grad: bool = True, threads: int = 1):
    """Generalized JSD between the logits of two linear heads, s = h_s w_s^T and
    t = h_t w_t^T, the fused-linear divergence the pages name as missing ('[VocabTP]
    Add vocabulary-parallel generalized JSD with Triton kernels', section Scope
    and limitations; 'Add vocabulary-parallel logprobs, entropy and KL ops',
    section Limitations). Steps: (1) the logits in float64 from the exactly
    upcast inputs by a library matmul; (2) the JSD row oracle on them; (3) the
    chain rule through the linear maps: dh = dS w, dw = dS^T h (and the same
    for the teacher). Returns (loss, kl_tm, kl_sm, dh_s, dw_s, dh_t, dw_t)."""
    h_s, w_s, h_t, w_t = (_f64(a) for a in (h_s, w_s, h_t, w_t))
    if h_s.ndim != 2 or w_s.ndim != 2 or h_t.ndim != 2 or w_t.ndim != 2:
        raise ValueError("hidden states are [N, H] and head weights [V, H]")
    if h_s.shape[1] != w_s.shape[1] or h_t.shape[1] != w_t.shape[1]:
        raise ValueError("hidden size of a head and its hidden states differ")
    if h_s.shape[0] != h_t.shape[0] or w_s.shape[0] != w_t.shape[0]:
        raise ValueError("student and teacher must share N and V")
    s = h_s @ w_s.T
    t = h_t @ w_t.T
    loss, a, b, ds, dt = jsd(s, t, beta, g, grad=grad, threads=threads)
    if not grad:
        return loss, a, b, None, None, None, None
    return loss, a, b, ds @ w_s, ds.T @ h_s, dt @ w_t, dt.T @ h_t


def cross_entropy(x, labels, ignore_index: int = -100, temperature: float = 1.0, g=None, grad: bool = True,
                  threads: int = 1):
    """Per-token cross-entropy -ln softmax(x / T)[label] ('Add vocabulary-parallel
    logprobs, entropy and KL ops', section How: the log-prob op at the label id,
    with ignore_index positions giving 0 and no gradient). Steps: (1) x / T in
    float64; (2) the log-prob row oracle at the label; (3) the value negated and
    the gradient negated and divided by T (chain rule through x / T).
    Returns (loss [N], dx, index_errors)."""
    x = _rows2d(x)
    n = x.shape[0]
    lab = np.ascontiguousarray(np.asarray(labels, dtype=np.int64)).reshape(n, 1)
    gg = None if g is None else -_f64(g).reshape(n, 1)
    out, dx, errors = logprobs(x / float(temperature), lab, ignore_index, gg, grad=grad, threads=threads)
    loss = -out[:, 0]
    if dx is not None:
        dx = dx / float(temperature)
    return loss, dx, errors


def topk_forward_kl(s, index, teacher_logp, ignore_index: int = -100, temperature: float = 1.0, g=None,
                    grad: bool = True, threads: int = 1):
    """Teacher top-k forward KL ('Add vocabulary-parallel logprobs, entropy and KL
    ops', section What: the student's log-probs at the teacher's top-k ids, then
    the sum over k of exp(teacher log-prob) times (teacher log-prob - student
    log-prob)). Steps: (1) s / T in float64; (2) the log-prob row oracle at the
    ids; (3) the weighted sum over k, skipping ignore_index positions and
    teacher log-probs of -inf (no mass); (4) the gradient: the log-prob
    gradient with upstream -g exp(teacher log-prob) per position, divided by T.
    Returns (kl [N], ds, index_errors)."""
    s = _rows2d(s)
    n = s.shape[0]
    idx = np.ascontiguousarray(np.asarray(index, dtype=np.int64)).reshape(n, -1)
    tl = _f64(teacher_logp).reshape(idx.shape)
    live = (idx != ignore_index) & (tl != -np.inf)
    w = np.where(live, np.exp(np.where(live, tl, 0.0)), 0.0)
    gg = None
    if g is not None or grad:
        gr = np.ones(n) if g is None else _f64(g).reshape(n)
        gg = -gr[:, None] * w
    lp, ds, errors = logprobs(s / float(temperature), idx, ignore_index, gg, grad=grad, threads=threads)
    terms = np.where(live, w * (np.where(live, tl, 0.0) - lp), 0.0)
    # a selected id the student masks while the teacher gives it mass: +inf
    kl = np.sum(terms, axis=1)
    if ds is not None:
        ds = ds / float(temperature)
        ds[~np.isfinite(kl)] = 0.0  # a row with no finite value takes no gradient
    return kl, ds, errors
