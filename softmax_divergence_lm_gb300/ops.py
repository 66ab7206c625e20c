"""PyTorch autograd wrappers over the libvpd C ABI.

Each op is a ``torch.autograd.Function`` whose forward and backward call the
CUDA kernels through :mod:`binding` on the current stream. Outputs are float32
per-token values; gradients come back in the logits' dtype. Only first-order
gradients exist: a second backward raises ('Add vocabulary-parallel logprobs,
entropy and KL ops', section Limitations). Temperature, masking and reduction
over tokens stay with the caller.
"""
from __future__ import annotations

import torch
from torch.autograd.function import once_differentiable

from . import binding as B


def _rows(x: torch.Tensor) -> int:
    return x.shape[0] if x.dim() == 2 else x.shape[0] * x.shape[1]


def _out_shape(x: torch.Tensor):
    return x.shape[:-1]


def _grad_like(x: torch.Tensor) -> torch.Tensor:
    return torch.empty(x.shape, dtype=x.dtype, device=x.device)


class _JSD(torch.autograd.Function):
    @staticmethod
    def forward(ctx, s, t, beta, segments):
        n = _rows(s)
        loss = torch.empty(n, dtype=torch.float32, device=s.device)
        saved = torch.empty(n, B.SAVED_PAIR, dtype=torch.float32, device=s.device)
        B.vpd_jsd_fwd(s, t, beta, segments, loss, saved)
        ctx.save_for_backward(s, t, saved)
        ctx.beta, ctx.segments = beta, segments
        return loss.view(_out_shape(s))

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        s, t, saved = ctx.saved_tensors
        ds = _grad_like(s) if ctx.needs_input_grad[0] else None
        dt = _grad_like(t) if ctx.needs_input_grad[1] else None
        g = g.reshape(-1).to(torch.float32).contiguous()
        B.vpd_jsd_bwd(s, t, ctx.beta, ctx.segments, g, saved, ds, dt)
        return ds, dt, None, None


class _KL(torch.autograd.Function):
    @staticmethod
    def forward(ctx, s, t, reverse, segments):
        n = _rows(s)
        loss = torch.empty(n, dtype=torch.float32, device=s.device)
        saved = torch.empty(n, B.SAVED_PAIR, dtype=torch.float32, device=s.device)
        B.vpd_kl_fwd(s, t, reverse, segments, loss, saved)
        ctx.save_for_backward(s, t, saved)
        ctx.reverse, ctx.segments = reverse, segments
        return loss.view(_out_shape(s))

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        s, t, saved = ctx.saved_tensors
        ds = _grad_like(s) if ctx.needs_input_grad[0] else None
        dt = _grad_like(t) if ctx.needs_input_grad[1] else None
        g = g.reshape(-1).to(torch.float32).contiguous()
        B.vpd_kl_bwd(s, t, ctx.reverse, ctx.segments, g, saved, ds, dt)
        return ds, dt, None, None


class _Entropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, segments):
        n = _rows(x)
        out = torch.empty(n, dtype=torch.float32, device=x.device)
        saved = torch.empty(n, B.SAVED_ENTROPY, dtype=torch.float32, device=x.device)
        B.vpd_entropy_fwd(x, segments, out, saved)
        ctx.save_for_backward(x, saved)
        ctx.segments = segments
        return out.view(_out_shape(x))

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        x, saved = ctx.saved_tensors
        dx = _grad_like(x)
        B.vpd_entropy_bwd(x, ctx.segments, g.reshape(-1).to(torch.float32).contiguous(), saved, dx)
        return dx, None


class _LogProbs(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, index, ignore_index, segments, squeeze):
        n = _rows(x)
        idx = index.reshape(n, -1).to(torch.int64).contiguous()
        k = idx.shape[1]
        out = torch.empty(n, k, dtype=torch.float32, device=x.device)
        saved = torch.empty(n, B.SAVED_LOGPROBS, dtype=torch.float32, device=x.device)
        err = torch.empty(1, dtype=torch.int32, device=x.device)
        B.vpd_logprobs_fwd(x, segments, idx, k, ignore_index, out, saved, err)
        if int(err.item()):  # the range check syncs, as in the pages' wrapper
            raise IndexError("logprobs: an index is outside [0, V) and is not ignore_index")
        ctx.save_for_backward(x, idx, saved)
        ctx.k, ctx.ignore_index, ctx.segments = k, ignore_index, segments
        shape = tuple(_out_shape(x)) + (() if squeeze else (k,))
        return out.view(shape)

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        x, idx, saved = ctx.saved_tensors
        dx = _grad_like(x)
        g = g.reshape(-1, ctx.k).to(torch.float32).contiguous()
        B.vpd_logprobs_bwd(x, ctx.segments, idx, ctx.k, ctx.ignore_index, g, saved, dx)
        return dx, None, None, None, None


class _CrossEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, labels, ignore_index, temperature, segments):
        n = _rows(x)
        lab = labels.reshape(n).to(torch.int64).contiguous()
        loss = torch.empty(n, dtype=torch.float32, device=x.device)
        saved = torch.empty(n, B.SAVED_LOGPROBS, dtype=torch.float32, device=x.device)
        err = torch.empty(1, dtype=torch.int32, device=x.device)
        B.vpd_cross_entropy_fwd(x, segments, lab, ignore_index, temperature, loss, saved, err)
        if int(err.item()):
            raise IndexError("cross_entropy: a label is outside [0, V) and is not ignore_index")
        ctx.save_for_backward(x, lab, saved)
        ctx.ignore_index, ctx.temperature, ctx.segments = ignore_index, temperature, segments
        return loss.view(_out_shape(x))

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        x, lab, saved = ctx.saved_tensors
        dx = _grad_like(x)
        B.vpd_cross_entropy_bwd(x, ctx.segments, lab, ctx.ignore_index, ctx.temperature,
                                g.reshape(-1).to(torch.float32).contiguous(), saved, dx)
        return dx, None, None, None, None


class _TopkKL(torch.autograd.Function):
    @staticmethod
    def forward(ctx, s, index, teacher_logp, ignore_index, temperature, segments):
        n = _rows(s)
        idx = index.reshape(n, -1).to(torch.int64).contiguous()
        k = idx.shape[1]
        tl = teacher_logp.reshape(n, k).to(torch.float32).contiguous()
        kl = torch.empty(n, dtype=torch.float32, device=s.device)
        saved = torch.empty(n, B.SAVED_LOGPROBS, dtype=torch.float32, device=s.device)
        err = torch.empty(1, dtype=torch.int32, device=s.device)
        B.vpd_topk_kl_fwd(s, segments, idx, k, ignore_index, tl, temperature, kl, saved, err)
        if int(err.item()):
            raise IndexError("topk_forward_kl: an index is outside [0, V) and is not ignore_index")
        ctx.save_for_backward(s, idx, tl, saved)
        ctx.k, ctx.ignore_index, ctx.temperature, ctx.segments = k, ignore_index, temperature, segments
        return kl.view(_out_shape(s))

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        s, idx, tl, saved = ctx.saved_tensors
        ds = _grad_like(s)
        B.vpd_topk_kl_bwd(s, ctx.segments, idx, ctx.k, ctx.ignore_index, tl, ctx.temperature,
                          g.reshape(-1).to(torch.float32).contiguous(), saved, ds)
        return ds, None, None, None, None, None


def _seg(segments):
    return None if segments is None else tuple(int(w) for w in segments)


def jsd(student: torch.Tensor, teacher: torch.Tensor, beta: float = 0.5, segments=None) -> torch.Tensor:
    """Generalized JSD_beta per token ('[VocabTP] Add vocabulary-parallel
    generalized JSD with Triton kernels'); beta = 0 / 1 are forward / reverse KL."""
    return _JSD.apply(student, teacher, float(beta), _seg(segments))


def kl_div(student: torch.Tensor, teacher: torch.Tensor, reverse: bool = False, segments=None) -> torch.Tensor:
    """KL(P_t || P_s), or KL(P_s || P_t) with reverse=True, per token."""
    return _KL.apply(student, teacher, bool(reverse), _seg(segments))


def entropy(logits: torch.Tensor, segments=None) -> torch.Tensor:
    """Entropy of softmax(logits) per token."""
    return _Entropy.apply(logits, _seg(segments))


def logprobs(logits: torch.Tensor, index: torch.Tensor, ignore_index: int = -100, segments=None) -> torch.Tensor:
    """log softmax(logits) at index ([..] for one id per token, [.., k] for top-k);
    positions equal to ignore_index return 0."""
    squeeze = index.dim() == logits.dim() - 1
    return _LogProbs.apply(logits, index, int(ignore_index), _seg(segments), squeeze)


def jsd_fwdbwd(student, teacher, beta, grad_loss=None, segments=None, grad_dtype=None,
               student_grad=True, teacher_grad=True):
    """One-call forward+backward (single HBM read of each row pair when it fits
    on chip). Returns (loss, saved, ds, dt); ds / dt are None when not asked."""
    n = _rows(student)
    dev = student.device
    loss = torch.empty(n, dtype=torch.float32, device=dev)
    saved = torch.empty(n, B.SAVED_PAIR, dtype=torch.float32, device=dev)
    gd = grad_dtype or student.dtype
    ds = torch.empty(student.shape, dtype=gd, device=dev) if student_grad else None
    dt = torch.empty(teacher.shape, dtype=gd, device=dev) if teacher_grad else None
    B.vpd_jsd_fwdbwd(student, teacher, float(beta), _seg(segments), grad_loss, loss, saved, ds, dt)
    return loss.view(_out_shape(student)), saved, ds, dt


def cross_entropy(logits: torch.Tensor, labels: torch.Tensor, ignore_index: int = -100, temperature: float = 1.0,
                  segments=None) -> torch.Tensor:
    """Per-token -log softmax(logits / temperature)[label]; ignore_index gives 0."""
    return _CrossEntropy.apply(logits, labels, int(ignore_index), float(temperature), _seg(segments))


def topk_forward_kl(student: torch.Tensor, teacher_topk_ids: torch.Tensor, teacher_topk_logp: torch.Tensor,
                    ignore_index: int = -100, temperature: float = 1.0, segments=None) -> torch.Tensor:
    """Teacher top-k forward KL per token ('Add vocabulary-parallel logprobs,
    entropy and KL ops', section What): sum_k exp(tl_k) (tl_k - log p_s[id_k]),
    the teacher's top-k log-probs tl given (detached)."""
    return _TopkKL.apply(student, teacher_topk_ids, teacher_topk_logp, int(ignore_index), float(temperature),
                         _seg(segments))
