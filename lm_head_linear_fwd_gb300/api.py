"""PyTorch-facing API of the loss head: allocation, streams and autograd.

PyTorch only allocates device memory and supplies the current stream; every
step of the computation runs in libflce.so's kernels, reached through the
C ABI (``_abi``).  There is no CPU or eager-PyTorch fallback: a missing
library or a non-CUDA tensor raises.

Low-level calls (same names as the C entry points):
    ce_logits_fwd, ce_logits_bwd, ce_logits_fwd_bwd, flce_fwd, flce_bwd,
    flce_fwd_bwd, flce_gemm
Autograd front ends:
    ce_logits(logits, labels, *, ignore_index, reduction, num_label_tokens,
              inplace_grad=False, mask=None, save_lse=True, eager=False)
    flce(H, W, labels, bias=None, *, ignore_index, reduction, num_label_tokens,
         chunk=None, mask=None, eager=False)
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch
from torch.autograd.function import once_differentiable

from . import _abi

_DT = {torch.bfloat16: _abi.FLCE_BF16, torch.float32: _abi.FLCE_F32}
_RED = {"sum": _abi.FLCE_SUM, "mean": _abi.FLCE_MEAN}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}: expected bfloat16 or float32")
    return _DT[t.dtype]


def _red_code(reduction: str) -> int:
    if reduction not in _RED:
        raise ValueError(f"reduction must be 'sum' or 'mean', got {reduction!r}")
    return _RED[reduction]


def _nlt(num_label_tokens) -> int:
    if num_label_tokens is None:
        return -1
    n = int(num_label_tokens)
    if n < 0:
        raise ValueError("num_label_tokens must be >= 0")
    return n


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the loss head has no CPU path)")
    return t


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def new_status(device) -> torch.Tensor:
    """A zeroed device status word (see the Errors section of flce.h)."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(status: torch.Tensor, where: str = "device") -> None:
    """Reads the device status word (synchronises) and raises if it is set."""
    code = int(status.item())
    if code != _abi.FLCE_OK:
        raise _abi.FlceError(code, where)


def _labels(labels: torch.Tensor, N: int) -> torch.Tensor:
    _cuda(labels, "labels")
    if labels.dtype != torch.int64 or labels.dim() != 1 or labels.shape[0] != N:
        raise ValueError(f"labels must be int64 of shape [{N}]")
    return labels.contiguous()


# ---------------------------------------------------------------- CE on logits

@dataclasses.dataclass
class ForwardOut:
    """Device outputs of a forward call (reusable through ``out=``)."""
    loss: torch.Tensor           # [1] f32
    n_valid: torch.Tensor        # [1] i64
    lse: torch.Tensor            # [N] f32
    loss_rows: Optional[torch.Tensor]
    label_logit: Optional[torch.Tensor]
    status: torch.Tensor         # [1] i32


def ce_logits_workspace_bytes(N: int, V: int) -> int:
    """Bytes of device workspace ce_logits_fwd needs for [N, V] logits."""
    return int(_abi.ce_logits_workspace_bytes(N, V))


def ce_logits_fwd(logits, labels, ignore_index=-100, reduction="sum", num_label_tokens=None, *,
                  want_rows=False, want_label_logit=False, ws=None, status=None,
                  out=None) -> ForwardOut:
    """Forward of cross-entropy on given logits [N, V] (bf16 or fp32, row
    stride free, unit stride along V).  Returns the loss, n_valid, the per-row
    lse (what the backward needs) and, on request, per-row losses and the
    gathered label logits.  ``ws``/``status``/``out`` let a caller reuse
    buffers (a CUDA graph, a loop); otherwise they are allocated here."""
    _cuda(logits, "logits")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D with unit stride along the vocabulary")
    N, V = logits.shape
    labels = _labels(labels, N)
    dev = logits.device
    if out is None:
        out = ForwardOut(
            loss=torch.empty(1, dtype=torch.float32, device=dev),
            n_valid=torch.empty(1, dtype=torch.int64, device=dev),
            lse=torch.empty(N, dtype=torch.float32, device=dev),
            loss_rows=torch.empty(N, dtype=torch.float32, device=dev) if want_rows else None,
            label_logit=torch.empty(N, dtype=torch.float32, device=dev) if want_label_logit else None,
            status=status if status is not None else new_status(dev))
    nbytes = ce_logits_workspace_bytes(N, V)
    if ws is None:
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    rc = _abi.ce_logits_fwd(_ptr(logits), _dtype_code(logits), N, V, logits.stride(0),
                            _ptr(labels), int(ignore_index), _red_code(reduction),
                            _nlt(num_label_tokens), _ptr(out.loss), _ptr(out.n_valid),
                            _ptr(out.lse), _ptr(out.loss_rows), _ptr(out.label_logit),
                            _ptr(ws), ws.numel(), _ptr(out.status), _stream(dev))
    _abi.check(rc, "ce_logits_fwd")
    return out


def ce_logits_bwd(logits, labels, lse, n_valid, grad_loss, ignore_index=-100, reduction="sum",
                  num_label_tokens=None, inplace_grad=False, grad_logits=None,
                  status=None) -> torch.Tensor:
    """Gradient of the loss with respect to the logits.  ``lse=None``: no saved
    lse, each row's lse is formed again from the logits in the kernel."""
    _cuda(logits, "logits")
    N, V = logits.shape
    labels = _labels(labels, N)
    dev = logits.device
    if inplace_grad:
        grad_logits = logits
    elif grad_logits is None:
        grad_logits = torch.empty((N, V), dtype=logits.dtype, device=dev)
    if grad_logits.dtype != logits.dtype or grad_logits.stride(1) != 1:
        raise ValueError("grad_logits must have the logits dtype and unit column stride")
    g = grad_loss.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
    status = status if status is not None else new_status(dev)
    rc = _abi.ce_logits_bwd(_ptr(logits), _dtype_code(logits), N, V, logits.stride(0),
                            _ptr(labels), int(ignore_index), _red_code(reduction),
                            _nlt(num_label_tokens), _ptr(lse), _ptr(n_valid), _ptr(g),
                            1 if inplace_grad else 0, _ptr(grad_logits), grad_logits.stride(0),
                            _ptr(status), _stream(dev))
    _abi.check(rc, "ce_logits_bwd")
    return grad_logits


def ce_logits_fwd_bwd_workspace_bytes(N: int, V: int) -> int:
    """Bytes of device workspace ce_logits_fwd_bwd needs for [N, V] logits."""
    return int(_abi.ce_logits_fwd_bwd_workspace_bytes(N, V))


def ce_logits_fwd_bwd(logits, labels, ignore_index=-100, reduction="sum", num_label_tokens=None,
                      grad_loss=None, *, inplace_grad=False, grad_logits=None, want_lse=False,
                      ws=None, status=None, out=None):
    """Loss and gradient of the logits in one call (the gradient for the
    incoming gradient ``grad_loss``, a [1] tensor; None means 1).  Aligned rows
    are read once.  Returns (ForwardOut, grad_logits); ``ForwardOut.lse`` is
    None unless ``want_lse`` (then valid on rows with a valid label).
    ``ws``/``status``/``out``/``grad_logits`` let a caller reuse buffers."""
    _cuda(logits, "logits")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D with unit stride along the vocabulary")
    N, V = logits.shape
    labels = _labels(labels, N)
    dev = logits.device
    if inplace_grad:
        grad_logits = logits
    elif grad_logits is None:
        grad_logits = torch.empty((N, V), dtype=logits.dtype, device=dev)
    if grad_logits.dtype != logits.dtype or grad_logits.stride(1) != 1:
        raise ValueError("grad_logits must have the logits dtype and unit column stride")
    g = None
    if grad_loss is not None:
        g = grad_loss.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
    if out is None:
        out = ForwardOut(
            loss=torch.empty(1, dtype=torch.float32, device=dev),
            n_valid=torch.empty(1, dtype=torch.int64, device=dev),
            lse=torch.empty(N, dtype=torch.float32, device=dev) if want_lse else None,
            loss_rows=None, label_logit=None,
            status=status if status is not None else new_status(dev))
    nbytes = ce_logits_fwd_bwd_workspace_bytes(N, V)
    if ws is None:
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    rc = _abi.ce_logits_fwd_bwd(_ptr(logits), _dtype_code(logits), N, V, logits.stride(0),
                                _ptr(labels), int(ignore_index), _red_code(reduction),
                                _nlt(num_label_tokens), _ptr(g), _ptr(out.loss),
                                _ptr(out.n_valid), _ptr(out.lse), 1 if inplace_grad else 0,
                                _ptr(grad_logits), grad_logits.stride(0), _ptr(ws), ws.numel(),
                                _ptr(out.status), _stream(dev))
    _abi.check(rc, "ce_logits_fwd_bwd")
    return out, grad_logits


class _CELogitsEager(torch.autograd.Function):
    """The gradient formed during the forward (ce_logits_fwd_bwd with g = 1),
    scaled by the incoming gradient in the backward."""

    @staticmethod
    def forward(ctx, logits, labels, ignore_index, reduction, num_label_tokens, inplace_grad):
        out, grad = ce_logits_fwd_bwd(logits, labels, ignore_index, reduction, num_label_tokens,
                                      inplace_grad=inplace_grad)
        ctx.grad = grad
        ctx.status = out.status
        return out.loss.reshape(())

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        grad, ctx.grad = ctx.grad, None
        if grad is None:
            raise RuntimeError("ce_logits(eager=True): the gradient was already handed out; "
                               "a second backward is not possible")
        grad_scale_(grad, g)
        return grad, None, None, None, None, None


class _CELogits(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, labels, ignore_index, reduction, num_label_tokens, inplace_grad,
                save_lse=True):
        out = ce_logits_fwd(logits, labels, ignore_index, reduction, num_label_tokens)
        ctx.save_lse = save_lse
        if save_lse:
            ctx.save_for_backward(logits, labels, out.lse, out.n_valid)
        else:  # the backward forms the lse again from the logits
            ctx.save_for_backward(logits, labels, out.n_valid)
        ctx.args = (ignore_index, reduction, num_label_tokens, inplace_grad)
        ctx.status = out.status
        ctx.consumed = False
        return out.loss.reshape(())

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        if ctx.save_lse:
            logits, labels, lse, n_valid = ctx.saved_tensors
        else:
            (logits, labels, n_valid), lse = ctx.saved_tensors, None
        ignore_index, reduction, nlt, inplace = ctx.args
        if inplace and ctx.consumed:
            raise RuntimeError("ce_logits(inplace_grad=True): the logits were already overwritten "
                               "by their gradient; a second backward is not possible")
        ctx.consumed = True
        grad = ce_logits_bwd(logits, labels, lse, n_valid, g, ignore_index, reduction, nlt,
                             inplace_grad=inplace, status=ctx.status)
        return grad, None, None, None, None, None, None


def _fold_mask(labels, mask, ignore_index):
    if mask is None:
        return labels
    return labels.masked_fill(mask.to(device=labels.device) == 0, ignore_index)


def _rows(x, labels, mask, what):
    """Leading dimensions flattened into rows: x [..., K] -> [N, K] (a view when
    the strides allow it; autograd maps the gradient back), labels and mask
    [...] -> [N]."""
    if not isinstance(x, torch.Tensor) or x.dim() < 2:
        raise ValueError(f"{what} must be at least 2-D")
    lead = x.shape[:-1]
    if tuple(labels.shape) != tuple(lead):
        raise ValueError(f"labels must have the leading shape {tuple(lead)} of {what}")
    if mask is not None and tuple(mask.shape) != tuple(lead):
        raise ValueError(f"mask must have the shape {tuple(lead)} of the labels")
    if x.dim() == 2:
        return x, labels, mask
    return (x.reshape(-1, x.shape[-1]), labels.reshape(-1),
            None if mask is None else mask.reshape(-1))


def ce_logits(logits, labels, *, ignore_index=-100, reduction="sum", num_label_tokens=None,
              inplace_grad=False, mask=None, save_lse=True, eager=False):
    """Masked cross-entropy on given logits [N, V] (bf16 or fp32).

    ``inplace_grad=True`` writes the gradient into the logits storage during
    backward (the logits are destroyed); it is keyword-only and off by default.
    ``mask`` (same shape as labels) marks rows to ignore with 0.
    ``save_lse=False`` keeps only the logits and labels (and the valid-row
    count) for the backward, which then forms each row's lse again.
    ``eager=True`` forms the gradient during the forward, reading each row
    once for both, and keeps it until the backward scales it by the incoming
    gradient (no work when that is 1); with ``inplace_grad=True`` the logits
    are overwritten by their gradient already in the forward, and must then
    be contiguous.  Leading dimensions are flattened: logits [..., V] with
    labels (and mask) [...]."""
    logits, labels, mask = _rows(logits, labels, mask, "logits")
    labels = _fold_mask(labels, mask, ignore_index)
    if eager:
        _cuda(logits, "logits")
        if inplace_grad and not logits.is_contiguous():
            raise ValueError("ce_logits(eager=True, inplace_grad=True) needs contiguous logits")
        return _CELogitsEager.apply(logits, labels, int(ignore_index), reduction,
                                    num_label_tokens, bool(inplace_grad))
    return _CELogits.apply(logits, labels, int(ignore_index), reduction, num_label_tokens,
                           bool(inplace_grad), bool(save_lse))


def mask_packed_labels(labels: torch.Tensor, doc_ids: torch.Tensor, ignore_index: int = -100):
    """In place: labels [B, T] become ignore_index on padding (doc id 0) and on
    the last token of every packed document (see flce_mask_packed_labels)."""
    _cuda(labels, "labels")
    _cuda(doc_ids, "doc_ids")
    if labels.shape != doc_ids.shape or labels.dim() != 2:
        raise ValueError("labels and doc_ids must both be [B, T]")
    if labels.dtype != torch.int64 or doc_ids.dtype != torch.int64:
        raise TypeError("labels and doc_ids must be int64")
    if not labels.is_contiguous():
        raise ValueError("labels must be contiguous (it is written in place)")
    doc_ids = doc_ids.contiguous()
    B, T = labels.shape
    rc = _abi.flce_mask_packed_labels(_ptr(labels), _ptr(doc_ids), B, T, int(ignore_index),
                                      _stream(labels.device))
    _abi.check(rc, "flce_mask_packed_labels")
    return labels


# ---------------------------------------------------------- fused linear CE

def flce_workspace_bytes(dt_code: int, N: int, D: int, V: int, chunk: int = 0) -> int:
    """Bytes of device workspace flce_fwd / flce_bwd need (chunk 0: the default;
    chunk > 0: rows per backward chunk; chunk < 0: vocabulary slices of -chunk
    columns)."""
    return int(_abi.flce_workspace_bytes(dt_code, N, D, V, chunk))


def flce_default_chunk(dt_code: int, N: int, D: int, V: int) -> int:
    """Rows per backward chunk when no chunk is given (sizes the dZ buffer)."""
    return int(_abi.flce_default_chunk(dt_code, N, D, V))


def _flce_inputs(H, W, bias):
    _cuda(H, "H")
    _cuda(W, "W")
    if H.dim() != 2 or W.dim() != 2 or H.shape[1] != W.shape[1]:
        raise ValueError("H must be [N, D] and W [V, D]")
    if H.dtype != W.dtype or (bias is not None and bias.dtype != H.dtype):
        raise TypeError("H, W and bias must share one dtype")
    if not H.is_contiguous() or not W.is_contiguous():
        raise ValueError("H and W must be contiguous")
    if bias is not None:
        _cuda(bias, "bias")
        if bias.shape != (W.shape[0],) or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous [V] tensor")
    return H.shape[0], H.shape[1], W.shape[0]


def flce_fwd(H, W, labels, bias=None, ignore_index=-100, reduction="sum", num_label_tokens=None,
             *, want_rows=False, want_label_logit=False, ws=None, status=None,
             out=None) -> ForwardOut:
    """Forward of fused linear cross-entropy: logits = H @ W.T (+ bias) are
    reduced tile by tile and never stored.  H [N, D], W [V, D], bias [V] or
    None, one dtype (bf16, or fp32 computed in tf32).  Returns the loss,
    n_valid and the per-row lse the backward needs."""
    N, D, V = _flce_inputs(H, W, bias)
    labels = _labels(labels, N)
    dev = H.device
    dt = _dtype_code(H)
    if out is None:
        out = ForwardOut(
            loss=torch.empty(1, dtype=torch.float32, device=dev),
            n_valid=torch.empty(1, dtype=torch.int64, device=dev),
            lse=torch.empty(N, dtype=torch.float32, device=dev),
            loss_rows=torch.empty(N, dtype=torch.float32, device=dev) if want_rows else None,
            label_logit=torch.empty(N, dtype=torch.float32, device=dev) if want_label_logit else None,
            status=status if status is not None else new_status(dev))
    if ws is None:
        ws = torch.empty(flce_workspace_bytes(dt, N, D, V), dtype=torch.uint8, device=dev)
    rc = _abi.flce_fwd(_ptr(H), _ptr(W), _ptr(bias), dt, N, D, V, _ptr(labels), int(ignore_index),
                       _red_code(reduction), _nlt(num_label_tokens), _ptr(out.loss),
                       _ptr(out.n_valid), _ptr(out.lse), _ptr(out.loss_rows),
                       _ptr(out.label_logit), _ptr(ws), ws.numel(), _ptr(out.status),
                       _stream(dev))
    _abi.check(rc, "flce_fwd")
    return out


@dataclasses.dataclass
class BackwardOut:
    """Gradients of a backward call (None where not requested)."""
    grad_H: Optional[torch.Tensor]
    grad_W: Optional[torch.Tensor]     # fp32
    grad_bias: Optional[torch.Tensor]  # fp32


def flce_bwd(H, W, labels, lse, n_valid, grad_loss, bias=None, ignore_index=-100, reduction="sum",
             num_label_tokens=None, chunk=None, *, want_grad_H=True, want_grad_W=True,
             want_grad_bias=None, grad_W=None, accumulate_grad_W=False, grad_H=None,
             grad_bias=None, ws=None, status=None) -> BackwardOut:
    """Backward of fused linear cross-entropy, recomputing the logits chunk
    by chunk: grad_H (dtype of H), grad_W (fp32; added to ``grad_W`` when
    ``accumulate_grad_W``) and grad_bias (fp32), from the forward's lse and
    n_valid and the incoming gradient ``grad_loss``."""
    N, D, V = _flce_inputs(H, W, bias)
    labels = _labels(labels, N)
    dev = H.device
    dt = _dtype_code(H)
    ch = 0 if chunk is None else int(chunk)
    if want_grad_bias is None:
        want_grad_bias = bias is not None
    if want_grad_H and grad_H is None:
        grad_H = torch.empty((N, D), dtype=H.dtype, device=dev)
    if want_grad_W and grad_W is None:
        grad_W = torch.empty((V, D), dtype=torch.float32, device=dev)
    if want_grad_bias and grad_bias is None:
        grad_bias = torch.empty(V, dtype=torch.float32, device=dev)
    if not want_grad_H:
        grad_H = None
    if not want_grad_W:
        grad_W = None
    if not want_grad_bias:
        grad_bias = None
    if ws is None:
        ws = torch.empty(flce_workspace_bytes(dt, N, D, V, ch), dtype=torch.uint8, device=dev)
    g = grad_loss.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
    status = status if status is not None else new_status(dev)
    rc = _abi.flce_bwd(_ptr(H), _ptr(W), _ptr(bias), dt, N, D, V, _ptr(labels), int(ignore_index),
                       _red_code(reduction), _nlt(num_label_tokens), _ptr(lse), _ptr(n_valid),
                       _ptr(g), ch, _ptr(grad_H), _ptr(grad_W), 1 if accumulate_grad_W else 0,
                       _ptr(grad_bias), _ptr(ws), ws.numel(), _ptr(status), _stream(dev))
    _abi.check(rc, "flce_bwd")
    return BackwardOut(grad_H, grad_W, grad_bias)


def flce_fwd_bwd(H, W, labels, bias=None, ignore_index=-100, reduction="sum",
                 num_label_tokens=None, chunk=None, grad_loss=None, *, want_grad_H=True,
                 want_grad_W=True, want_grad_bias=None, want_rows=False, grad_W=None,
                 accumulate_grad_W=False, ws=None, status=None):
    """Loss and gradients in one call (6NDV flops).  Returns (ForwardOut, BackwardOut).
    grad_loss None means g = 1."""
    N, D, V = _flce_inputs(H, W, bias)
    labels = _labels(labels, N)
    dev = H.device
    dt = _dtype_code(H)
    ch = 0 if chunk is None else int(chunk)
    if want_grad_bias is None:
        want_grad_bias = bias is not None
    out = ForwardOut(loss=torch.empty(1, dtype=torch.float32, device=dev),
                     n_valid=torch.empty(1, dtype=torch.int64, device=dev),
                     lse=torch.empty(N, dtype=torch.float32, device=dev),
                     loss_rows=torch.empty(N, dtype=torch.float32, device=dev) if want_rows else None,
                     label_logit=None,
                     status=status if status is not None else new_status(dev))
    gH = torch.empty((N, D), dtype=H.dtype, device=dev) if want_grad_H else None
    if want_grad_W and grad_W is None:
        grad_W = torch.empty((V, D), dtype=torch.float32, device=dev)
    gW = grad_W if want_grad_W else None
    gb = torch.empty(V, dtype=torch.float32, device=dev) if want_grad_bias else None
    if ws is None:
        ws = torch.empty(int(_abi.flce_fwd_bwd_workspace_bytes(dt, N, D, V, ch)),
                         dtype=torch.uint8, device=dev)
    g = None
    if grad_loss is not None:
        g = grad_loss.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
    rc = _abi.flce_fwd_bwd(_ptr(H), _ptr(W), _ptr(bias), dt, N, D, V, _ptr(labels),
                           int(ignore_index), _red_code(reduction), _nlt(num_label_tokens), _ptr(g),
                           ch, _ptr(out.loss), _ptr(out.n_valid), _ptr(out.lse),
                           _ptr(out.loss_rows), _ptr(gH), _ptr(gW),
                           1 if accumulate_grad_W else 0, _ptr(gb), _ptr(ws), ws.numel(),
                           _ptr(out.status), _stream(dev))
    _abi.check(rc, "flce_fwd_bwd")
    return out, BackwardOut(gH, gW, gb)


def grad_scale_(x: torch.Tensor, g: torch.Tensor) -> torch.Tensor:
    """x *= g in place on the device (no work when g == 1)."""
    _cuda(x, "x")
    g = g.to(device=x.device, dtype=torch.float32).reshape(1).contiguous()
    rc = _abi.flce_grad_scale(_ptr(x), _dtype_code(x), x.numel(), _ptr(g), _stream(x.device))
    _abi.check(rc, "flce_grad_scale")
    return x


class _FLCEEager(torch.autograd.Function):
    """Gradients formed during the forward (flce_fwd_bwd with g = 1), scaled by
    the incoming gradient in the backward."""

    @staticmethod
    def forward(ctx, H, W, labels, bias, ignore_index, reduction, num_label_tokens, chunk):
        out, bw = flce_fwd_bwd(H, W, labels, bias, ignore_index, reduction, num_label_tokens,
                               chunk, want_grad_H=H.requires_grad, want_grad_W=W.requires_grad,
                               want_grad_bias=bias is not None and bias.requires_grad)
        ctx.grads = (bw.grad_H, bw.grad_W, bw.grad_bias)
        return out.loss.reshape(())

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        gH, gW, gb = ctx.grads
        ctx.grads = (None, None, None)
        if gH is None and gW is None and gb is None:
            raise RuntimeError("flce(eager=True): the gradients were already handed out; "
                               "a second backward is not possible")
        for t in (gH, gW, gb):
            if t is not None:
                grad_scale_(t, g)
        return gH, gW, None, gb, None, None, None, None


class _FLCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W, labels, bias, ignore_index, reduction, num_label_tokens, chunk):
        out = flce_fwd(H, W, labels, bias, ignore_index, reduction, num_label_tokens)
        ctx.save_for_backward(H, W, labels, bias, out.lse, out.n_valid)
        ctx.args = (ignore_index, reduction, num_label_tokens, chunk)
        ctx.status = out.status
        return out.loss.reshape(())

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        H, W, labels, bias, lse, n_valid = ctx.saved_tensors
        ignore_index, reduction, nlt, chunk = ctx.args
        need_H, need_W, _, need_b = ctx.needs_input_grad[:4]
        out = flce_bwd(H, W, labels, lse, n_valid, g, bias, ignore_index, reduction, nlt, chunk,
                       want_grad_H=need_H, want_grad_W=need_W,
                       want_grad_bias=bool(need_b and bias is not None), status=ctx.status)
        # grad_W / grad_bias are accumulated in fp32; autograd casts them to the
        # parameter dtype when that differs.
        return out.grad_H, out.grad_W, None, out.grad_bias, None, None, None, None


def flce(H, W, labels, bias=None, *, ignore_index=-100, reduction="mean", num_label_tokens=None,
         chunk=None, mask=None, eager=False):
    """Fused linear cross-entropy: loss of logits = H @ W.T (+ bias), never materialised.

    H: [N, D], W: [V, D] (tied-embedding layout), bias: [V] or None, labels:
    [N] int64.  Default: the backward recomputes the logits chunk by chunk
    (``chunk`` rows at a time; None picks the library default), 8NDV flops in
    all.  ``eager=True`` forms the gradients during the forward (6NDV flops)
    and keeps them, fp32 grad_W included, until the backward scales them.
    Leading dimensions are flattened: H [..., D] with labels (and mask) [...]."""
    H, labels, mask = _rows(H, labels, mask, "H")
    labels = _fold_mask(labels, mask, ignore_index)
    fn = _FLCEEager if eager else _FLCE
    return fn.apply(H, W, labels, bias, int(ignore_index), reduction, num_label_tokens, chunk)


# ------------------------------------------------------------------- raw GEMM

def flce_gemm(A, B, C, a_mn_major=False, b_mn_major=False, accumulate=False, status=None):
    """C (+)= op(A) @ op(B).T on the tensor cores (see include/flce_gemm.h).

    A is [M, K] (K-major) or [K, M] (MN-major); B is [N, K] or [K, N]; C is
    [M, N] float32."""
    _cuda(A, "A")
    _cuda(B, "B")
    _cuda(C, "C")
    if A.dtype != B.dtype or C.dtype != torch.float32:
        raise TypeError("A and B share a dtype; C is float32")
    M = A.shape[1] if a_mn_major else A.shape[0]
    K = A.shape[0] if a_mn_major else A.shape[1]
    Nn = B.shape[1] if b_mn_major else B.shape[0]
    Kb = B.shape[0] if b_mn_major else B.shape[1]
    if K != Kb or tuple(C.shape) != (M, Nn):
        raise ValueError("inconsistent GEMM shapes")
    status = status if status is not None else new_status(A.device)
    rc = _abi.flce_gemm(_dtype_code(A), int(a_mn_major), int(b_mn_major), M, Nn, K, _ptr(A),
                        A.stride(0), _ptr(B), B.stride(0), _ptr(C), C.stride(0),
                        int(accumulate), _ptr(status), _stream(A.device))
    _abi.check(rc, "flce_gemm")
    return C
