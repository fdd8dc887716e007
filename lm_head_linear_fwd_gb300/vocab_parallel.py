"""Vocabulary-parallel fused linear cross-entropy ("Loss Parallel").

Each rank holds a contiguous slice of the vocabulary: rows [v0, v0 + V_r) of
W (and of the bias), all of H and the labels.  The forward needs three
reductions of [N]-vectors over the ranks (MAX of the per-row maxima, SUM of
the rescaled sums, SUM of the label logits), the backward one (SUM of the
grad_H partials); grad_W and grad_bias stay with their shard.  See the
vocabulary-parallel section of include/flce.h.

The arithmetic runs in the library's kernels (``CudaShardOps``); this module
only orders the phases and the collectives, through an ``exchange`` with
``max_`` / ``sum_`` methods (``TorchDistExchange`` for a process group).
"""
from __future__ import annotations

import dataclasses

import torch
import torch.distributed as dist

from . import _abi
from .api import _cuda, _dtype_code, _labels, _nlt, _ptr, _red_code, _stream, new_status


class TorchDistExchange:
    """In-place reductions over a torch.distributed process group."""

    def __init__(self, group=None):
        self.group = group

    def _active(self):
        return dist.is_available() and dist.is_initialized()

    def max_(self, t):
        if self._active():
            dist.all_reduce(t, op=dist.ReduceOp.MAX, group=self.group)
        return t

    def sum_(self, t):
        if self._active():
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=self.group)
        return t


@dataclasses.dataclass
class ShardForward:
    """Forward results of a vocabulary shard, already reduced over the ranks."""
    loss: torch.Tensor      # [1] f32, identical on every rank
    n_valid: torch.Tensor   # [1] i64
    lse: torch.Tensor       # [N] f32 (global)
    status: torch.Tensor


class CudaShardOps:
    """The per-rank steps, each one library call."""

    def partials(self, H, W_shard, labels, v0, V_total, bias, ignore_index, status):
        _cuda(H, "H")
        N, D = H.shape
        V = W_shard.shape[0]
        dt = _dtype_code(H)
        dev = H.device
        m = torch.empty(N, dtype=torch.float32, device=dev)
        s = torch.empty_like(m)
        zy = torch.empty_like(m)
        ws = torch.empty(int(_abi.flce_workspace_bytes(dt, N, D, V, 0)), dtype=torch.uint8,
                         device=dev)
        rc = _abi.flce_fwd_shard(_ptr(H), _ptr(W_shard), _ptr(bias), dt, N, D, V, int(v0),
                                 int(V_total), _ptr(labels), int(ignore_index), _ptr(m), _ptr(s),
                                 _ptr(zy), _ptr(ws), ws.numel(), _ptr(status), _stream(dev))
        _abi.check(rc, "flce_fwd_shard")
        return m, s, zy

    def rescale(self, m, s, m_global):
        out = torch.empty_like(s)
        rc = _abi.flce_shard_rescale(_ptr(m), _ptr(s), _ptr(m_global), m.numel(), _ptr(out),
                                     _stream(m.device))
        _abi.check(rc, "flce_shard_rescale")
        return out

    def finish(self, m_global, s_global, zy_global, labels, V_total, ignore_index, reduction,
               num_label_tokens, status):
        N = labels.numel()
        dev = labels.device
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        loss = torch.empty(1, dtype=torch.float32, device=dev)
        n_valid = torch.empty(1, dtype=torch.int64, device=dev)
        ws = torch.empty(max(256, (N * 4 + 255) // 256 * 256), dtype=torch.uint8, device=dev)
        rc = _abi.flce_shard_finish(_ptr(m_global), _ptr(s_global), _ptr(zy_global),
                                    _ptr(labels), N, int(V_total), int(ignore_index),
                                    _red_code(reduction), _nlt(num_label_tokens), _ptr(lse), None,
                                    _ptr(loss), _ptr(n_valid), _ptr(ws), ws.numel(), _ptr(status),
                                    _stream(dev))
        _abi.check(rc, "flce_shard_finish")
        return lse, loss, n_valid

    def backward(self, H, W_shard, labels, v0, V_total, bias, ignore_index, reduction,
                 num_label_tokens, lse, n_valid, grad_loss, chunk, want_grad_H, want_grad_W,
                 status):
        N, D = H.shape
        V = W_shard.shape[0]
        dt = _dtype_code(H)
        dev = H.device
        # fp32 partial: summed over the ranks before the one rounding to H's dtype
        gH = torch.empty((N, D), dtype=torch.float32, device=dev) if want_grad_H else None
        gW = torch.empty((V, D), dtype=torch.float32, device=dev) if want_grad_W else None
        gb = torch.empty(V, dtype=torch.float32, device=dev) if bias is not None else None
        ch = 0 if chunk is None else int(chunk)
        ws = torch.empty(int(_abi.flce_workspace_bytes(dt, N, D, V, ch)), dtype=torch.uint8,
                         device=dev)
        g = grad_loss.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
        rc = _abi.flce_bwd_shard(_ptr(H), _ptr(W_shard), _ptr(bias), dt, N, D, V, int(v0),
                                 int(V_total), _ptr(labels), int(ignore_index),
                                 _red_code(reduction), _nlt(num_label_tokens), _ptr(lse),
                                 _ptr(n_valid), _ptr(g), ch, _ptr(gH), _ptr(gW), 0, _ptr(gb),
                                 _ptr(ws), ws.numel(), _ptr(status), _stream(dev))
        _abi.check(rc, "flce_bwd_shard")
        return gH, gW, gb


class CudaLogitsShardOps(CudaShardOps):
    """The per-rank steps of CE on a vocabulary shard of given logits."""

    def partials(self, logits, _unused, labels, v0, V_total, _bias, ignore_index, status):
        _cuda(logits, "logits")
        if logits.dim() != 2 or logits.stride(1) != 1:
            raise ValueError("logits shard must be 2-D with unit column stride")
        N, V = logits.shape
        dev = logits.device
        m = torch.empty(N, dtype=torch.float32, device=dev)
        s = torch.empty_like(m)
        zy = torch.empty_like(m)
        rc = _abi.ce_logits_fwd_shard(_ptr(logits), _dtype_code(logits), N, V, logits.stride(0),
                                      int(v0), int(V_total), _ptr(labels), int(ignore_index),
                                      _ptr(m), _ptr(s), _ptr(zy), _ptr(status), _stream(dev))
        _abi.check(rc, "ce_logits_fwd_shard")
        return m, s, zy

    def logits_backward(self, logits, labels, v0, V_total, ignore_index, reduction,
                        num_label_tokens, lse, n_valid, grad_loss, inplace_grad, status):
        N, V = logits.shape
        dev = logits.device
        grad = logits if inplace_grad else torch.empty((N, V), dtype=logits.dtype, device=dev)
        g = grad_loss.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
        rc = _abi.ce_logits_bwd_shard(_ptr(logits), _dtype_code(logits), N, V, logits.stride(0),
                                      int(v0), int(V_total), _ptr(labels), int(ignore_index),
                                      _red_code(reduction), _nlt(num_label_tokens), _ptr(lse),
                                      _ptr(n_valid), _ptr(g), 1 if inplace_grad else 0,
                                      _ptr(grad), grad.stride(0), _ptr(status), _stream(dev))
        _abi.check(rc, "ce_logits_bwd_shard")
        return grad


def ce_forward(logits_shard, labels, vocab_offset, V_total, *, ignore_index=-100,
               reduction="sum", num_label_tokens=None, exchange=None, ops=None,
               status=None) -> ShardForward:
    """CE on this rank's vocabulary shard of given logits, reduced over the ranks."""
    ops = ops or CudaLogitsShardOps()
    return forward(logits_shard, None, labels, vocab_offset, V_total, None,
                   ignore_index=ignore_index, reduction=reduction,
                   num_label_tokens=num_label_tokens, exchange=exchange, ops=ops, status=status)


def ce_backward(logits_shard, labels, vocab_offset, V_total, fwd: ShardForward, grad_loss, *,
                ignore_index=-100, reduction="sum", num_label_tokens=None, inplace_grad=False,
                ops=None):
    """dZ of this rank's columns (no exchange needed)."""
    ops = ops or CudaLogitsShardOps()
    return ops.logits_backward(logits_shard, labels, vocab_offset, V_total, ignore_index,
                               reduction, num_label_tokens, fwd.lse, fwd.n_valid, grad_loss,
                               inplace_grad, fwd.status)


def forward(H, W_shard, labels, vocab_offset, V_total, bias_shard=None, *, ignore_index=-100,
            reduction="mean", num_label_tokens=None, exchange=None, ops=None,
            status=None) -> ShardForward:
    """Forward of this rank's vocabulary shard, reduced over the ranks."""
    ops = ops or CudaShardOps()
    exchange = exchange or TorchDistExchange()
    status = status if status is not None else new_status(H.device)
    labels = _labels(labels, H.shape[0]) if H.is_cuda else labels
    m, s, zy = ops.partials(H, W_shard, labels, vocab_offset, V_total, bias_shard, ignore_index,
                            status)
    m_global = exchange.max_(m.clone())
    s_scaled = exchange.sum_(ops.rescale(m, s, m_global))
    zy_global = exchange.sum_(zy)
    lse, loss, n_valid = ops.finish(m_global, s_scaled, zy_global, labels, V_total, ignore_index,
                                    reduction, num_label_tokens, status)
    return ShardForward(loss, n_valid, lse, status)


def backward(H, W_shard, labels, vocab_offset, V_total, fwd: ShardForward, grad_loss,
             bias_shard=None, *, ignore_index=-100, reduction="mean", num_label_tokens=None,
             chunk=None, want_grad_H=True, want_grad_W=True, exchange=None, ops=None):
    """(grad_H summed over the ranks, this shard's fp32 grad_W, its grad_bias).

    The ranks' grad_H partials are fp32; they are summed in fp32 and the sum is
    rounded once to H's dtype."""
    ops = ops or CudaShardOps()
    exchange = exchange or TorchDistExchange()
    gH, gW, gb = ops.backward(H, W_shard, labels, vocab_offset, V_total, bias_shard, ignore_index,
                              reduction, num_label_tokens, fwd.lse, fwd.n_valid, grad_loss, chunk,
                              want_grad_H, want_grad_W, fwd.status)
    if gH is not None:
        gH = exchange.sum_(gH).to(H.dtype)
    return gH, gW, gb
