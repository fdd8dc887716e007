"""Data-parallel use of the loss head.

Tokens are independent, so each rank runs the whole path (forward and
backward kernels) on its own rows and no collective sits on the data path.
Two reductions make the per-rank results add up to those of one global
problem:

* ``global_num_label_tokens``: the valid-label count of every rank, summed.
  Passed as ``num_label_tokens`` to every rank's call, it makes each rank's
  loss and gradients exactly its share of the global mean (the
  ``num_label_tokens`` divisor of Automodel PR #2996, first commit message).
* ``combine_loss``: the per-rank summed losses and counts, summed, for
  reporting the global loss.

grad_W / grad_bias are then all-reduced like any data-parallel gradient by
the trainer.  ``shard_rows`` gives each rank a contiguous, balanced slice.
The collectives run on whatever process group is passed (NCCL for CUDA
tensors, gloo for CPU tensors).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _abi


def shard_rows(N: int, rank: int, world: int):
    """Contiguous slice [start, stop) of N rows for `rank` out of `world`
    (sizes differ by at most one)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(N, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def local_valid_count(labels: torch.Tensor, V: int, ignore_index: int = -100) -> torch.Tensor:
    """[1] int64 on the labels' device: labels that are not ignore_index and lie
    in [0, V), counted by the library's kernel."""
    if not labels.is_cuda:
        raise ValueError("labels must be a CUDA tensor")
    labels = labels.contiguous()
    out = torch.empty(1, dtype=torch.int64, device=labels.device)
    rc = _abi.flce_count_valid(labels.data_ptr(), labels.numel(), int(V), int(ignore_index),
                               out.data_ptr(), torch.cuda.current_stream(labels.device).cuda_stream)
    _abi.check(rc, "flce_count_valid")
    return out


def all_reduce_count(count: torch.Tensor, group=None) -> torch.Tensor:
    """Sum of a [1] int64 count over the ranks of `group` (in place)."""
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(count, op=dist.ReduceOp.SUM, group=group)
    return count


def global_num_label_tokens(labels: torch.Tensor, V: int, ignore_index: int = -100,
                            group=None) -> int:
    """The valid-label count over all ranks (one scalar all-reduce)."""
    return int(all_reduce_count(local_valid_count(labels, V, ignore_index), group).item())


def combine_loss(loss_sum: torch.Tensor, n_valid: torch.Tensor, group=None):
    """Global (sum, count, mean) from per-rank summed losses and counts (one
    all-reduce of two numbers, in float64)."""
    t = torch.stack([loss_sum.reshape(()).to(torch.float64),
                     n_valid.reshape(()).to(torch.float64)])
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    s, n = float(t[0]), int(round(float(t[1])))
    return s, n, (s / n if n > 0 else 0.0)
