"""Data-parallel rows: each rank holds a shard of the batch's rows.

The method partitions over rows: a shard's logits, row lse, loss and dX rows
depend on its own rows only. Two quantities couple the shards:

* the mean's denominator d (the number of valid rows, or the sum of their
  class weights; linear_cross_entropy.py, ``_ChunkContext.neg_weight_target``
  divides every row weight by it), which must be the WHOLE batch's for the
  shards' gradients to be their exact shares: each rank computes its local
  d with the library, the ranks all-reduce it (sum) and pass the total to the
  library as the given denominator;
* dW, db and the scalar loss, which are sums over rows: each rank's are its
  share, all-reduced (sum). dX rows stay on their rank.

So one step is: local d -> all-reduce(d) -> one library call per rank with
that d -> all-reduce(dW, db, loss). Gradients are requested in fp32 and
reduced in fp32 (a sum of bf16 shares would round once per rank), then cast
to ``grad_dtype``. With NCCL the reductions run on the device tensors; a
gloo group gets host copies.

``compute`` is the object that does the per-rank arithmetic: the library by
default (``LibraryCompute``); anything with the same two methods (tests use
a float64 one) can stand in for it, so the combination logic is testable on
CPU ranks.
"""

from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import lce_forward_backward, lce_mean_denominator


class LibraryCompute:
    """Per-rank arithmetic in liblce.so."""

    def denominator(self, target, C, ignore_index, class_weight):
        return lce_mean_denominator(target, C, ignore_index, class_weight)

    def forward_backward(self, X, W, b, target, reduction, ignore_index, grad_out, class_weight, denominator,
                         want_dx, want_dw, want_db):
        return lce_forward_backward(X, W, b, target, reduction, ignore_index, grad_out, want_dx=want_dx,
                                    want_dw=want_dw, want_db=want_db, grad_dtype=torch.float32,
                                    class_weight=class_weight, denominator=denominator)


def _all_reduce(t: torch.Tensor, group) -> torch.Tensor:
    """Sum over the ranks, in place; a gloo group reduces a host copy of a
    device tensor."""
    if t.is_cuda and dist.get_backend(group) == "gloo":
        h = t.cpu()
        dist.all_reduce(h, op=dist.ReduceOp.SUM, group=group)
        t.copy_(h)
    else:
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return t


def sharded_forward_backward(X, W, b, target, reduction: str = "mean", ignore_index: int = -100, grad_out=None,
                             class_weight=None, group=None, compute=None, grad_dtype=None, want_dx: bool = True,
                             want_dw: bool = True, want_db: bool = True):
    """Loss and gradients of the whole batch, from this rank's row shard.

    X [n_r, D], target [n_r]: this rank's rows (any split; a rank may hold
    none). W [C, D], b [C] or None, class_weight [C] or None: the same on
    every rank. grad_out: None or a scalar (mean, sum; the same on every
    rank), or this rank's rows' [n_r] upstream gradient (none).

    Returns (loss, dX, dW, db): loss is the whole batch's scalar (mean, sum)
    or this rank's rows' losses (none); dX this rank's rows; dW and db the
    whole batch's, identical on every rank; gradients in grad_dtype (default:
    X's dtype).
    """
    if compute is None:
        compute = LibraryCompute()
    C = W.shape[0]
    denom = None
    if reduction == "mean":
        d = compute.denominator(target, C, ignore_index, class_weight).reshape(1).to(torch.float64)
        _all_reduce(d, group)
        denom = d.to(torch.float32)
    loss, dX, dW, db = compute.forward_backward(X, W, b, target, reduction, ignore_index, grad_out, class_weight,
                                                denom, want_dx, want_dw, want_db and b is not None)
    if dW is not None:
        _all_reduce(dW, group)
    if db is not None:
        _all_reduce(db, group)
    if reduction != "none":
        loss = loss.reshape(1).to(torch.float64)
        _all_reduce(loss, group)
        loss = loss.to(torch.float32)[0]
    out_dtype = X.dtype if grad_dtype is None else grad_dtype
    cast = lambda t: None if t is None else t.to(out_dtype)
    return loss, cast(dX), cast(dW), cast(db)


def shard_rows(n_rows: int, world_size: int, rank: int) -> slice:
    """The contiguous rows [lo, hi) of rank ``rank`` when n_rows are split as
    evenly as possible (the first n_rows % world_size ranks get one more)."""
    base, extra = divmod(n_rows, world_size)
    lo = rank * base + min(rank, extra)
    return slice(lo, lo + base + (1 if rank < extra else 0))


__all__ = ["LibraryCompute", "sharded_forward_backward", "shard_rows"]
