"""PyTorch autograd on top of the C ABI.

``linear_cross_entropy(input, weight, target, bias=None, reduction="mean",
ignore_index=-100)`` returns the loss of the fused linear + cross-entropy
as a differentiable tensor. Every step of the computation runs in
liblce.so; this module only decides what to compute when, following the
split of the batch-chunked op in PyTorch's ``linear_cross_entropy.py``:

* reduction "mean" / "sum": the forward computes the loss and, in the same
  library call, the gradients of every input that requires one (the scalar
  ops of the page precompute the gradients); the backward multiplies them
  by the upstream gradient in place, in the library (a kernel that reads the
  upstream gradient on the device and does nothing when it is 1).
* reduction "none": the forward computes the per-row losses and lse and
  keeps the inputs; the backward recomputes the logits tile by tile from
  them and forms the vector-Jacobian product with the per-row upstream
  gradient in one call (the page's reduction="none" backward, which cannot
  keep the per-sample softmax).

Leading dimensions of ``input`` are flattened (``input.reshape(-1, D)``), as
in PyTorch commit ddfa80bd "Fix NJT linear_backward() memory usage".
Higher-order gradients are not supported.
"""

from __future__ import annotations

import torch

from . import lce_backward, lce_forward, lce_forward_backward, lce_scale_gradients


class _ScalarReduction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, W, b, target, reduction, ignore_index, class_weight, allow_retain_graph, plan):
        want_dx, want_dw, want_db = ctx.needs_input_grad[0], ctx.needs_input_grad[1], ctx.needs_input_grad[2]
        if want_dx or want_dw or want_db:
            loss, dX, dW, db = lce_forward_backward(X, W, b, target, reduction, ignore_index, None,
                                                    want_dx=want_dx, want_dw=want_dw,
                                                    want_db=want_db and b is not None, class_weight=class_weight,
                                                    **plan)
        else:
            loss = lce_forward(X, W, b, target, reduction, ignore_index, class_weight=class_weight)
            dX = dW = db = None
        ctx.grads = (dX, dW, db)
        ctx.allow_retain_graph = allow_retain_graph
        return loss

    @staticmethod
    def backward(ctx, grad_loss):
        if ctx.grads is None:
            raise RuntimeError("linear_cross_entropy: backward ran twice through a scalar-reduction loss whose "
                               "gradients were already handed out; pass allow_retain_graph=True to keep them")
        dX, dW, db = ctx.grads
        if ctx.allow_retain_graph:
            # keep the precomputed buffers for a later backward: scale copies
            dX, dW, db = (None if x is None else x.clone() for x in (dX, dW, db))
        else:
            ctx.grads = None
        # in place, in the library; its kernel leaves them untouched when the
        # upstream gradient is 1 (decided on the device: no host sync)
        lce_scale_gradients(dX, dW, db, grad_loss)
        return dX, dW, db, None, None, None, None, None, None


class _NoReduction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, X, W, b, target, ignore_index, class_weight, plan):
        loss, lse = lce_forward(X, W, b, target, "none", ignore_index, want_lse=True, class_weight=class_weight)
        ctx.save_for_backward(X, W, b, target, lse)
        ctx.ignore_index = ignore_index
        ctx.class_weight = class_weight
        ctx.plan = plan
        return loss

    @staticmethod
    def backward(ctx, grad_loss):
        X, W, b, target, lse = ctx.saved_tensors
        need = ctx.needs_input_grad
        dX, dW, db = lce_backward(X, W, b, target, lse, "none", ctx.ignore_index,
                                  grad_loss.to(torch.float32).reshape(-1).contiguous(),
                                  want_dx=need[0], want_dw=need[1], want_db=need[2] and b is not None,
                                  class_weight=ctx.class_weight, **ctx.plan)
        return dX, dW, db, None, None, None, None


def linear_cross_entropy(input, weight, target, bias=None, reduction="mean", ignore_index=-100, class_weight=None,
                         allow_retain_graph=False, chunk_rows=0, buffer_bytes=None):
    """Loss of cross_entropy(input @ weight.T + bias, target) without the
    [rows, classes] logits, differentiable in input, weight and bias.

    input [..., D] (fp32, bf16 or fp16), weight [C, D], bias [C] or None
    (same dtype), target [...] int64, class_weight [C] or None (per-class
    weights of cross entropy, not differentiated). Returns a float32 scalar
    (mean, sum) or a float32 tensor of target's shape (none).

    allow_retain_graph (mean / sum only, as the page's option of that name):
    False hands the precomputed gradient buffers to the backward, which
    scales them in place, so a second backward through the same loss raises
    RuntimeError; True keeps them and scales copies (one more gradient-sized
    allocation per backward). reduction "none" recomputes in its backward and
    supports retain_graph either way.

    chunk_rows / buffer_bytes choose the workspace plan of the gradient call
    (the page's batch_chunk_size / chunking_method): 0 / None is the
    library's default (a gradient buffer of at most 1 GiB); chunk_rows > 0
    gives batch chunks of that many rows with every class (e.g.
    lce_aspect_ratio_chunk_rows(N, D, C) for the page's "aspect_ratio");
    buffer_bytes bounds the buffer at that many bytes instead.
    """
    if reduction not in ("mean", "sum", "none"):
        raise ValueError(f"reduction must be mean, sum or none, got {reduction!r}")
    D = input.shape[-1]
    X = input.reshape(-1, D).contiguous()
    t = target.reshape(-1).contiguous()
    if t.shape[0] != X.shape[0]:
        raise ValueError("target must have one entry per row of input")
    W = weight.contiguous()
    b = None if bias is None else bias.contiguous()
    plan = {"chunk_rows": chunk_rows, "buffer_bytes": buffer_bytes}
    if reduction == "none":
        return _NoReduction.apply(X, W, b, t, ignore_index, class_weight, plan).reshape(target.shape)
    return _ScalarReduction.apply(X, W, b, t, reduction, ignore_index, class_weight, allow_retain_graph, plan)
