"""Float64 CPU oracle for the fused linear + cross-entropy loss.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or
executes this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code, helper or constant with the CUDA library.

What it computes is the plain definition of the method, written out step by
step in float64 with numpy (the matmul is the only library primitive used):

  z[n, j]   = sum_d X[n, d] * W[j, d] + b[j]                  (logits)
  valid_n   = target_n != ignore_index ;  n_valid = sum valid_n
  lse_n     = m_n + log sum_j exp(z[n, j] - m_n),  m_n = max_j z[n, j]
  loss_n    = valid_n ? lse_n - z[n, target_n] : 0
  loss      = none: loss_n | sum: sum_n loss_n | mean: sum_n loss_n / n_valid
              (or / d for a given denominator d: a data-parallel shard of a
              batch divides by the whole batch's n_valid)
  w_n       = c_n * (mean: g / sum_n c_n | sum: g | none: g_n),
              c_n = valid_n * weight[target_n] (weight = 1 without class weights)
  (with class weights loss_n is c_n (lse_n - z[n, target_n]) and mean
   divides by sum_n c_n)
  G[n, j]   = w_n * (exp(z[n, j] - lse_n) - [j == target_n])
  dX = G W ,  dW = G^T X ,  db = sum_n G[n, :]

Sources (the web pages this method is taken from):
  * PyTorch source ``torch/nn/modules/linear_cross_entropy.py``
    (batch-chunked linear + cross-entropy): the loop body of
    ``_linear_cross_entropy_batch_chunked_accumulator`` (max shift, target
    gather, sum-exp, log, scaling of the logits by w/denominator, the input,
    weight and bias gradient updates) and ``_ChunkContext.neg_weight_target``
    (per-row weight: 0 on ignored rows, -1/d for mean with NaN when d == 0,
    -1 for sum, +1 forward / -grad_output backward for none).
  * PyTorch commit ddfa80bd "Fix NJT linear_backward() memory usage":
    dX = G W, dW = G^T X over rows flattened to 2-D, db = row sum of G.
  * Liger-Kernel issue #343 "cross entropy kernel: inplace modification of
    input": cross entropy on given logits whose gradient replaces the logits.

Sign convention: the page accumulates ``-w`` times the loss pieces and then
negates; here w_n is the positive weight of row n in the loss, so that
G = dLoss/dz directly. Both give the same loss and gradients.

Parity pins (see tests/test_oracle_pins.py): closed forms for uniform
logits and for X = 0, C = 1, the Sigma_j G = 0 invariant, ignored rows,
reduction identities, bias-shift invariance, row permutation, linearity in
the upstream gradient, float64 central finite differences, a pure-Python
brute force on tiny inputs, and torch's own float64 ``cross_entropy`` +
autograd. Every function below is pinned by at least one of them.
"""

from __future__ import annotations

import math

import numpy as np

REDUCTIONS = ("none", "sum", "mean")
DEFAULT_IGNORE_INDEX = -100
# Rows per block for the blockwise passes: keeps the [rows, C] float64 block
# bounded (256 x 131072 x 8 B = 268 MB) instead of holding the whole [N, C].
ROW_BLOCK = 256


class OracleError(ValueError):
    """Raised for inputs the method does not define (e.g. a target that is
    neither a class index nor ignore_index)."""


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _check_reduction(reduction: str) -> None:
    if reduction not in REDUCTIONS:
        raise OracleError(f"reduction must be one of {REDUCTIONS}, got {reduction!r}")


def valid_mask(target: np.ndarray, num_classes: int, ignore_index: int) -> np.ndarray:
    """valid_n = (target_n != ignore_index).

    linear_cross_entropy.py, ``_ChunkContext._mask``: a row is ignored iff its
    target equals ignore_index; an ignore_index inside [0, C) still leaves
    that class as an ordinary softmax column. A target that is neither
    ignore_index nor in [0, C) is undefined on the page (its gather would
    fault) and raises here.
    """
    target = np.asarray(target, dtype=np.int64)
    valid = target != ignore_index
    bad = valid & ((target < 0) | (target >= num_classes))
    if bad.any():
        raise OracleError(
            f"target out of range [0, {num_classes}) at rows {np.nonzero(bad)[0][:8].tolist()}"
        )
    return valid


def corrected_target(target: np.ndarray, valid: np.ndarray) -> np.ndarray:
    """Target with ignored rows mapped to class 0 so gathers stay in bounds
    (linear_cross_entropy.py, ``_ChunkContext.corrected_target``). Those rows
    carry w_n = 0, so the class chosen does not matter."""
    return np.where(valid, np.asarray(target, dtype=np.int64), 0)


def class_weight_of_rows(target, valid, class_weight):
    """c_n = weight[target_n] on valid rows (1 without class weights), 0 on
    ignored rows (linear_cross_entropy.py, neg_weight_target: the masked
    index_select of the per-class weight)."""
    v = valid.astype(np.float64)
    if class_weight is None:
        return v
    cw = _f64(class_weight).reshape(-1)
    return v * cw[corrected_target(target, valid)]


def row_weights(target, num_classes, reduction, ignore_index=DEFAULT_IGNORE_INDEX, grad_out=None,
                class_weight=None, denominator=None):
    """Per-row loss weight w_n, with the upstream gradient folded in.

    linear_cross_entropy.py, ``_ChunkContext.neg_weight_target``: ignored
    rows get 0, valid rows the class weight weight[target_n] (1 without
    class weights); mean divides by d = sum of those weights and gives NaN
    for every row when d == 0; sum uses them as they are; none multiplies
    them by grad_output[n] in the backward. For mean and sum the scalar
    upstream gradient multiplies the precomputed gradients
    (``_linear_cross_entropy_batch_chunked_backward``:
    ``grad.mul_(grad_output)``); it is folded into w_n here. grad_out=None
    means 1.0 for mean/sum and is required for none. denominator: None, or
    the d that mean divides by instead of these rows' own (a shard of a
    larger batch divides by the whole batch's d, so that the shards' results
    add up to the whole batch's).
    """
    _check_reduction(reduction)
    valid = valid_mask(target, num_classes, ignore_index)
    v = class_weight_of_rows(np.asarray(target, dtype=np.int64), valid, class_weight)
    if reduction == "none":
        if grad_out is None:
            raise OracleError("reduction='none' needs a per-row upstream gradient")
        g = _f64(grad_out).reshape(-1)
        if g.shape[0] != v.shape[0]:
            raise OracleError("grad_out must have one entry per row for reduction='none'")
        return v * g
    g = 1.0 if grad_out is None else float(np.asarray(grad_out, dtype=np.float64).reshape(-1)[0])
    if reduction == "sum":
        return v * g
    d = v.sum() if denominator is None else float(denominator)
    inv = math.nan if d == 0 else 1.0 / d
    return v * (inv * g)  # 0 * NaN = NaN: all rows NaN when n_valid == 0


def logits_block(X, W, b=None) -> np.ndarray:
    """z = X W^T + b for a block of rows (the page's ``ctx.mm`` plus the bias
    add); X [n, D], W [C, D], b [C] or None."""
    z = _f64(X) @ _f64(W).T
    if b is not None:
        z = z + _f64(b)[None, :]
    return z


def log_sum_exp(z: np.ndarray) -> np.ndarray:
    """Textbook row log-sum-exp with the max shift: m + log sum exp(z - m)
    (the page's ``amax`` / ``sub_`` / ``sumexp_`` / ``log`` sequence)."""
    m = z.max(axis=1)
    with np.errstate(invalid="ignore", over="ignore"):
        return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def _reduce(loss_rows: np.ndarray, c: np.ndarray, reduction: str, denominator=None):
    """c: per-row class weights (0 on ignored rows; the valid mask without
    class weights); mean divides by their sum, or by the given denominator."""
    if reduction == "none":
        return loss_rows
    total = float(loss_rows.sum())
    if reduction == "sum":
        return total
    d = float(np.asarray(c, dtype=np.float64).sum()) if denominator is None else float(denominator)
    # mean over the valid rows; N == 0 or all rows ignored gives NaN
    # (linear_cross_entropy.py: the empty-batch mean and neg_weight_target's
    # d == 0 case).
    return math.nan if d == 0 else total / d


def ce_from_logits(logits, target, reduction="mean", ignore_index=DEFAULT_IGNORE_INDEX,
                   grad_out=None, want_grad=True, class_weight=None, denominator=None):
    """Cross entropy on given logits [N, V], and the gradient that replaces them.

    Liger-Kernel issue #343: one pass gives the loss and writes
    dLoss/dlogits (times the upstream gradient) into the logits buffer. This
    returns (loss, grad) instead of overwriting anything; grad[n, j] =
    w_n * (softmax(z_n)_j - [j == target_n]).
    """
    z = _f64(logits)
    N, V = z.shape
    target = np.asarray(target, dtype=np.int64).reshape(-1)
    valid = valid_mask(target, V, ignore_index)
    tc = corrected_target(target, valid)
    c = class_weight_of_rows(target, valid, class_weight)
    loss_rows = np.zeros(N)
    grad = np.zeros_like(z) if want_grad else None
    w = None
    if want_grad:
        w = row_weights(target, V, reduction, ignore_index, grad_out, class_weight, denominator)
    for r0 in range(0, N, ROW_BLOCK):
        r1 = min(N, r0 + ROW_BLOCK)
        zb = z[r0:r1]
        lse = log_sum_exp(zb)
        rows = np.arange(r1 - r0)
        zt = zb[rows, tc[r0:r1]]
        with np.errstate(invalid="ignore"):  # an ignored row's placeholder column may be -inf
            loss_rows[r0:r1] = np.where(valid[r0:r1], c[r0:r1] * (lse - zt), 0.0)
        if want_grad:
            P = np.exp(zb - lse[:, None])
            P[rows, tc[r0:r1]] -= valid[r0:r1].astype(np.float64)
            grad[r0:r1] = w[r0:r1, None] * P
    return _reduce(loss_rows, c, reduction, denominator), grad


def lce_forward(X, W, b, target, reduction="mean", ignore_index=DEFAULT_IGNORE_INDEX, class_weight=None,
                denominator=None):
    """Loss of the fused linear + cross-entropy, and lse per row.

    Returns (loss, lse[N]); loss is a float for sum/mean and loss_n [N] for
    none. linear_cross_entropy.py: the chunked forward (``ctx.mm``, max
    shift, ``dotgather``, ``sumexp_``, ``output.sub_(log ...)``) and the
    reduction='none' loss-only branch.
    """
    _check_reduction(reduction)
    X = _f64(X)
    W = _f64(W)
    N = X.shape[0]
    C = W.shape[0]
    target = np.asarray(target, dtype=np.int64).reshape(-1)
    valid = valid_mask(target, C, ignore_index)
    tc = corrected_target(target, valid)
    c = class_weight_of_rows(target, valid, class_weight)
    lse = np.zeros(N)
    loss_rows = np.zeros(N)
    for r0 in range(0, N, ROW_BLOCK):
        r1 = min(N, r0 + ROW_BLOCK)
        z = logits_block(X[r0:r1], W, b)
        lse[r0:r1] = log_sum_exp(z)
        zt = z[np.arange(r1 - r0), tc[r0:r1]]
        with np.errstate(invalid="ignore"):  # an ignored row's placeholder column may be -inf
            loss_rows[r0:r1] = np.where(valid[r0:r1], c[r0:r1] * (lse[r0:r1] - zt), 0.0)
    return _reduce(loss_rows, c, reduction, denominator), lse


def lce_forward_backward(X, W, b, target, reduction="mean", ignore_index=DEFAULT_IGNORE_INDEX,
                         grad_out=None, class_weight=None, denominator=None):
    """Loss and all gradients (dX, dW, db) of the fused linear + cross-entropy.

    Returns (loss, dX[N, D], dW[C, D], db[C] or None). For mean/sum the
    gradients are those of the loss times the scalar upstream gradient
    (None = 1.0); for none they are the vector-Jacobian product with the
    per-row upstream gradient. linear_cross_entropy.py: scaling of the
    shifted exp-logits by w/denominator, then ``addmm`` / ``index_select``
    for the input gradient, ``addmm_`` / ``index_add_`` for the weight
    gradient and the row sum / ``index_add_`` for the bias gradient; commit
    ddfa80bd for dX = G W, dW = G^T X, db = sum_n G.
    """
    _check_reduction(reduction)
    X = _f64(X)
    W = _f64(W)
    N, D = X.shape
    C = W.shape[0]
    target = np.asarray(target, dtype=np.int64).reshape(-1)
    valid = valid_mask(target, C, ignore_index)
    tc = corrected_target(target, valid)
    c = class_weight_of_rows(target, valid, class_weight)
    w = row_weights(target, C, reduction, ignore_index, grad_out, class_weight, denominator)
    loss_rows = np.zeros(N)
    dX = np.zeros((N, D))
    dW = np.zeros((C, D))
    db = np.zeros(C) if b is not None else None
    for r0 in range(0, N, ROW_BLOCK):
        r1 = min(N, r0 + ROW_BLOCK)
        rows = np.arange(r1 - r0)
        z = logits_block(X[r0:r1], W, b)
        lse = log_sum_exp(z)
        zt = z[rows, tc[r0:r1]]
        with np.errstate(invalid="ignore"):  # an ignored row's placeholder column may be -inf
            loss_rows[r0:r1] = np.where(valid[r0:r1], c[r0:r1] * (lse - zt), 0.0)
        G = np.exp(z - lse[:, None])
        G[rows, tc[r0:r1]] -= valid[r0:r1].astype(np.float64)
        G *= w[r0:r1, None]
        dX[r0:r1] = G @ W
        dW += G.T @ X[r0:r1]
        if db is not None:
            db += G.sum(axis=0)
    return _reduce(loss_rows, c, reduction, denominator), dX, dW, db


# --------------------------------------------------------------------------
# Sampled evaluation for the large configurations. The same definitions,
# evaluated on a subset of the outputs: every row's lse is needed for the
# loss and for any dW row, so ``forward_stats`` makes one full blockwise
# pass; the sampled dX and dW rows then follow from the definitions above.
# --------------------------------------------------------------------------


def forward_stats(X, W, b, target, reduction="mean", ignore_index=DEFAULT_IGNORE_INDEX,
                  grad_out=None, want_db=False, row_block=ROW_BLOCK, class_weight=None):
    """One full blockwise pass: lse[N], loss_n[N], the reduced loss, w[N]
    and (optionally) db[C] = sum_n G[n, :]. X and W may be float32/bfloat16
    values held in float32 arrays; each block is upcast to float64. With
    class weights (the page's weight option), a valid row's loss is
    weight[t_n] (lse_n - z_t) and mean divides by the sum of those weights,
    as in lce_forward."""
    _check_reduction(reduction)
    N = X.shape[0]
    C = W.shape[0]
    target = np.asarray(target, dtype=np.int64).reshape(-1)
    valid = valid_mask(target, C, ignore_index)
    tc = corrected_target(target, valid)
    c = class_weight_of_rows(target, valid, class_weight)
    w = row_weights(target, C, reduction, ignore_index,
                    grad_out if (grad_out is not None or reduction != "none") else np.ones(N),
                    class_weight=class_weight)
    W64 = _f64(W)
    lse = np.zeros(N)
    loss_rows = np.zeros(N)
    db = np.zeros(C) if (want_db and b is not None) else None
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        rows = np.arange(r1 - r0)
        z = logits_block(X[r0:r1], W64, b)
        l = log_sum_exp(z)
        lse[r0:r1] = l
        loss_rows[r0:r1] = np.where(valid[r0:r1], c[r0:r1] * (l - z[rows, tc[r0:r1]]), 0.0)
        if db is not None:
            G = np.exp(z - l[:, None])
            G[rows, tc[r0:r1]] -= valid[r0:r1].astype(np.float64)
            db += (w[r0:r1, None] * G).sum(axis=0)
    return {
        "lse": lse,
        "loss_rows": loss_rows,
        "loss": _reduce(loss_rows, c, reduction),
        "w": w,
        "valid": valid,
        "db": db,
    }


def grad_rows(X, W, b, target, lse, w, rows, ignore_index=DEFAULT_IGNORE_INDEX):
    """G[rows, :] and dX[rows, :] = G[rows, :] W for sampled rows, given the
    full-pass lse and w."""
    rows = np.asarray(rows, dtype=np.int64)
    C = W.shape[0]
    target = np.asarray(target, dtype=np.int64).reshape(-1)
    valid = valid_mask(target[rows], C, ignore_index)
    tc = corrected_target(target[rows], valid)
    W64 = _f64(W)
    z = logits_block(X[rows], W64, b)
    G = np.exp(z - lse[rows][:, None])
    G[np.arange(len(rows)), tc] -= valid.astype(np.float64)
    G *= w[rows][:, None]
    return G, G @ W64


def dw_rows(X, W, b, target, lse, w, classes, ignore_index=DEFAULT_IGNORE_INDEX,
            row_block=4096):
    """dW[classes, :] = sum_n G[n, classes]^T X[n, :] over every row n, given
    the full-pass lse and w. Also returns db[classes]."""
    classes = np.asarray(classes, dtype=np.int64)
    N, D = X.shape
    target = np.asarray(target, dtype=np.int64).reshape(-1)
    valid = valid_mask(target, W.shape[0], ignore_index)
    Wc = _f64(W[classes])
    bc = None if b is None else _f64(b)[classes]
    out = np.zeros((len(classes), D))
    dbc = np.zeros(len(classes))
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        Xb = _f64(X[r0:r1])
        z = logits_block(Xb, Wc, bc)
        G = np.exp(z - lse[r0:r1, None])
        G -= ((target[r0:r1, None] == classes[None, :]) & valid[r0:r1, None]).astype(np.float64)
        G *= w[r0:r1, None]
        out += G.T @ Xb
        dbc += G.sum(axis=0)
    return out, dbc


def ce_rows(logits_rows, target_rows, w_rows, ignore_index=DEFAULT_IGNORE_INDEX):
    """Per-row loss and gradient rows of cross entropy on given logits, for
    sampled rows (w_rows from ``row_weights`` over all rows)."""
    z = _f64(logits_rows)
    V = z.shape[1]
    t = np.asarray(target_rows, dtype=np.int64).reshape(-1)
    valid = valid_mask(t, V, ignore_index)
    tc = corrected_target(t, valid)
    lse = log_sum_exp(z)
    r = np.arange(z.shape[0])
    loss_rows = np.where(valid, lse - z[r, tc], 0.0)
    G = np.exp(z - lse[:, None])
    G[r, tc] -= valid.astype(np.float64)
    G *= _f64(w_rows)[:, None]
    return loss_rows, G
