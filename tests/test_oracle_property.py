"""Property-based pins of the oracle: over randomly drawn tiny problems
(shapes, reduction, ignored rows, ignore_index inside or outside [0, C),
bias, class weights, upstream gradient), the oracle's loss, dX, dW and db
equal float64 torch autograd through torch.nn.functional.cross_entropy, and
its CE-from-logits equals the same on the logits. Independent of the CUDA
path; runs on the CPU."""

import numpy as np
import pytest
import torch

from oracle import lce_oracle as O

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")


@st.composite
def problems(draw):
    N = draw(st.integers(1, 9))
    D = draw(st.integers(1, 6))
    C = draw(st.integers(1, 9))
    reduction = draw(st.sampled_from(["mean", "sum", "none"]))
    inside = draw(st.booleans()) and C > 1
    ignore_index = draw(st.integers(0, C - 1)) if inside else -100
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    X = rng.normal(size=(N, D)) * draw(st.sampled_from([0.1, 1.0, 3.0]))
    W = rng.normal(size=(C, D)) * draw(st.sampled_from([0.1, 1.0, 3.0]))
    b = rng.normal(size=C) * 0.5 if draw(st.booleans()) else None
    t = rng.integers(0, C, size=N).astype(np.int64)
    n_ign = draw(st.integers(0, N))
    if reduction == "mean":
        n_ign = min(n_ign, N - 1)  # the all-ignored mean is pinned on its own (NaN)
    if n_ign and not inside:
        t[rng.permutation(N)[:n_ign]] = ignore_index
    elif inside:
        # rows whose target equals ignore_index are the ignored ones
        keep = rng.permutation(N)[n_ign:]
        for n in keep:
            if t[n] == ignore_index:
                t[n] = (ignore_index + 1) % C
        if reduction == "mean" and np.all(t == ignore_index):
            t[0] = (ignore_index + 1) % C
    cw = rng.uniform(0.2, 2.0, size=C) if draw(st.booleans()) else None
    if reduction == "none":
        g = rng.normal(size=N)
    elif reduction == "sum":
        g = float(draw(st.sampled_from([1.0, 0.5, -2.0])))
    else:
        g = None
    return X, W, b, t, reduction, ignore_index, g, cw


def _torch_reference(X, W, b, t, reduction, ignore_index, g, cw):
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    bt = None if b is None else torch.tensor(b, dtype=torch.float64, requires_grad=True)
    z = Xt @ Wt.T + (bt if bt is not None else 0.0)
    loss = torch.nn.functional.cross_entropy(
        z, torch.tensor(t), weight=None if cw is None else torch.tensor(cw, dtype=torch.float64),
        ignore_index=ignore_index, reduction=reduction)
    if reduction == "none":
        loss.backward(torch.tensor(g, dtype=torch.float64))
    else:
        loss.backward(torch.tensor(1.0 if g is None else g, dtype=torch.float64))
    return (loss.detach().numpy(), Xt.grad.numpy(), Wt.grad.numpy(),
            None if bt is None else bt.grad.numpy())


@hyp.settings(max_examples=150, deadline=None)
@hyp.given(problems())
def test_oracle_matches_torch_autograd(p):
    X, W, b, t, reduction, ignore_index, g, cw = p
    loss, dX, dW, db = O.lce_forward_backward(X, W, b, t, reduction, ignore_index, g, class_weight=cw)
    rl, rX, rW, rb = _torch_reference(X, W, b, t, reduction, ignore_index, g, cw)
    np.testing.assert_allclose(loss, rl, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dX, rX, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dW, rW, rtol=1e-9, atol=1e-12)
    if b is not None:
        np.testing.assert_allclose(db, rb, rtol=1e-9, atol=1e-12)
        # every row of G sums to 0 over the classes, hence so does db
        assert abs(db.sum()) <= 1e-9 * max(1.0, np.abs(db).sum())


@hyp.settings(max_examples=100, deadline=None)
@hyp.given(problems())
def test_ce_from_logits_matches_torch_autograd(p):
    X, W, b, t, reduction, ignore_index, g, cw = p
    logits = X @ W.T
    loss, grad = O.ce_from_logits(logits, t, reduction, ignore_index, g, class_weight=cw)
    zt = torch.tensor(logits, dtype=torch.float64, requires_grad=True)
    ref = torch.nn.functional.cross_entropy(
        zt, torch.tensor(t), weight=None if cw is None else torch.tensor(cw, dtype=torch.float64),
        ignore_index=ignore_index, reduction=reduction)
    ref.backward(torch.tensor(g if g is not None else 1.0, dtype=torch.float64))
    np.testing.assert_allclose(loss, ref.detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(grad, zt.grad.numpy(), rtol=1e-9, atol=1e-12)


@hyp.settings(max_examples=100, deadline=None)
@hyp.given(problems(), st.integers(0, 2**31 - 1))
def test_masked_classes_equal_deleted_classes(p, seed):
    """A bias of -inf on a random proper subset of the classes (none of them
    a target) gives the same loss and dX as the problem with those classes
    deleted and the targets renumbered, and zero dW rows and db entries for
    them."""
    X, W, b, t, reduction, ignore_index, g, cw = p
    C = W.shape[0]
    hyp.assume(C > 1)
    rng = np.random.default_rng(seed)
    valid = t != ignore_index
    used = np.zeros(C, dtype=bool)
    used[t[valid]] = True
    free = np.flatnonzero(~used)
    masked = np.zeros(C, dtype=bool)
    masked[free[rng.random(free.size) < 0.5]] = True
    hyp.assume(masked.any() and not masked.all())
    hyp.assume(not (0 <= ignore_index < C and masked[ignore_index]))
    keep = np.flatnonzero(~masked)
    renum = np.full(C, -1)
    renum[keep] = np.arange(keep.size)
    ign_r = renum[ignore_index] if 0 <= ignore_index < C else ignore_index
    tr = np.where(valid, renum[np.where(valid, t, 0)], ign_r)
    b0 = np.zeros(C) if b is None else b
    bm = b0.copy()
    bm[masked] = -np.inf
    cwr = None if cw is None else cw[keep]
    loss, dX, dW, db = O.lce_forward_backward(X, W, bm, t, reduction, ignore_index, g, class_weight=cw)
    rl, rX, rW, rb = O.lce_forward_backward(X, W[keep], b0[keep], tr, reduction, ign_r, g, class_weight=cwr)
    np.testing.assert_allclose(loss, rl, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dX, rX, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dW[keep], rW, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(db[keep], rb, rtol=1e-9, atol=1e-12)
    assert (dW[masked] == 0).all() and (db[masked] == 0).all()
