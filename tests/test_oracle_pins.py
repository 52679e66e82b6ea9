"""Pins for the float64 oracle: closed forms, invariants, finite differences,
torch's own float64 cross entropy + autograd, and planted mistakes that the
pins must catch. CPU only."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import lce_oracle as O

RNG = np.random.default_rng(1234)


def _rand_case(N=13, D=7, C=11, bias=True, n_ign=3, ignore_index=-100, seed=0):
    r = np.random.default_rng(seed)
    X = r.standard_normal((N, D))
    W = r.standard_normal((C, D)) * 0.7
    b = r.standard_normal(C) * 0.3 if bias else None
    t = r.integers(0, C, N)
    if n_ign:
        t[r.permutation(N)[:n_ign]] = ignore_index
    return X, W, b, t


def _torch_ref(X, W, b, t, reduction, ignore_index, grad_out):
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True) if b is not None else None
    z = F.linear(Xt, Wt, bt)
    loss = F.cross_entropy(z, torch.tensor(t, dtype=torch.int64), reduction=reduction,
                           ignore_index=ignore_index)
    if reduction == "none":
        loss.backward(torch.tensor(grad_out, dtype=torch.float64))
    else:
        g = 1.0 if grad_out is None else float(grad_out)
        (loss * g).backward()
    return (loss.detach().numpy(), Xt.grad.numpy(), Wt.grad.numpy(),
            None if bt is None else bt.grad.numpy())


def _matches_torch(fb, X, W, b, t, reduction, ignore_index, grad_out, tol=1e-10):
    loss, dX, dW, db = fb(X, W, b, t, reduction, ignore_index, grad_out)
    rl, rX, rW, rb = _torch_ref(X, W, b, t, reduction, ignore_index, grad_out)
    ok = np.allclose(loss, rl, rtol=tol, atol=tol)
    ok &= np.allclose(dX, rX, rtol=tol, atol=tol)
    ok &= np.allclose(dW, rW, rtol=tol, atol=tol)
    if b is not None:
        ok &= np.allclose(db, rb, rtol=tol, atol=tol)
    return bool(ok)


CASES = [
    ("mean", -100, None, True),
    ("mean", -100, 2.5, False),
    ("sum", -100, None, True),
    ("sum", 4, -0.75, True),  # ignore_index inside [0, C)
    ("none", -100, "vec", True),
    ("none", 2, "vec", False),
]


@pytest.mark.parametrize("reduction,ignore_index,g,bias", CASES)
def test_against_torch_cross_entropy_autograd(reduction, ignore_index, g, bias):
    X, W, b, t = _rand_case(bias=bias, ignore_index=ignore_index)
    if g == "vec":
        g = RNG.standard_normal(X.shape[0])
    assert _matches_torch(O.lce_forward_backward, X, W, b, t, reduction, ignore_index, g)
    loss_f, lse = O.lce_forward(X, W, b, t, reduction, ignore_index)
    loss_fb = O.lce_forward_backward(X, W, b, t, reduction, ignore_index, g)[0]
    np.testing.assert_allclose(loss_f, loss_fb, rtol=1e-13)
    z = X @ W.T + (b if b is not None else 0)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.tensor(z), 1).numpy(), rtol=1e-13)


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
def test_finite_differences(reduction):
    X, W, b, t = _rand_case(N=5, D=4, C=6, n_ign=1, seed=3)
    g = RNG.standard_normal(5) if reduction == "none" else 1.0

    def f(X_, W_, b_):
        loss, _ = O.lce_forward(X_, W_, b_, t, reduction)
        return float(np.dot(loss, g)) if reduction == "none" else float(loss)

    _, dX, dW, db = O.lce_forward_backward(X, W, b, t, reduction, grad_out=g)
    h = 1e-6
    for A, grad in ((X, dX), (W, dW), (b, db)):
        num = np.zeros_like(A)
        for idx in np.ndindex(A.shape):
            old = A[idx]
            A[idx] = old + h
            fp = f(X, W, b)
            A[idx] = old - h
            fm = f(X, W, b)
            A[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8)


def test_pure_python_brute_force_tiny():
    X, W, b, t = _rand_case(N=4, D=3, C=5, n_ign=1, seed=7)
    N, C = 4, 5
    losses = []
    for n in range(N):
        if t[n] == -100:
            losses.append(0.0)
            continue
        z = [sum(X[n, d] * W[j, d] for d in range(3)) + b[j] for j in range(C)]
        losses.append(math.log(sum(math.exp(v) for v in z)) - z[t[n]])
    loss, _ = O.lce_forward(X, W, b, t, "none")
    np.testing.assert_allclose(loss, losses, rtol=1e-12)


@pytest.mark.parametrize("C", [512, 8192, 128256, 131072])
def test_uniform_logits_closed_form(C):
    # W = 0, b = 0: every logit equal, so loss_n = ln C and G = w(1/C - onehot).
    N, D = 6, 4
    X = RNG.standard_normal((N, D))
    W = np.zeros((C, D))
    t = RNG.integers(0, C, N)
    t[1] = -100
    loss, dX, dW, db = O.lce_forward_backward(X, W, np.zeros(C), t, "mean")
    assert abs(loss - math.log(C)) < 1e-12
    nv = 5
    np.testing.assert_allclose(dX, 0.0, atol=1e-15)
    exp_db = np.full(C, nv / C / nv)
    for n in range(N):
        if t[n] != -100:
            exp_db[t[n]] -= 1.0 / nv
    np.testing.assert_allclose(db, exp_db, rtol=1e-10, atol=1e-15)
    exp_dW = np.zeros((C, D))
    for n in range(N):
        if t[n] != -100:
            exp_dW += X[n][None, :] / C / nv
            exp_dW[t[n]] -= X[n] / nv
    np.testing.assert_allclose(dW, exp_dW, rtol=1e-10, atol=1e-14)


def test_zero_input_closed_form():
    # X = 0, b = 0: z = 0, P = 1/C, dX_n = w_n (mean_j W_j - W_t), dW = 0.
    N, D, C = 7, 5, 9
    X = np.zeros((N, D))
    W = RNG.standard_normal((C, D))
    t = RNG.integers(0, C, N)
    loss, dX, dW, db = O.lce_forward_backward(X, W, np.zeros(C), t, "sum", grad_out=1.5)
    assert abs(loss - N * math.log(C)) < 1e-12
    for n in range(N):
        np.testing.assert_allclose(dX[n], 1.5 * (W.mean(0) - W[t[n]]), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dW, 0.0, atol=1e-15)
    counts = np.bincount(t, minlength=C)
    np.testing.assert_allclose(db, 1.5 * (N / C - counts), rtol=1e-12, atol=1e-13)


def test_single_class():
    X, W, b, t = _rand_case(N=5, D=3, C=1, n_ign=0)
    t[:] = 0
    loss, dX, dW, db = O.lce_forward_backward(X, W, b, t, "sum")
    assert loss == 0.0
    for a in (dX, dW, db):
        np.testing.assert_allclose(a, 0.0, atol=1e-15)


def test_invariants():
    X, W, b, t = _rand_case(N=40, D=9, C=17, n_ign=6, seed=11)
    valid = t != -100
    ln, dXn, dWn, dbn = O.lce_forward_backward(X, W, b, t, "none", grad_out=np.ones(40))
    ls, dXs, dWs, dbs = O.lce_forward_backward(X, W, b, t, "sum")
    lm, dXm, dWm, dbm = O.lce_forward_backward(X, W, b, t, "mean")
    # reductions
    assert abs(ls - ln.sum()) < 1e-12
    assert abs(lm - ls / valid.sum()) < 1e-12
    np.testing.assert_allclose(dXs, dXn, rtol=1e-13)
    np.testing.assert_allclose(dXm * valid.sum(), dXs, rtol=1e-12)
    # ignored rows
    assert np.all(ln[~valid] == 0.0) and np.all(dXs[~valid] == 0.0)
    # rows of G sum to zero, hence db and the columns of dW sum to zero
    assert abs(dbs.sum()) < 1e-11
    np.testing.assert_allclose(dWs.sum(0), 0.0, atol=1e-11)
    # a constant added to every bias changes nothing
    l2, dX2, dW2, db2 = O.lce_forward_backward(X, W, b + 3.25, t, "sum")
    assert abs(l2 - ls) < 1e-11
    np.testing.assert_allclose(dX2, dXs, atol=1e-12)
    np.testing.assert_allclose(dW2, dWs, atol=1e-12)
    # permuting rows permutes loss and dX, leaves dW and db
    p = np.random.default_rng(5).permutation(40)
    l3, dX3, dW3, db3 = O.lce_forward_backward(X[p], W, b, t[p], "none", grad_out=np.ones(40))
    np.testing.assert_allclose(l3, ln[p], rtol=1e-13)
    np.testing.assert_allclose(dX3, dXn[p], rtol=1e-13)
    np.testing.assert_allclose(dW3, dWn, atol=1e-12)
    np.testing.assert_allclose(db3, dbn, atol=1e-12)
    # gradients are linear in the upstream gradient
    g = np.random.default_rng(6).standard_normal(40)
    _, dXg, dWg, dbg = O.lce_forward_backward(X, W, b, t, "none", grad_out=g)
    _, dXg2, dWg2, dbg2 = O.lce_forward_backward(X, W, b, t, "none", grad_out=-2 * g)
    np.testing.assert_allclose(dXg2, -2 * dXg, rtol=1e-12)
    np.testing.assert_allclose(dWg2, -2 * dWg, rtol=1e-12, atol=1e-14)
    _, dXs3, _, _ = O.lce_forward_backward(X, W, b, t, "sum", grad_out=3.0)
    np.testing.assert_allclose(dXs3, 3 * dXs, rtol=1e-12)


def test_mean_all_ignored_is_nan():
    # linear_cross_entropy.py, neg_weight_target: d == 0 divides by NaN, so the
    # loss and every gradient are NaN (torch's own cross_entropy returns zero
    # gradients here; the chunked page does not).
    X, W, b, t = _rand_case(N=4, D=3, C=5, n_ign=0)
    t[:] = -100
    loss, dX, dW, db = O.lce_forward_backward(X, W, b, t, "mean")
    assert math.isnan(loss)
    assert np.isnan(dX).all() and np.isnan(dW).all() and np.isnan(db).all()
    loss_f, _ = O.lce_forward(X, W, b, t, "mean")
    assert math.isnan(loss_f)


def test_empty_batch():
    X = np.zeros((0, 3))
    W = RNG.standard_normal((5, 3))
    t = np.zeros(0, dtype=np.int64)
    assert math.isnan(O.lce_forward(X, W, None, t, "mean")[0])
    assert O.lce_forward(X, W, None, t, "sum")[0] == 0.0
    assert O.lce_forward(X, W, None, t, "none")[0].shape == (0,)


def test_out_of_range_target_raises():
    X, W, b, t = _rand_case(N=4, D=3, C=5, n_ign=0)
    t[2] = 5
    with pytest.raises(O.OracleError):
        O.lce_forward(X, W, b, t, "sum")
    t[2] = -1
    with pytest.raises(O.OracleError):
        O.lce_forward(X, W, b, t, "sum")


@pytest.mark.parametrize("reduction,g", [("mean", None), ("sum", 0.5), ("none", "vec")])
def test_ce_from_logits_against_torch(reduction, g):
    r = np.random.default_rng(21)
    N, V = 9, 33
    z = r.standard_normal((N, V)) * 2
    t = r.integers(0, V, N)
    t[3] = -100
    if g == "vec":
        g = r.standard_normal(N)
    loss, grad = O.ce_from_logits(z, t, reduction, -100, g)
    zt = torch.tensor(z, requires_grad=True)
    l = F.cross_entropy(zt, torch.tensor(t), reduction=reduction, ignore_index=-100)
    if reduction == "none":
        l.backward(torch.tensor(g))
    else:
        (l * (1.0 if g is None else g)).backward()
    np.testing.assert_allclose(loss, l.detach().numpy(), rtol=1e-12)
    np.testing.assert_allclose(grad, zt.grad.numpy(), rtol=1e-11, atol=1e-14)
    # uniform logits: ln V and w (1/V - onehot)
    lu, gu = O.ce_from_logits(np.zeros((N, V)), t, "sum")
    assert abs(lu - (N - 1) * math.log(V)) < 1e-11
    assert abs(gu.sum()) < 1e-12


def test_sampled_paths_match_full():
    X, W, b, t = _rand_case(N=300, D=8, C=40, n_ign=20, seed=9)
    cw = RNG.uniform(0.3, 2.0, 40)
    cases = [("mean", 1.7, None), ("none", RNG.standard_normal(300), None), ("mean", 1.7, cw), ("sum", None, cw),
             ("none", RNG.standard_normal(300), cw)]
    for reduction, g, c in cases:
        loss, dX, dW, db = O.lce_forward_backward(X, W, b, t, reduction, grad_out=g, class_weight=c)
        st = O.forward_stats(X, W, b, t, reduction, grad_out=g, want_db=True, row_block=64, class_weight=c)
        np.testing.assert_allclose(st["loss"], loss, rtol=1e-12)
        np.testing.assert_allclose(st["db"], db, rtol=1e-10, atol=1e-13)
        rows = np.array([0, 5, 77, 299])
        _, dXr = O.grad_rows(X, W, b, t, st["lse"], st["w"], rows)
        np.testing.assert_allclose(dXr, dX[rows], rtol=1e-12, atol=1e-14)
        cls = np.array([0, 3, 39])
        dWc, dbc = O.dw_rows(X, W, b, t, st["lse"], st["w"], cls, row_block=50)
        np.testing.assert_allclose(dWc, dW[cls], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(dbc, db[cls], rtol=1e-10, atol=1e-13)
    z = X @ W.T
    w = O.row_weights(t, 40, "mean")
    lr, G = O.ce_rows(z[[1, 2]], t[[1, 2]], w[[1, 2]])
    _, Gfull = O.ce_from_logits(z, t, "mean")
    np.testing.assert_allclose(G, Gfull[[1, 2]], rtol=1e-12, atol=1e-15)


# ---- planted mistakes: each must be caught by the torch cross-check ----

def _mut_drop_bias(X, W, b=None):
    return O._f64(X) @ O._f64(W).T


def _mut_lse_no_shift_back(z):
    m = z.max(axis=1)
    return np.log(np.exp(z - m[:, None]).sum(axis=1))


def _mut_transposed_weight_grad(X, W, b, t, reduction, ignore_index, grad_out):
    loss, dX, dW, db = O.lce_forward_backward(X, W, b, t, reduction, ignore_index, grad_out)
    return loss, dX, dW[::-1].copy(), db


def _mut_mean_over_all_rows(target, num_classes, reduction, ignore_index=-100, grad_out=None, class_weight=None,
                            denominator=None):
    valid = O.valid_mask(target, num_classes, ignore_index).astype(np.float64)
    if reduction == "mean":
        return valid / len(valid)
    return valid * (1.0 if grad_out is None or reduction == "none" else grad_out)


@pytest.mark.parametrize("mutant", ["drop_bias", "lse_shift", "weight_grad_order", "mean_denominator"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    X, W, b, t = _rand_case(seed=2)
    fb = O.lce_forward_backward
    if mutant == "drop_bias":
        monkeypatch.setattr(O, "logits_block", _mut_drop_bias)
    elif mutant == "lse_shift":
        monkeypatch.setattr(O, "log_sum_exp", _mut_lse_no_shift_back)
    elif mutant == "weight_grad_order":
        fb = _mut_transposed_weight_grad
    elif mutant == "mean_denominator":
        monkeypatch.setattr(O, "row_weights", _mut_mean_over_all_rows)
    assert not _matches_torch(fb, X, W, b, t, "mean", -100, None)


@pytest.mark.parametrize("reduction,ignore_index,g", [("mean", -100, None), ("sum", 3, 0.5), ("none", -100, "vec")])
def test_class_weights_against_torch(reduction, ignore_index, g):
    # per-class weights (the page's ``weight``): w_n = weight[t_n]; mean divides by sum of weight[t_n]
    X, W, b, t = _rand_case(N=17, D=6, C=9, ignore_index=ignore_index, seed=41)
    cw = np.random.default_rng(42).uniform(0.2, 2.0, 9)
    if g == "vec":
        g = np.random.default_rng(43).standard_normal(17)
    loss, dX, dW, db = O.lce_forward_backward(X, W, b, t, reduction, ignore_index, g, class_weight=cw)
    Xt = torch.tensor(X, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    l = F.cross_entropy(F.linear(Xt, Wt, bt), torch.tensor(t), weight=torch.tensor(cw), reduction=reduction,
                        ignore_index=ignore_index)
    if reduction == "none":
        l.backward(torch.tensor(g))
    else:
        (l * (1.0 if g is None else g)).backward()
    np.testing.assert_allclose(loss, l.detach().numpy(), rtol=1e-12)
    np.testing.assert_allclose(dX, Xt.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-10, atol=1e-13)
    lf, _ = O.lce_forward(X, W, b, t, reduction, ignore_index, class_weight=cw)
    np.testing.assert_allclose(lf, loss, rtol=1e-13)
    z = X @ W.T + b
    lc, gc = O.ce_from_logits(z, t, reduction, ignore_index, g, class_weight=cw)
    np.testing.assert_allclose(lc, loss, rtol=1e-12)
    np.testing.assert_allclose(gc @ W, dX, rtol=1e-10, atol=1e-13)
    # weight 1 everywhere is the unweighted loss
    l1, dX1, _, _ = O.lce_forward_backward(X, W, b, t, reduction, ignore_index, g, class_weight=np.ones(9))
    l0, dX0, _, _ = O.lce_forward_backward(X, W, b, t, reduction, ignore_index, g)
    np.testing.assert_allclose(l1, l0, rtol=1e-13)
    np.testing.assert_allclose(dX1, dX0, rtol=1e-13)


def test_class_weights_zero_sum_is_nan():
    X, W, b, t = _rand_case(N=5, D=3, C=4, n_ign=0, seed=44)
    cw = np.zeros(4)
    loss, dX, _, _ = O.lce_forward_backward(X, W, b, t, "mean", class_weight=cw)
    assert math.isnan(loss) and np.isnan(dX).all()


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_masked_classes_equal_deleted_classes(reduction):
    """A bias of -inf on a set of classes gives those classes probability 0:
    loss and dX equal those of the problem with the classes deleted (with
    targets renumbered), and the masked classes' dW rows and db entries are
    0. The same holds for cross entropy on logits masked column-wise."""
    X, W, b, t = _rand_case(N=17, D=6, C=19, n_ign=3, seed=31)
    masked = np.zeros(19, dtype=bool)
    masked[[2, 5, 6, 13]] = True
    t[t >= 0] = np.flatnonzero(~masked)[t[t >= 0] % (~masked).sum()]
    g = np.random.default_rng(5).standard_normal(17) if reduction == "none" else 0.5
    bm = b.copy()
    bm[masked] = -np.inf
    loss, dX, dW, db = O.lce_forward_backward(X, W, bm, t, reduction, -100, g)
    keep = np.flatnonzero(~masked)
    renum = np.full(19, -1)
    renum[keep] = np.arange(keep.size)
    tr = np.where(t >= 0, renum[np.maximum(t, 0)], -100)
    rl, rX, rW, rb = O.lce_forward_backward(X, W[keep], b[keep], tr, reduction, -100, g)
    np.testing.assert_allclose(loss, rl, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dX, rX, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(dW[keep], rW, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(db[keep], rb, rtol=1e-11, atol=1e-14)
    assert (dW[masked] == 0).all() and (db[masked] == 0).all()
    z = X @ W.T + bm
    lz, gz = O.ce_from_logits(z, t, reduction, -100, g)
    lr, gr = O.ce_from_logits(z[:, keep], tr, reduction, -100, g)
    np.testing.assert_allclose(lz, lr, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(gz[:, keep], gr, rtol=1e-11, atol=1e-14)
    assert (gz[:, masked] == 0).all()


@pytest.mark.parametrize("class_weights", [False, True])
@pytest.mark.parametrize("g", [None, 1.75])
def test_given_denominator_shards_add_up_to_the_batch(class_weights, g):
    """Data-parallel shards of one batch, each dividing by the WHOLE batch's
    mean denominator: their losses, dW and db sum to the whole batch's and
    their dX rows are the whole batch's rows (an empty shard and a shard of
    ignored rows included)."""
    X, W, b, t = _rand_case(N=23, D=6, C=9, n_ign=4, seed=77)
    t[17:20] = -100  # the third shard below holds only ignored rows
    cw = np.random.default_rng(5).uniform(0.2, 2.0, 9) if class_weights else None
    whole = O.lce_forward_backward(X, W, b, t, "mean", -100, g, class_weight=cw)
    valid = t != -100
    d = float(valid.sum()) if cw is None else float(cw[t[valid]].sum())
    cuts = [0, 9, 9, 17, 20, 23]  # shards [0,9), [9,9) (empty), [9,17), [17,20), [20,23)
    loss = 0.0
    dX = np.zeros_like(X)
    dW = np.zeros_like(W)
    db = np.zeros_like(b)
    for a, e in zip(cuts[:-1], cuts[1:]):
        sl, sX, sW, sb = O.lce_forward_backward(X[a:e], W, b, t[a:e], "mean", -100, g, class_weight=cw,
                                                denominator=d)
        if e > a:
            loss += sl
        dX[a:e] = sX
        dW += sW
        db += sb
    assert math.isclose(loss, whole[0], rel_tol=1e-12)
    for got, ref in ((dX, whole[1]), (dW, whole[2]), (db, whole[3])):
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_given_denominator_against_torch():
    """A shard's mean with denominator d is torch's weighted sum of the shard's
    row losses divided by d, gradients included (torch float64 autograd)."""
    X, W, b, t = _rand_case(N=10, D=5, C=7, n_ign=2, seed=79)
    cw = np.random.default_rng(6).uniform(0.5, 1.5, 7)
    d = 37.5
    loss, dX, dW, db = O.lce_forward_backward(X, W, b, t, "mean", -100, 0.5, class_weight=cw, denominator=d)
    Xt = torch.tensor(X, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    ref = F.cross_entropy(F.linear(Xt, Wt, bt), torch.tensor(t), weight=torch.tensor(cw), reduction="sum",
                          ignore_index=-100) / d
    (ref * 0.5).backward()
    assert math.isclose(loss, ref.item(), rel_tol=1e-12)
    for got, r in ((dX, Xt.grad), (dW, Wt.grad), (db, bt.grad)):
        assert np.allclose(got, r.numpy(), rtol=1e-10, atol=1e-14)
    # the same through cross entropy on given logits
    z = O.logits_block(X, W, b)
    l2, gz = O.ce_from_logits(z, t, "mean", -100, class_weight=cw, denominator=d)
    zt = torch.tensor(z, requires_grad=True)
    r2 = F.cross_entropy(zt, torch.tensor(t), weight=torch.tensor(cw), reduction="sum", ignore_index=-100) / d
    r2.backward()
    assert math.isclose(l2, r2.item(), rel_tol=1e-12)
    assert np.allclose(gz, zt.grad.numpy(), rtol=1e-10, atol=1e-14)
    # a zero denominator gives NaN, as the page's d == 0 does
    l0, gX0, _, _ = O.lce_forward_backward(X, W, b, t, "mean", -100, denominator=0.0)
    assert math.isnan(l0) and np.isnan(gX0).all()
