"""The data-parallel combination logic (linear_cross_entropy_lce_gb300.dp) on
gloo ranks on the CPU: each rank holds a row shard, the float64 oracle
stands in for the per-rank library call, and the combined loss and
gradients must equal the oracle on the whole batch. Uneven shards, a rank
with no rows, class weights and every reduction."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import lce_oracle as O


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleCompute:
    """The per-rank arithmetic of LibraryCompute, done by the oracle."""

    def denominator(self, target, C, ignore_index, class_weight):
        t = target.numpy()
        cw = None if class_weight is None else class_weight.numpy()
        c = O.class_weight_of_rows(t, O.valid_mask(t, C, ignore_index), cw)
        return torch.tensor([c.sum()], dtype=torch.float32)

    def forward_backward(self, X, W, b, target, reduction, ignore_index, grad_out, class_weight, denominator,
                         want_dx, want_dw, want_db):
        g = grad_out
        if isinstance(g, torch.Tensor):
            g = g.numpy()
        loss, dX, dW, db = O.lce_forward_backward(
            X.numpy(), W.numpy(), None if b is None else b.numpy(), target.numpy(), reduction, ignore_index, g,
            class_weight=None if class_weight is None else class_weight.numpy(),
            denominator=None if denominator is None else float(denominator[0]))
        t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a))
        return torch.tensor(loss) if reduction != "none" else t(loss), t(dX), t(dW), t(db) if want_db else None


def _problem(N, reduction, class_weights):
    r = np.random.default_rng(11)
    D, C = 6, 13
    X = r.standard_normal((N, D))
    W = r.standard_normal((C, D)) * 0.6
    b = r.standard_normal(C) * 0.2
    t = r.integers(0, C, N)
    t[r.permutation(N)[:3]] = -100
    cw = r.uniform(0.3, 2.0, C) if class_weights else None
    g = r.standard_normal(N) if reduction == "none" else (0.8 if reduction == "sum" else None)
    return X, W, b, t, cw, g


def _worker(rank, world, port, cuts, reduction, class_weights, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from linear_cross_entropy_lce_gb300.dp import sharded_forward_backward

    N = cuts[-1]
    X, W, b, t, cw, g = _problem(N, reduction, class_weights)
    lo, hi = cuts[rank], cuts[rank + 1]
    gl = g[lo:hi] if reduction == "none" else g
    T = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a))
    loss, dX, dW, db = sharded_forward_backward(T(X[lo:hi]), T(W), T(b), T(t[lo:hi]), reduction, -100,
                                                T(gl) if reduction == "none" else gl, T(cw),
                                                compute=OracleCompute())
    out[rank] = (np.asarray(loss.numpy()), dX.numpy(), dW.numpy(), db.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("cuts,reduction,class_weights", [
    ([0, 17, 40], "mean", False),
    ([0, 17, 40], "mean", True),
    ([0, 0, 25, 40], "mean", True),   # rank 0 holds no rows
    ([0, 30, 40], "sum", False),
    ([0, 9, 21, 40], "none", True),
])
def test_shards_combine_to_the_whole_batch(cuts, reduction, class_weights):
    world = len(cuts) - 1
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, cuts, reduction, class_weights, out), nprocs=world, join=True)
    N = cuts[-1]
    X, W, b, t, cw, g = _problem(N, reduction, class_weights)
    rl, rX, rW, rb = O.lce_forward_backward(X, W, b, t, reduction, -100, g, class_weight=cw)
    # the denominator travels as an fp32 scalar (as it does to the library):
    # a class-weight sum rounds there by up to 2^-24 relative
    tol = dict(rtol=1e-6, atol=1e-12)
    dX = np.concatenate([out[r][1] for r in range(world)])
    assert np.allclose(dX, rX, **tol)
    for r in range(world):
        loss, _, dW, db = out[r]
        if reduction == "none":
            assert np.allclose(loss, rl[cuts[r]:cuts[r + 1]], **tol)
        else:
            assert abs(float(loss) - rl) <= 1e-6 * abs(rl)  # the loss is reduced in fp32
        assert np.allclose(dW, rW, **tol)
        assert np.allclose(db, rb, **tol)


def test_shard_rows_split():
    from linear_cross_entropy_lce_gb300.dp import shard_rows

    for n in (0, 1, 7, 8192, 8193):
        for world in (1, 2, 3, 8):
            parts = [shard_rows(n, world, r) for r in range(world)]
            assert parts[0].start == 0 and parts[-1].stop == n
            assert all(a.stop == b.start for a, b in zip(parts, parts[1:]))
            sizes = [p.stop - p.start for p in parts]
            assert max(sizes) - min(sizes) <= 1
