"""Data-parallel row shards through the library: two gloo ranks on the one
GPU each run their rows through liblce.so with the whole batch's mean
denominator (lce_mean_denominator, all-reduced), the ranks all-reduce host
copies of dW, db and the loss, and the result must match the float64 oracle
on the whole batch element by element. The ranks' kernels never wait on one
another: each launch depends only on its own rank's data."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(case):
    from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs

    N, D, C, dtype, reduction, bias, cw = case
    inp = make_linear_inputs(N, D, C, dtype, "cuda", seed=N + C, bias=bias, w_std=0.5, b_std=0.3,
                             n_ignored=N // 11)
    g = None
    gen = torch.Generator(device="cuda").manual_seed(5)
    if reduction == "none":
        g = torch.randn(N, generator=gen, device="cuda")
    elif reduction == "sum":
        g = torch.tensor(1.5, device="cuda")
    cwt = torch.rand(C, generator=gen, device="cuda") + 0.5 if cw else None
    return inp["X"], inp["W"], inp["b"], inp["target"], g, cwt


def _worker(rank, world, port, case, cuts, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from linear_cross_entropy_lce_gb300.dp import sharded_forward_backward

    X, W, b, t, g, cw = _inputs(case)
    reduction = case[4]
    lo, hi = cuts[rank], cuts[rank + 1]
    gl = g[lo:hi].contiguous() if reduction == "none" else g
    loss, dX, dW, db = sharded_forward_backward(X[lo:hi].contiguous(), W, b, t[lo:hi].contiguous(), reduction,
                                                -100, gl, cw)
    torch.cuda.synchronize()
    out[rank] = (to64(loss), to64(dX), to64(dW), to64(db))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(600)
@pytest.mark.parametrize("case,cuts", [
    ((1500, 64, 2000, torch.bfloat16, "mean", True, True), [0, 700, 1500]),
    ((1500, 64, 2000, torch.bfloat16, "mean", False, False), [0, 0, 1500]),  # rank 0 holds no rows
    ((900, 136, 3001, torch.bfloat16, "sum", True, False), [0, 451, 900]),
    ((600, 72, 1800, torch.float16, "none", True, True), [0, 333, 600]),
])
def test_two_shards_match_the_whole_batch(cuda_lib, case, cuts):
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, case, cuts, out), nprocs=world, join=True)
    X, W, b, t, g, cw = _inputs(case)
    reduction = case[4]
    rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), reduction, -100,
                                            None if g is None else to64(g),
                                            class_weight=None if cw is None else to64(cw))
    tol = TOL[case[3]]
    dX = np.concatenate([out[r][1] for r in range(world)])
    assert rel_max(dX, rX) < tol["grad"]
    for r in range(world):
        loss, _, dW, db = out[r]
        if reduction == "none":
            assert rel_max(loss, rl[cuts[r]:cuts[r + 1]]) < tol["loss"]
        else:
            assert rel_scalar(float(loss), rl) < tol["loss"]
        assert rel_max(dW, rW) < tol["grad"]
        if b is not None:
            assert rel_max(db, rb) < tol["grad"]
