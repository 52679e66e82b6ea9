"""Per-class CE weights through the _ex entry points (and the binding's
class_weight argument), against the float64 oracle."""

import math

import numpy as np
import pytest
import torch

from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs, make_logits_inputs
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu


def _cw(C, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.rand(C, generator=g, device="cuda") * 1.8 + 0.2


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("N", [300, 1500])
def test_weighted_lce(cuda_lib, dtype, reduction, N):
    inp = make_linear_inputs(N, 64, 1000, dtype, "cuda", seed=N + 7, bias=True, w_std=0.3, b_std=0.2,
                             n_ignored=N // 15)
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    cw = _cw(1000, N)
    g = torch.randn(N, device="cuda") if reduction == "none" else (torch.tensor(0.5, device="cuda")
                                                                    if reduction == "sum" else None)
    loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, reduction, -100, g, class_weight=cw)
    lf = cuda_lib.lce_forward(X, W, b, t, reduction, -100, class_weight=cw)
    torch.cuda.synchronize()
    rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), reduction, -100,
                                            None if g is None else to64(g), class_weight=to64(cw))
    tol = TOL[dtype]
    if reduction == "none":
        assert rel_max(to64(loss), rl) < tol["loss"] and rel_max(to64(lf), rl) < tol["loss"]
    else:
        assert rel_scalar(loss.item(), rl) < tol["loss"] and rel_scalar(lf.item(), rl) < tol["loss"]
    for got, ref in ((dX, rX), (dW, rW), (db, rb)):
        assert rel_max(to64(got), ref) < tol["grad"]


@pytest.mark.parametrize("dtype,V", [(torch.float32, 40000), (torch.bfloat16, 777)])
def test_weighted_ce_from_logits(cuda_lib, dtype, V):
    inp = make_logits_inputs(40, V, dtype, "cuda", seed=V, std=2.0, n_ignored=3)
    logits, t = inp["logits"], inp["target"]
    cw = _cw(V, 5)
    snap = to64(logits)
    loss = cuda_lib.lce_cross_entropy_from_logits(logits, t, "mean", -100, class_weight=cw)
    torch.cuda.synchronize()
    rl, rg = O.ce_from_logits(snap, t.cpu().numpy(), "mean", -100, class_weight=to64(cw))
    assert rel_scalar(loss.item(), rl) < TOL[dtype]["loss"]
    assert rel_max(to64(logits), rg) < TOL[dtype]["grad"]


def test_weighted_mean_zero_weight_sum_is_nan(cuda_lib):
    inp = make_linear_inputs(50, 32, 100, torch.bfloat16, "cuda", seed=3)
    cw = torch.zeros(100, device="cuda")
    loss, dX, dW, _ = cuda_lib.lce_forward_backward(inp["X"], inp["W"], None, inp["target"], "mean",
                                                    class_weight=cw)
    torch.cuda.synchronize()
    assert math.isnan(loss.item()) and torch.isnan(dX).all() and torch.isnan(dW).all()
