"""fp16 inputs on the tensor-core path (the backward keeps the row weights
out of the 16-bit gradient tile) against the float64 oracle."""

import math

import numpy as np
import pytest
import torch

from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs, make_logits_inputs
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu
F16 = torch.float16


def _run(cuda_lib, inp, reduction, grad_dtype=None, chunk_rows=0, class_weight=None, ignore_index=-100):
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    N = X.shape[0]
    g = None
    if reduction == "none":
        g = torch.randn(N, generator=torch.Generator(device="cuda").manual_seed(5), device="cuda")
    elif reduction == "sum":
        g = torch.tensor(0.8, device="cuda")
    loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, reduction, ignore_index, g, grad_dtype=grad_dtype,
                                                     chunk_rows=chunk_rows, class_weight=class_weight)
    torch.cuda.synchronize()
    rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), reduction, ignore_index,
                                            None if g is None else to64(g),
                                            class_weight=None if class_weight is None else to64(class_weight))
    tol = TOL[F16]
    gtol = TOL[torch.bfloat16]["grad"] if grad_dtype == torch.bfloat16 else tol["grad"]
    if reduction == "none":
        assert rel_max(to64(loss), rl) < tol["loss"]
    else:
        assert rel_scalar(loss.item(), rl) < tol["loss"], (loss.item(), rl)
    assert rel_max(to64(dX), rX) < gtol, "dX"
    assert rel_max(to64(dW), rW) < gtol, "dW"
    if b is not None:
        assert rel_max(to64(db), rb) < gtol, "db"
    return loss, dX, dW, db


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("bias", [True, False])
def test_fp16_ragged(cuda_lib, reduction, bias):
    inp = make_linear_inputs(300, 96, 1000, F16, "cuda", seed=17, bias=bias, w_std=0.3, b_std=0.3, n_ignored=13)
    _run(cuda_lib, inp, reduction)
    lf = cuda_lib.lce_forward(inp["X"], inp["W"], inp["b"], inp["target"], reduction)
    rl, _ = O.lce_forward(to64(inp["X"]), to64(inp["W"]), to64(inp["b"]), inp["target"].cpu().numpy(), reduction)
    if reduction == "none":
        assert rel_max(to64(lf), rl) < TOL[F16]["loss"]
    else:
        assert rel_scalar(lf.item(), rl) < TOL[F16]["loss"]


@pytest.mark.parametrize("grad_dtype", [torch.float16, torch.float32, torch.bfloat16])
def test_fp16_grad_dtypes_and_chunks(cuda_lib, grad_dtype):
    inp = make_linear_inputs(333, 64, 700, F16, "cuda", seed=18, bias=True, w_std=0.4, b_std=0.2, n_ignored=5)
    _run(cuda_lib, inp, "mean", grad_dtype=grad_dtype, chunk_rows=128)


@pytest.mark.parametrize("N,reduction", [(1500, "mean"), (1100, "none")])
def test_fp16_row_slabs_and_large_batch_weight(cuda_lib, N, reduction):
    # mean over 1500 rows: w = 1/1500 per row is applied in fp32, not stored in the fp16 G tile
    inp = make_linear_inputs(N, 128, 2000, F16, "cuda", seed=N + 1, bias=True, w_std=0.1, b_std=0.2,
                             n_ignored=N // 20)
    _run(cuda_lib, inp, reduction)


def test_fp16_class_weights_and_nan(cuda_lib):
    inp = make_linear_inputs(200, 48, 300, F16, "cuda", seed=19, bias=True, w_std=0.3, b_std=0.1, n_ignored=9)
    cw = torch.rand(300, device="cuda") + 0.25
    _run(cuda_lib, inp, "mean", class_weight=cw)
    t = torch.full((200,), -100, dtype=torch.int64, device="cuda")
    loss, dX, dW, db = cuda_lib.lce_forward_backward(inp["X"], inp["W"], inp["b"], t, "mean")
    torch.cuda.synchronize()
    assert math.isnan(loss.item()) and torch.isnan(dX).all() and torch.isnan(dW).all() and torch.isnan(db).all()


@pytest.mark.parametrize("V", [50000, 777])
def test_fp16_ce_from_logits(cuda_lib, V):
    inp = make_logits_inputs(33, V, F16, "cuda", seed=V, std=2.0, n_ignored=3)
    logits, t = inp["logits"], inp["target"]
    snap = to64(logits)
    loss = cuda_lib.lce_cross_entropy_from_logits(logits, t, "sum", -100, torch.tensor(0.5, device="cuda"))
    torch.cuda.synchronize()
    rl, rg = O.ce_from_logits(snap, t.cpu().numpy(), "sum", -100, 0.5)
    assert rel_scalar(loss.item(), rl) < TOL[F16]["loss"]
    assert rel_max(to64(logits), rg) < TOL[F16]["grad"]
