"""The autograd wrapper over the C ABI: loss and .grad of input, weight and
bias against the float64 oracle, with leading dimensions, an upstream
gradient, reduction none and retain_graph."""

import numpy as np
import pytest
import torch

from linear_cross_entropy_lce_gb300.autograd import linear_cross_entropy
from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_autograd_matches_oracle(cuda_lib, dtype, reduction):
    inp = make_linear_inputs(6 * 50, 64, 700, dtype, "cuda", seed=31, bias=True, w_std=0.3, b_std=0.2,
                             n_ignored=9)
    X = inp["X"].reshape(6, 50, 64).requires_grad_(True)  # leading dims are flattened
    W = inp["W"].clone().requires_grad_(True)
    b = inp["b"].clone().requires_grad_(True)
    t = inp["target"].reshape(6, 50)
    loss = linear_cross_entropy(X, W, t, b, reduction)
    if reduction == "none":
        assert loss.shape == (6, 50)
        g = torch.randn(6, 50, device="cuda")
        loss.backward(g)
        gn = to64(g).reshape(-1)
    else:
        (loss * 1.5).backward()
        gn = 1.5
    rl, rX, rW, rb = O.lce_forward_backward(to64(X.detach()).reshape(-1, 64), to64(W.detach()),
                                            to64(b.detach()), t.reshape(-1).cpu().numpy(), reduction, -100, gn)
    tol = TOL[dtype]
    if reduction == "none":
        assert rel_max(to64(loss.detach()).reshape(-1), rl) < tol["loss"]
    else:
        assert rel_scalar(loss.item(), rl) < tol["loss"]
    assert X.grad.shape == X.shape and X.grad.dtype == dtype
    assert rel_max(to64(X.grad).reshape(-1, 64), rX) < tol["grad"]
    assert rel_max(to64(W.grad), rW) < tol["grad"]
    assert rel_max(to64(b.grad), rb) < tol["grad"]


def test_autograd_retain_graph_and_partial_grads(cuda_lib):
    inp = make_linear_inputs(128, 32, 300, torch.bfloat16, "cuda", seed=32, w_std=0.4)
    X = inp["X"].requires_grad_(True)
    W = inp["W"]  # no gradient wanted for the weight
    # allow_retain_graph keeps the precomputed gradients: two backwards with
    # an upstream gradient of 2 give the same (scaled once) gradient
    loss = linear_cross_entropy(X, W, inp["target"], reduction="mean", allow_retain_graph=True)
    (loss * 2.0).backward(retain_graph=True)
    g1 = X.grad.clone()
    X.grad = None
    (loss * 2.0).backward()
    assert torch.equal(g1, X.grad)
    assert W.grad is None
    X.grad = None
    ref = linear_cross_entropy(X, W, inp["target"], reduction="mean")
    ref.backward()
    assert rel_max(to64(g1), 2.0 * to64(X.grad)) < 1e-2
    # without it the buffers are handed out and scaled in place: a second
    # backward through the same loss raises, as the page's option says
    loss = linear_cross_entropy(X, W, inp["target"], reduction="mean")
    (loss * 3.0).backward(retain_graph=True)
    with pytest.raises(RuntimeError):
        loss.backward()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_scale_gradients_in_place(cuda_lib, dtype):
    """lce_scale_gradients: buffers times a device scalar, untouched when it
    is 1; ragged lengths and an unaligned start take the scalar tail path."""
    g = torch.Generator(device="cuda").manual_seed(5)
    dX = torch.randn(1001, generator=g, device="cuda").to(dtype)
    dW = torch.randn(37, 129, generator=g, device="cuda").to(dtype)
    base = torch.randn(301, generator=g, device="cuda").to(dtype)
    db = base[1:]  # 2 or 4 bytes past a 16-byte boundary
    first = base[0].clone()
    keep = [x.clone() for x in (dX, dW, db)]
    cuda_lib.lce_scale_gradients(dX, dW, db, torch.ones((), device="cuda"))
    torch.cuda.synchronize()
    for a, k in zip((dX, dW, db), keep):
        assert torch.equal(a, k)
    cuda_lib.lce_scale_gradients(dX, None, db, torch.tensor(-0.75, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(dW, keep[1])
    for a, k in ((dX, keep[0]), (db, keep[2])):
        assert torch.equal(a, (k.float() * -0.75).to(dtype))
    assert torch.equal(base[0], first)  # the element before db is untouched


@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_autograd_plan_options(cuda_lib, reduction):
    """chunk_rows (the page's aspect_ratio chunk size: batch chunks) and
    buffer_bytes (classes recomputed beyond a small buffer) give the same
    gradients as the default plan, within the bf16 tolerance of the oracle."""
    N, D, C = 1500, 64, 3000
    inp = make_linear_inputs(N, D, C, torch.bfloat16, "cuda", seed=37, bias=True, w_std=0.4, b_std=0.2,
                             n_ignored=40)
    rows = cuda_lib.lce_aspect_ratio_chunk_rows(N, D, C)
    g = torch.randn(N, device="cuda") if reduction == "none" else None
    ref = O.lce_forward_backward(to64(inp["X"]), to64(inp["W"]), to64(inp["b"]), inp["target"].cpu().numpy(),
                                 reduction, -100, None if g is None else to64(g))
    for plan in ({"chunk_rows": rows}, {"buffer_bytes": N * 512 * 2}):
        X = inp["X"].clone().requires_grad_(True)
        W = inp["W"].clone().requires_grad_(True)
        b = inp["b"].clone().requires_grad_(True)
        loss = linear_cross_entropy(X, W, inp["target"], b, reduction, **plan)
        if reduction == "none":
            loss.backward(g)
        else:
            loss.backward()
        tol = TOL[torch.bfloat16]
        assert rel_max(to64(X.grad), ref[1]) < tol["grad"], plan
        assert rel_max(to64(W.grad), ref[2]) < tol["grad"], plan
        assert rel_max(to64(b.grad), ref[3]) < tol["grad"], plan
