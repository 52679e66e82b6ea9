"""Fused linear + cross-entropy on the GPU against the float64 oracle, at
sizes the oracle finishes in seconds: the tiny and mid workloads, ragged
shapes that span several tiles with tails, several batch chunks, every
reduction, and the degenerate cases."""

import math

import numpy as np
import pytest
import torch

import linear_cross_entropy_lce_gb300 as lce_mod
from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs, make_workload
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu


def _grad_arg(reduction, N, seed=0):
    if reduction == "none":
        g = torch.Generator(device="cuda").manual_seed(seed)
        return torch.randn(N, generator=g, device="cuda")
    if reduction == "sum":
        return torch.tensor(1.25, device="cuda")
    return None


def _poison(t):
    if t is not None:
        t.fill_(float("nan"))


def _check(cuda_lib, inp, reduction, ignore_index=-100, grad_dtype=None, chunk_rows=0, workspace=None,
           grad_tol=None):
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    dtype = X.dtype
    g = inp.get("grad_out")
    if g is None:
        g = _grad_arg(reduction, X.shape[0])
    loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, reduction, ignore_index, g,
                                                     grad_dtype=grad_dtype, chunk_rows=chunk_rows,
                                                     workspace=workspace)
    torch.cuda.synchronize()
    gn = None if g is None else to64(g)
    rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), reduction, ignore_index,
                                            gn)
    tol = TOL[dtype]
    # bf16 anywhere (inputs, hence the bf16 G operand, or bf16 gradient
    # storage) puts the gradients under the bf16 tolerance
    any_bf16 = torch.bfloat16 in (dtype, grad_dtype)
    gt = grad_tol if grad_tol is not None else TOL[torch.bfloat16 if any_bf16 else dtype]["grad"]
    if reduction == "none":
        assert rel_max(to64(loss), rl) < tol["loss"], "loss"
    else:
        assert rel_scalar(loss.item(), rl) < tol["loss"], ("loss", loss.item(), rl)
    assert rel_max(to64(dX), rX) < gt, "dX"
    assert rel_max(to64(dW), rW) < gt, "dW"
    if b is not None:
        assert rel_max(to64(db), rb) < gt, "db"
    # forward-only entry point gives the same loss and the row lse
    lf, lse = cuda_lib.lce_forward(X, W, b, t, reduction, ignore_index, want_lse=True)
    torch.cuda.synchronize()
    rlf, rlse = O.lce_forward(to64(X), to64(W), to64(b), t.cpu().numpy(), reduction, ignore_index)
    assert rel_max(to64(lse), rlse) < tol["loss"]
    if reduction == "none":
        assert rel_max(to64(lf), rlf) < tol["loss"]
    else:
        assert rel_scalar(lf.item(), rlf) < tol["loss"]


def test_tiny_fp32_workload(cuda_lib):
    _check(cuda_lib, make_workload("tiny_fp32", "cuda"), "mean")


def test_fp32_mid_workload(cuda_lib):
    _check(cuda_lib, make_workload("fp32_mid", "cuda"), "sum")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("bias", [True, False])
def test_ragged_shapes(cuda_lib, dtype, reduction, bias):
    # N, C, D not multiples of the 128 x 256 x 64 tiles; several tiles each way
    inp = make_linear_inputs(300, 96, 1000, dtype, "cuda", seed=7, bias=bias, x_std=1.0, w_std=0.3,
                             b_std=0.5, n_ignored=17)
    _check(cuda_lib, inp, reduction)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
def test_several_chunks(cuda_lib, dtype, grad_dtype):
    # chunk_rows=128 over N=333 rows: 3 chunks, dW accumulated across them
    inp = make_linear_inputs(333, 64, 700, dtype, "cuda", seed=3, bias=True, w_std=0.4, b_std=0.2,
                             n_ignored=5)
    _check(cuda_lib, inp, "mean", grad_dtype=grad_dtype, chunk_rows=128)


def test_workspace_decides_chunks(cuda_lib):
    inp = make_linear_inputs(1000, 32, 512, torch.bfloat16, "cuda", seed=4, bias=False, w_std=0.5)
    need_small = lce_mod.lce_workspace_size(lce_mod.LCE_OP_FORWARD_BACKWARD, 1000, 32, 512, lce_mod.LCE_BF16,
                                            lce_mod.LCE_RED_SUM, lce_mod.LCE_BF16, 256)
    ws = torch.empty(need_small, dtype=torch.uint8, device="cuda")
    _check(cuda_lib, inp, "sum", workspace=ws)
    too_small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(lce_mod.LceError):
        cuda_lib.lce_forward_backward(inp["X"], inp["W"], None, inp["target"], "sum", workspace=too_small)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ignore_index_inside_range_and_subset_of_grads(cuda_lib, dtype):
    inp = make_linear_inputs(200, 40 if dtype == torch.float32 else 48, 300, dtype, "cuda", seed=9, bias=True,
                             w_std=0.3, b_std=0.1)
    t = inp["target"]
    t[::7] = 5  # rows with target 5 are ignored, class 5 stays a softmax column
    _check(cuda_lib, inp, "mean", ignore_index=5)
    X, W, b = inp["X"], inp["W"], inp["b"]
    l1, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, "mean", 5, want_dw=False, want_db=False)
    l2, dX2, dW2, db2 = cuda_lib.lce_forward_backward(X, W, b, t, "mean", 5, want_dx=False)
    torch.cuda.synchronize()
    assert dW is None and db is None and dX2 is None
    rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), "mean", 5)
    assert rel_max(to64(dX), rX) < TOL[dtype]["grad"]
    assert rel_max(to64(dW2), rW) < TOL[dtype]["grad"]
    assert rel_max(to64(db2), rb) < TOL[dtype]["grad"]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_degenerate_cases(cuda_lib, dtype):
    D = 16
    # N = 0: mean NaN, sum 0, gradients of W and b zero
    X = torch.empty(0, D, dtype=dtype, device="cuda")
    W = torch.randn(10, D, device="cuda").to(dtype)
    b = torch.randn(10, device="cuda").to(dtype)
    t = torch.empty(0, dtype=torch.int64, device="cuda")
    loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, "mean")
    torch.cuda.synchronize()
    assert math.isnan(loss.item()) and dX.shape == (0, D)
    assert (dW == 0).all() and (db == 0).all()
    assert cuda_lib.lce_forward_backward(X, W, b, t, "sum")[0].item() == 0.0
    # every row ignored under mean: NaN loss and NaN gradients
    inp = make_linear_inputs(20, D, 10, dtype, "cuda", seed=1, bias=True)
    tt = torch.full((20,), -100, dtype=torch.int64, device="cuda")
    loss, dX, dW, db = cuda_lib.lce_forward_backward(inp["X"], inp["W"], inp["b"], tt, "mean")
    torch.cuda.synchronize()
    assert math.isnan(loss.item()) and torch.isnan(dX).all() and torch.isnan(dW).all() and torch.isnan(db).all()
    # ... and under sum: zero loss, zero gradients
    loss, dX, dW, db = cuda_lib.lce_forward_backward(inp["X"], inp["W"], inp["b"], tt, "sum")
    torch.cuda.synchronize()
    assert loss.item() == 0.0 and (dX == 0).all() and (dW == 0).all() and (db == 0).all()
    # one class: loss 0, gradients 0
    inp = make_linear_inputs(50, D, 1, dtype, "cuda", seed=2, bias=True)
    loss, dX, dW, db = cuda_lib.lce_forward_backward(inp["X"], inp["W"], inp["b"],
                                                     torch.zeros(50, dtype=torch.int64, device="cuda"), "sum")
    torch.cuda.synchronize()
    assert abs(loss.item()) < 1e-6 and dX.abs().max().item() < 1e-6 and dW.abs().max().item() < 1e-6


def test_out_of_range_target_sets_status(cuda_lib):
    inp = make_linear_inputs(40, 32, 100, torch.bfloat16, "cuda", seed=5)
    t = inp["target"].clone()
    t[3] = 100
    t[7] = -5
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    loss, dX, dW, db = cuda_lib.lce_forward_backward(inp["X"], inp["W"], None, t, "none", -100,
                                                     torch.ones(40, device="cuda"), workspace=ws)
    assert cuda_lib.lce_read_device_status(ws) == 8
    assert loss[3].item() == 0.0 and loss[7].item() == 0.0
    assert (dX[3] == 0).all() and (dX[7] == 0).all()
    tn = t.cpu().numpy().copy()
    tn[[3, 7]] = -100  # the library treats those rows as ignored
    rl, rX, rW, _ = O.lce_forward_backward(to64(inp["X"]), to64(inp["W"]), None, tn, "none", -100, np.ones(40))
    assert rel_max(to64(dX), rX) < 2e-2 and rel_max(to64(dW), rW) < 2e-2


def test_outputs_fully_written(cuda_lib):
    """Poisoned (NaN) output buffers: every element must be overwritten."""
    inp = make_linear_inputs(260, 64, 520, torch.bfloat16, "cuda", seed=8, bias=True, w_std=0.2, b_std=0.1)
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    lib = lce_mod.load_library()
    import ctypes
    N, D = X.shape
    C = W.shape[0]
    dX = torch.full((N, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    dW = torch.full((C, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    db = torch.full((C,), float("nan"), dtype=torch.bfloat16, device="cuda")
    loss = torch.full((1,), float("nan"), device="cuda")
    nb = lib.lce_workspace_size(1, N, D, C, 1, 2, 1, 0)
    ws = torch.full((nb,), 255, dtype=torch.uint8, device="cuda")
    p = lambda x: ctypes.c_void_p(x.data_ptr())
    st = lib.lce_forward_backward(p(X), p(W), p(b), p(t), N, D, C, 1, 0, 2, -100, None, p(loss), p(dX), p(dW),
                                  p(db), 1, p(ws), nb, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.isfinite(dX).all() and torch.isfinite(dW).all() and torch.isfinite(db).all()
    assert math.isfinite(loss.item())


@pytest.mark.parametrize("N,chunk_rows,reduction", [(1500, 0, "mean"), (2500, 1024, "sum"), (1100, 0, "none")])
def test_row_slabs(cuda_lib, N, chunk_rows, reduction):
    # bf16 backward over >= 1024 rows: the chunk is cut into row slabs and the
    # logits GEMM of slab k forms G of slab k-1 (with the bias gradient)
    inp = make_linear_inputs(N, 128, 2000, torch.bfloat16, "cuda", seed=N, bias=True, w_std=0.1, b_std=0.2,
                             n_ignored=N // 20)
    _check(cuda_lib, inp, reduction, chunk_rows=chunk_rows)


@pytest.mark.parametrize("want", [(True, False, False), (False, True, True), (True, True, False), (False, False, True)])
def test_row_slabs_grad_subsets(cuda_lib, want):
    # the last slab's G is formed inside the dX GEMM when dX is wanted, by
    # its own kernel otherwise; either way dW and db see all of G
    want_dx, want_dw, want_db = want
    N, D, C = 2100, 64, 3000
    inp = make_linear_inputs(N, D, C, torch.bfloat16, "cuda", seed=77, bias=True, w_std=0.1, b_std=0.2,
                             n_ignored=40)
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, "mean", want_dx=want_dx, want_dw=want_dw,
                                                     want_db=want_db)
    torch.cuda.synchronize()
    rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), "mean")
    tol = TOL[torch.bfloat16]
    assert rel_scalar(loss.item(), rl) < tol["loss"]
    for on, got, ref in ((want_dx, dX, rX), (want_dw, dW, rW), (want_db, db, rb)):
        if on:
            assert rel_max(to64(got), ref) < tol["grad"]
        else:
            assert got is None


@pytest.mark.parametrize("dtype,N", [(torch.bfloat16, 1500), (torch.float32, 700), (torch.float16, 1300)])
def test_classes_masked_by_bias(cuda_lib, dtype, N):
    """A bias of -inf masks classes: two whole 256-column segments and every
    seventh class. Masked classes get probability 0, so their dW rows and db
    entries are 0 and everything else matches the oracle (no NaN from a
    segment whose logits are all -inf). bf16 at 1500 rows runs the row slabs."""
    D, C = 64, 3000
    inp = make_linear_inputs(N, D, C, dtype, "cuda", seed=N + 5, bias=True, w_std=0.1, b_std=0.2,
                             n_ignored=N // 25)
    b = inp["b"]
    masked = torch.zeros(C, dtype=torch.bool, device="cuda")
    masked[256:768] = True
    masked[3::7] = True
    b[masked] = -math.inf
    t = inp["target"]
    valid = t != -100
    free = torch.nonzero(~masked).flatten()
    t[valid] = free[t[valid] % free.numel()]
    for reduction in ("mean", "none"):
        _check(cuda_lib, inp, reduction)
    loss, dX, dW, db = cuda_lib.lce_forward_backward(inp["X"], inp["W"], b, t, "mean")
    torch.cuda.synchronize()
    assert torch.isfinite(loss) and torch.isfinite(dX).all() and torch.isfinite(dW).all()
    assert (dW[masked] == 0).all() and (db[masked] == 0).all()
