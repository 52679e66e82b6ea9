"""The bounded-memory backward on the GPU against the float64 oracle.

When the [rows, classes] gradient buffer may not hold every class, the
forward sweep stores the softmax of the first Cb classes only and the rest
are recomputed chunk by chunk (their logits a second time, formed straight
into gradient tiles), dX summed over the chunks in fp32 and each chunk's dW
rows written whole. lce_backward does the same for every class from a given
row lse. These tests force small buffers on small problems so that several
recomputed chunks, ragged last chunks, row slabs and batch chunks all occur,
and compare every output element by element with the oracle."""

import ctypes

import numpy as np
import pytest
import torch

import linear_cross_entropy_lce_gb300 as lce_mod
from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu


def _plan(op, N, D, C, dt, gdt, ws):
    """The plan a call makes for ws bytes (lce_test_plan through the binding)."""
    return lce_mod.plan_of(op, N, D, C, dt, gdt, ws)


def _tol(dtype, grad_dtype):
    g = TOL[dtype]["grad"]
    if grad_dtype in (torch.bfloat16, torch.float16):
        g = max(g, TOL[grad_dtype]["grad"])
    return TOL[dtype]["loss"], g


def _grad_out(reduction, N, seed):
    if reduction == "none":
        return torch.randn(N, generator=torch.Generator(device="cuda").manual_seed(seed), device="cuda")
    if reduction == "sum":
        return torch.tensor(0.75, device="cuda")
    return None


def _oracle(X, W, b, t, reduction, g, ignore_index=-100, cw=None):
    return O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), reduction, ignore_index,
                                  None if g is None else to64(g), class_weight=None if cw is None else to64(cw))


def _compare(loss, dX, dW, db, ref, reduction, tl, tg):
    rl, rX, rW, rb = ref
    if loss is not None:
        if reduction == "none":
            assert rel_max(to64(loss), rl) < tl, "loss"
        else:
            assert rel_scalar(loss.item(), rl) < tl, ("loss", loss.item(), rl)
    assert rel_max(to64(dX), rX) < tg, "dX"
    assert rel_max(to64(dW), rW) < tg, "dW"
    if db is not None:
        assert rel_max(to64(db), rb) < tg, "db"


CASES = [
    # N, D, C, dtype, reduction, bias, class weights, grad dtype, buffer classes
    (700, 136, 3001, torch.bfloat16, "mean", True, False, None, 1024),
    (1500, 64, 2000, torch.bfloat16, "sum", False, True, torch.float32, 512),   # row slabs + recomputation
    (300, 200, 5000, torch.float16, "none", True, False, None, 1024),
    (1025, 64, 777, torch.bfloat16, "mean", True, False, torch.bfloat16, 256),  # ragged last chunk of 9 classes
    (2100, 48, 1300, torch.float16, "mean", False, True, torch.float32, 256),
    (96, 520, 4100, torch.bfloat16, "none", True, False, torch.float32, 768),
]


@pytest.mark.parametrize("N,D,C,dtype,reduction,bias,cw,gdt,cols", CASES)
def test_recomputed_classes_match_oracle(cuda_lib, N, D, C, dtype, reduction, bias, cw, gdt, cols):
    inp = make_linear_inputs(N, D, C, dtype, "cuda", seed=N + C, bias=bias, w_std=0.5, b_std=0.3,
                             n_ignored=N // 17)
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    cwt = None
    if cw:
        cwt = torch.rand(C, generator=torch.Generator(device="cuda").manual_seed(3), device="cuda") + 0.25
    g = _grad_out(reduction, N, 7)
    esz = 2
    budget = N * cols * esz
    dt = lce_mod._DTYPE[dtype]
    gd = lce_mod._DTYPE[gdt or dtype]
    red = lce_mod._REDUCTION[reduction]
    ws = lce_mod.lce_workspace_size_for_buffer(lce_mod.LCE_OP_FORWARD_BACKWARD, N, D, C, dt, red, gd, budget)
    plan = _plan(lce_mod.LCE_OP_FORWARD_BACKWARD, N, D, C, dt, gd, ws)
    assert plan["Cb"] == cols and plan["nvc"] >= 1 and plan["nchunks"] == 1, plan
    workspace = torch.empty(ws, dtype=torch.uint8, device="cuda")
    loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, reduction, -100, g, grad_dtype=gdt,
                                                     workspace=workspace, class_weight=cwt)
    torch.cuda.synchronize()
    assert cuda_lib.lce_read_device_status(workspace) == 0
    tl, tg = _tol(dtype, gdt)
    _compare(loss, dX, dW, db, _oracle(X, W, b, t, reduction, g, cw=cwt), reduction, tl, tg)


def test_recomputed_and_batch_chunks_together(cuda_lib):
    """A workspace small enough that the rows are split into batch chunks and
    each chunk recomputes classes: dW summed over the batch chunks in fp32,
    dX over the class chunks."""
    N, D, C, dtype = 1500, 64, 2000, torch.bfloat16
    inp = make_linear_inputs(N, D, C, dtype, "cuda", seed=41, bias=True, w_std=0.5, b_std=0.3, n_ignored=30)
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    dt = lce_mod.LCE_BF16
    ws = None
    for budget in range(N * 256 * 2 - 1, 2 * 256 * 256, -4096):
        cand = cuda_lib.lce_workspace_size_for_buffer(lce_mod.LCE_OP_FORWARD_BACKWARD, N, D, C, dt,
                                                      lce_mod.LCE_RED_MEAN, dt, budget)
        p = _plan(lce_mod.LCE_OP_FORWARD_BACKWARD, N, D, C, dt, dt, cand)
        if p["nchunks"] > 1 and p["nvc"] > 0:
            ws = cand
            break
    assert ws is not None
    workspace = torch.empty(ws, dtype=torch.uint8, device="cuda")
    loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, "mean", -100, workspace=workspace)
    torch.cuda.synchronize()
    tl, tg = _tol(dtype, None)
    _compare(loss, dX, dW, db, _oracle(X, W, b, t, "mean", None), "mean", tl, tg)


def test_masked_classes_in_a_recomputed_chunk(cuda_lib):
    """A bias of -inf on whole tiles and on single classes inside recomputed
    chunks: probability 0, so their dW rows and db entries are 0, and the
    rest equals the problem with those classes deleted."""
    N, D, C = 600, 64, 2300
    inp = make_linear_inputs(N, D, C, torch.bfloat16, "cuda", seed=43, bias=True, w_std=0.5, b_std=0.3)
    X, W, b, t = inp["X"], inp["W"], inp["b"].clone(), inp["target"].clone()
    masked = torch.zeros(C, dtype=torch.bool, device="cuda")
    masked[1024:1280] = True          # a whole tile of the first recomputed chunk
    masked[1500:2300:37] = True       # scattered classes
    b[masked] = float("-inf")
    keep = (~masked).nonzero().squeeze(1)
    t = keep[torch.randint(0, keep.numel(), (N,), generator=torch.Generator(device="cuda").manual_seed(1),
                           device="cuda")]
    ws = cuda_lib.lce_workspace_size_for_buffer(lce_mod.LCE_OP_FORWARD_BACKWARD, N, D, C, lce_mod.LCE_BF16,
                                                lce_mod.LCE_RED_MEAN, lce_mod.LCE_BF16, N * 1024 * 2)
    workspace = torch.empty(ws, dtype=torch.uint8, device="cuda")
    loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, "mean", -100, workspace=workspace)
    torch.cuda.synchronize()
    assert torch.isfinite(dX).all() and torch.isfinite(dW).all() and torch.isfinite(db[keep]).all()
    assert (dW[masked] == 0).all() and (db[masked] == 0).all()
    # the same problem with the masked classes deleted
    remap = torch.full((C,), -1, dtype=torch.int64, device="cuda")
    remap[keep] = torch.arange(keep.numel(), device="cuda")
    ref = O.lce_forward_backward(to64(X), to64(W[keep]), to64(b[keep]), remap[t].cpu().numpy(), "mean")
    tl, tg = _tol(torch.bfloat16, None)
    assert rel_scalar(loss.item(), ref[0]) < tl
    assert rel_max(to64(dX), ref[1]) < tg
    assert rel_max(to64(dW[keep]), ref[2]) < tg
    assert rel_max(to64(db[keep]), ref[3]) < tg


BACKWARD_CASES = [
    # N, D, C, dtype, reduction, bias, grad dtype, buffer classes (None: default plan)
    (700, 136, 3001, torch.bfloat16, "none", True, None, None),
    (700, 136, 3001, torch.bfloat16, "none", True, None, 512),
    (1100, 64, 1000, torch.float16, "none", True, torch.float32, 256),
    (513, 72, 1800, torch.bfloat16, "mean", False, None, 768),
    (300, 40, 2500, torch.bfloat16, "sum", True, torch.bfloat16, None),
    (200, 33, 900, torch.float32, "none", True, None, None),  # fp32 inputs: lse not used
]


@pytest.mark.parametrize("N,D,C,dtype,reduction,bias,gdt,cols", BACKWARD_CASES)
def test_backward_from_lse_matches_oracle(cuda_lib, N, D, C, dtype, reduction, bias, gdt, cols):
    inp = make_linear_inputs(N, D, C, dtype, "cuda", seed=N + 2 * C, bias=bias, w_std=0.5, b_std=0.3,
                             n_ignored=N // 13)
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    g = _grad_out(reduction, N, 9)
    _, lse = cuda_lib.lce_forward(X, W, b, t, reduction, -100, want_lse=True)
    kw = {} if cols is None else {"buffer_bytes": N * cols * 2}
    dX, dW, db = cuda_lib.lce_backward(X, W, b, t, lse, reduction, -100, g, grad_dtype=gdt, **kw)
    torch.cuda.synchronize()
    tl, tg = _tol(dtype, gdt)
    _compare(None, dX, dW, db, _oracle(X, W, b, t, reduction, g), reduction, tl, tg)
    # and the same gradients as the fused call
    _, fX, fW, fb = cuda_lib.lce_forward_backward(X, W, b, t, reduction, -100, g, grad_dtype=gdt)
    torch.cuda.synchronize()
    assert rel_max(to64(dX), to64(fX)) < tg and rel_max(to64(dW), to64(fW)) < tg


def test_backward_degenerate_cases(cuda_lib):
    # no rows: dW and db are zero
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(300, 64, device="cuda").to(torch.bfloat16)
    b = torch.randn(300, device="cuda").to(torch.bfloat16)
    t = torch.empty(0, dtype=torch.int64, device="cuda")
    lse = torch.empty(0, dtype=torch.float32, device="cuda")
    dX, dW, db = cuda_lib.lce_backward(X, W, b, t, lse, "mean")
    torch.cuda.synchronize()
    assert dX.shape == (0, 64) and (dW == 0).all() and (db == 0).all()
    # every row ignored under mean: NaN gradients (the valid count is 0)
    inp = make_linear_inputs(40, 64, 300, torch.bfloat16, "cuda", seed=5, bias=True)
    t = torch.full((40,), -100, dtype=torch.int64, device="cuda")
    _, lse = cuda_lib.lce_forward(inp["X"], inp["W"], inp["b"], t, "mean", -100, want_lse=True)
    dX, dW, db = cuda_lib.lce_backward(inp["X"], inp["W"], inp["b"], t, lse, "mean")
    torch.cuda.synchronize()
    assert torch.isnan(dX).all() and torch.isnan(dW).all() and torch.isnan(db).all()
    # one class: every gradient is 0
    inp = make_linear_inputs(50, 16, 1, torch.bfloat16, "cuda", seed=6, bias=True)
    _, lse = cuda_lib.lce_forward(inp["X"], inp["W"], inp["b"], inp["target"], "sum", -100, want_lse=True)
    dX, dW, db = cuda_lib.lce_backward(inp["X"], inp["W"], inp["b"], inp["target"], lse, "sum")
    torch.cuda.synchronize()
    assert (dX == 0).all() and (dW == 0).all() and (db == 0).all()
    # a missing lse is an argument error
    with pytest.raises(lce_mod.LceError):
        lib = cuda_lib.load_library()
        ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
        P = lambda x: ctypes.c_void_p(x.data_ptr())
        code = lib.lce_backward(P(inp["X"]), P(inp["W"]), None, P(inp["target"]), None, 50, 16, 1, 1, 0, 1,
                                -100, None, P(dX), None, None, 1, P(ws), ws.numel(), None)
        cuda_lib._check(code, "lce_backward")
