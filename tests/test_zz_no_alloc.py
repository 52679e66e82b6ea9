"""The allocation-free cross entropy entry point, for callers that cannot
allocate device memory when they need the loss (for example code inside a
caching allocator's hooks, or a runtime with a fixed memory budget that only
passes the buffers it owns). Called through the C ABI twice in a row, with
different inputs, it must match the regular entry point (which takes a
caller-allocated workspace) within the test tolerances. Collected last so
that a run stopping at its first failure has run every other test."""

import ctypes

import numpy as np
import pytest
import torch

import linear_cross_entropy_lce_gb300 as lce
from linear_cross_entropy_lce_gb300.workloads import make_logits_inputs
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, logits, t, reduction, g):
    N, V = logits.shape
    red = {"none": 0, "sum": 1, "mean": 2}[reduction]
    dt = lce.LCE_BF16 if logits.dtype == torch.bfloat16 else lce.LCE_F32
    loss = torch.empty(N if red == 0 else 1, dtype=torch.float32, device=logits.device)
    status = torch.full((1,), -1, dtype=torch.int32, device=logits.device)
    rc = lib.lce_cross_entropy_from_logits_noalloc(
        _p(logits), _p(t), N, V, dt, red, -100, _p(g), _p(loss), _p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lce.status_string(rc)
    return loss, status


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_workspace_entry_point(cuda_lib, dtype):
    lib = lce.load_library()
    calls = [  # two calls in a row with different data, sizes and reductions
        (make_logits_inputs(300, 40000, dtype, "cuda", seed=21, std=2.0, n_ignored=7), "mean", None),
        (make_logits_inputs(77, 5000, dtype, "cuda", seed=22, std=1.5, n_ignored=3), "none",
         torch.randn(77, device="cuda")),
    ]
    tol = TOL[dtype]
    for inp, reduction, g in calls:
        a = inp["logits"]
        snap = to64(a)  # the logits before either call overwrites its copy
        b = a.clone()
        t = inp["target"]
        ref_loss = lce.lce_cross_entropy_from_logits(a, t, reduction, -100, g)
        loss, status = _noalloc(lib, b, t, reduction, g)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        if reduction == "none":
            assert rel_max(to64(loss), to64(ref_loss)) < tol["loss"]
        else:
            assert rel_scalar(loss.item(), ref_loss.item()) < tol["loss"]
        assert rel_max(to64(b), to64(a)) < tol["grad"]
        # and against the float64 oracle directly
        rl, rg = O.ce_from_logits(snap, t.cpu().numpy(), reduction, -100, None if g is None else to64(g))
        if reduction == "none":
            assert rel_max(to64(loss), rl) < tol["loss"]
        else:
            assert rel_scalar(loss.item(), rl) < tol["loss"]
        assert rel_max(to64(b), rg) < tol["grad"]


def test_noalloc_at_the_row_limit(cuda_lib):
    """N == LCE_NOALLOC_MAX_ROWS fits the fixed scratch and matches the
    workspace entry point and the oracle (a narrow vocabulary keeps the
    logits at 32 MiB)."""
    lib = lce.load_library()
    N, V = lce.LCE_NOALLOC_MAX_ROWS, 8
    inp = make_logits_inputs(N, V, torch.float32, "cuda", seed=24, std=1.0, n_ignored=11)
    a = inp["logits"]
    t = inp["target"]
    snap = to64(a)
    b = a.clone()
    ref_loss = lce.lce_cross_entropy_from_logits(a, t, "mean", -100)
    loss, status = _noalloc(lib, b, t, "mean", None)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tol = TOL[torch.float32]
    assert rel_scalar(loss.item(), ref_loss.item()) < tol["loss"]
    assert rel_max(to64(b), to64(a)) < tol["grad"]
    rl, rg = O.ce_from_logits(snap, t.cpu().numpy(), "mean", -100)
    assert rel_scalar(loss.item(), rl) < tol["loss"]
    assert np.isfinite(to64(b)).all()
    assert rel_max(to64(b), rg) < tol["grad"]


def test_noalloc_limits_and_status(cuda_lib):
    lib = lce.load_library()
    fake = ctypes.c_void_p(4096)
    # more rows than the fixed scratch holds: rejected before any work
    too_many = lce.LCE_NOALLOC_MAX_ROWS + 1
    assert lib.lce_cross_entropy_from_logits_noalloc(fake, fake, too_many, 8, 0, 2, -100, None, fake, None,
                                                     None) == 2
    # a target out of range is reported through device_status
    inp = make_logits_inputs(9, 256, torch.float32, "cuda", seed=23)
    t = inp["target"].clone()
    t[4] = 256
    loss, status = _noalloc(lib, inp["logits"], t, "sum", None)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
