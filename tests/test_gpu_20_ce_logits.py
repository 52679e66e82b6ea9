"""Cross entropy on given logits with the gradient written in place, against
the float64 oracle on a snapshot of the logits taken before the call."""

import math

import numpy as np
import pytest
import torch

from linear_cross_entropy_lce_gb300.workloads import make_logits_inputs, make_workload
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu

CASES = [
    # (N, V, dtype, reduction, n_ignored)  resident kernel unless noted
    (37, 1000, torch.float32, "mean", 3),
    (64, 40000, torch.float32, "sum", 5),       # cluster of 4
    (16, 131072, torch.float32, "mean", 0),     # cluster of 8
    (19, 1001, torch.float32, "mean", 2),       # V % 4 != 0: streaming kernel
    (9, 200003, torch.float32, "sum", 1),       # V * 4 bytes not a multiple of 16: streaming kernel
    (12, 150000, torch.float32, "mean", 2),     # cluster of 16 (non-portable size)
    (6, 262144, torch.float32, "none", 1),      # cluster of 16, full slices
    (10, 200000, torch.bfloat16, "sum", 1),     # cluster of 16, bf16
    (5, 262148, torch.float32, "mean", 1),      # V > 16 * 16384: streaming kernel
    (33, 50000, torch.bfloat16, "mean", 4),
    (20, 777, torch.bfloat16, "none", 2),       # streaming (V % 8 != 0)
    (25, 4096, torch.float32, "none", 3),
]


@pytest.mark.parametrize("N,V,dtype,reduction,n_ign", CASES)
def test_ce_logits_small(cuda_lib, N, V, dtype, reduction, n_ign):
    inp = make_logits_inputs(N, V, dtype, "cuda", seed=N + V, std=2.0, n_ignored=n_ign)
    logits, t = inp["logits"], inp["target"]
    snap = to64(logits)
    tn = t.cpu().numpy()
    g = None
    if reduction == "none":
        g = torch.randn(N, device="cuda")
    elif reduction == "sum":
        g = torch.tensor(0.75, device="cuda")
    loss = cuda_lib.lce_cross_entropy_from_logits(logits, t, reduction, -100, g)
    torch.cuda.synchronize()
    gn = None if g is None else to64(g)
    ref_loss, ref_grad = O.ce_from_logits(snap, tn, reduction, -100, gn)
    tol = TOL[dtype]
    if reduction == "none":
        assert rel_max(to64(loss), ref_loss) < tol["loss"]
    else:
        assert rel_scalar(loss.item(), ref_loss) < tol["loss"]
    assert rel_max(to64(logits), ref_grad) < tol["grad"]


def test_ce_logits_full_size_sampled(cuda_lib):
    """[16384, 131072] fp32, mean: the profiled shape of the in-place kernel."""
    inp = make_workload("ce_logits_fp32", device="cuda")
    logits, t = inp["logits"], inp["target"]
    N, V = logits.shape
    rows = np.sort(np.random.default_rng(0).choice(N, 512, replace=False))
    rows_t = torch.from_numpy(rows).cuda()
    snap_rows = to64(logits[rows_t])
    tn = t.cpu().numpy()
    # full float64 pass for the mean loss, on a host copy taken before the call
    host = logits.cpu()
    ref_loss, _ = O.ce_from_logits(host.numpy(), tn, "mean", -100, want_grad=False)
    del host
    loss = cuda_lib.lce_cross_entropy_from_logits(logits, t, "mean", -100)
    torch.cuda.synchronize()
    assert rel_scalar(loss.item(), ref_loss) < 1e-5
    w = O.row_weights(tn, V, "mean")
    _, G = O.ce_rows(snap_rows, tn[rows], w[rows])
    assert rel_max(to64(logits[rows_t]), G) < 1e-4


def test_ce_logits_edge_cases(cuda_lib):
    # every row ignored under mean: NaN loss and NaN gradient
    inp = make_logits_inputs(6, 300, torch.float32, "cuda", seed=1)
    t = torch.full((6,), -100, dtype=torch.int64, device="cuda")
    logits = inp["logits"]
    loss = cuda_lib.lce_cross_entropy_from_logits(logits, t, "mean")
    torch.cuda.synchronize()
    assert math.isnan(loss.item()) and torch.isnan(logits).all()
    # N = 0
    e = torch.empty(0, 300, device="cuda")
    te = torch.empty(0, dtype=torch.int64, device="cuda")
    assert math.isnan(cuda_lib.lce_cross_entropy_from_logits(e, te, "mean").item())
    assert cuda_lib.lce_cross_entropy_from_logits(e, te, "sum").item() == 0.0
    # a target out of range: status bit, that row gets loss 0 and gradient 0
    inp = make_logits_inputs(5, 64, torch.float32, "cuda", seed=2)
    logits, t = inp["logits"], inp["target"].clone()
    t[2] = 64
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    loss = cuda_lib.lce_cross_entropy_from_logits(logits, t, "none", -100, torch.ones(5, device="cuda"),
                                                  workspace=ws)
    assert cuda_lib.lce_read_device_status(ws) == 8
    assert loss[2].item() == 0.0 and (logits[2] == 0).all()


@pytest.mark.parametrize("V,dtype", [
    (40000, torch.float32),     # resident, cluster of 4
    (131072, torch.float32),    # resident, cluster of 8
    (50000, torch.bfloat16),    # resident, bf16
    (1001, torch.float32),      # streaming
])
def test_ce_logits_masked_columns(cuda_lib, V, dtype):
    """Logits masked with -inf (a vocabulary mask): a contiguous block that
    covers whole per-thread slices of the resident kernel, scattered entries
    on every other row, and one row that is -inf everywhere but its target.
    Masked columns get probability 0, hence gradient 0; the last row has
    loss 0 and gradient 0."""
    N = 9
    inp = make_logits_inputs(N, V, dtype, "cuda", seed=V + 7, std=2.0, n_ignored=1)
    logits, t = inp["logits"], inp["target"].clone()
    logits[:, V // 4: V // 2] = -math.inf
    logits[::2, ::3] = -math.inf
    # targets in columns that stay finite: j < V // 4 and j % 3 == 1
    valid = t != -100
    t[valid] = 1 + 3 * (torch.arange(int(valid.sum()), device="cuda") * 37 % (V // 12))
    r = int(torch.nonzero(valid)[-1])
    keep = logits[r, t[r]].clone()
    logits[r] = -math.inf
    logits[r, t[r]] = keep
    snap = to64(logits)
    tn = t.cpu().numpy()
    loss = cuda_lib.lce_cross_entropy_from_logits(logits, t, "none", -100, torch.ones(N, device="cuda"))
    torch.cuda.synchronize()
    ref_loss, ref_grad = O.ce_from_logits(snap, tn, "none", -100, np.ones(N))
    tol = TOL[dtype]
    got = to64(logits)
    assert np.isfinite(got).all()
    assert rel_max(to64(loss), ref_loss) < tol["loss"]
    assert rel_max(got, ref_grad) < tol["grad"]
    assert (got[np.isneginf(snap)] == 0).all()
    assert loss[r].item() == 0.0 and (got[r] == 0).all()
