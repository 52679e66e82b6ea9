"""Full-size bf16 heads, in the launch configuration the benchmark times
(the default workspace plan, whose gradient buffer is bounded by 1 GiB, so
part or all of the classes are recomputed), against the float64 oracle: a
full blockwise pass gives every row's lse, the loss and db; dX is checked
on sampled rows and dW on sampled classes (the most frequent targets,
classes no row targets, and random ones, in stored and recomputed class
chunks alike)."""

import numpy as np
import pytest
import torch

from linear_cross_entropy_lce_gb300.workloads import WORKLOADS, make_workload
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample_classes(t, C, rng, k=256):
    valid = t[t != -100]
    counts = np.bincount(valid, minlength=C)
    top = np.argsort(-counts)[:8]
    unused = np.nonzero(counts == 0)[0]
    none8 = unused[rng.choice(len(unused), min(8, len(unused)), replace=False)] if len(unused) else []
    rest = rng.choice(C, k - len(top) - len(none8), replace=False)
    return np.unique(np.concatenate([top, none8, rest]).astype(np.int64))


@pytest.mark.timeout(3600)
@pytest.mark.parametrize("name", ["bf16_llm_head", "bf16_large_head"])
def test_full_size_head(cuda_lib, name):
    w = WORKLOADS[name]
    inp = make_workload(name, "cuda")
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    g = inp["grad_out"]
    if w.reduction == "none":
        # the benchmark's launch configuration for reduction none: the
        # forward (loss and lse), then the backward from that lse (every
        # class recomputed under the default 1 GiB buffer)
        loss_f, lse = cuda_lib.lce_forward(X, W, b, t, w.reduction, -100, want_lse=True)
        dX, dW, db = cuda_lib.lce_backward(X, W, b, t, lse, w.reduction, -100, g)
        loss = loss_f
    else:
        loss_f = cuda_lib.lce_forward(X, W, b, t, w.reduction, -100)
        loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, w.reduction, -100, g)
    torch.cuda.synchronize()
    # exact host copies of the bf16 inputs (float32 holds every bf16 value)
    Xh = X.float().cpu().numpy()
    Wh = W.float().cpu().numpy()
    bh = None if b is None else b.double().cpu().numpy()
    th = t.cpu().numpy()
    gh = None if g is None else g.double().cpu().numpy()
    st = O.forward_stats(Xh, Wh, bh, th, w.reduction, grad_out=gh, want_db=b is not None, row_block=512)
    tol = TOL[torch.bfloat16]
    if w.reduction == "none":
        assert rel_max(loss.double().cpu().numpy(), st["loss_rows"]) < tol["loss"]
        assert rel_max(loss_f.double().cpu().numpy(), st["loss_rows"]) < tol["loss"]
    else:
        assert rel_scalar(loss.item(), st["loss"]) < tol["loss"]
        assert rel_scalar(loss_f.item(), st["loss"]) < tol["loss"]
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(w.N, 256, replace=False))
    _, dXr = O.grad_rows(Xh, Wh, bh, th, st["lse"], st["w"], rows)
    assert rel_max(dX[torch.from_numpy(rows).cuda()].double().cpu().numpy(), dXr) < tol["grad"]
    cls = _sample_classes(th, w.C, rng)
    dWc, dbc = O.dw_rows(Xh, Wh, bh, th, st["lse"], st["w"], cls)
    assert rel_max(dW[torch.from_numpy(cls).cuda()].double().cpu().numpy(), dWc) < tol["grad"]
    if b is not None:
        assert rel_max(db.double().cpu().numpy(), st["db"]) < tol["grad"]
    assert torch.isfinite(dX).all() and torch.isfinite(dW).all()


@pytest.mark.timeout(3600)
def test_full_size_llm_head_whole_buffer(cuda_lib):
    """The LLM head with every class stored (no recomputation): the plan
    the benchmark reports beside the bounded one."""
    w = WORKLOADS["bf16_llm_head"]
    inp = make_workload("bf16_llm_head", "cuda")
    X, W, t = inp["X"], inp["W"], inp["target"]
    loss, dX, dW, _ = cuda_lib.lce_forward_backward(X, W, None, t, w.reduction, -100, chunk_rows=w.N)
    torch.cuda.synchronize()
    Xh = X.float().cpu().numpy()
    Wh = W.float().cpu().numpy()
    th = t.cpu().numpy()
    st = O.forward_stats(Xh, Wh, None, th, w.reduction, row_block=512)
    tol = TOL[torch.bfloat16]
    assert rel_scalar(loss.item(), st["loss"]) < tol["loss"]
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(w.N, 128, replace=False))
    _, dXr = O.grad_rows(Xh, Wh, None, th, st["lse"], st["w"], rows)
    assert rel_max(dX[torch.from_numpy(rows).cuda()].double().cpu().numpy(), dXr) < tol["grad"]
    cls = _sample_classes(th, w.C, rng, k=128)
    dWc, _ = O.dw_rows(Xh, Wh, None, th, st["lse"], st["w"], cls)
    assert rel_max(dW[torch.from_numpy(cls).cuda()].double().cpu().numpy(), dWc) < tol["grad"]


@pytest.mark.timeout(3600)
def test_full_size_llm_head_f16_class_weights(cuda_lib):
    """The widened rows at full size, as the bench's variants run them: the
    LLM head's inputs in fp16 with per-class weights (uniform in [0.5, 1.5),
    seed 7), default plan (classes beyond the 1 GiB buffer recomputed),
    against the float64 oracle on the exact fp16 values."""
    w = WORKLOADS["bf16_llm_head"]
    inp = make_workload("bf16_llm_head", "cuda")
    X, W, t = inp["X"].half(), inp["W"].half(), inp["target"]
    gen = torch.Generator(device="cuda").manual_seed(7)
    cw = torch.rand(w.C, generator=gen, device="cuda") + 0.5
    loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, None, t, "mean", -100, class_weight=cw)
    torch.cuda.synchronize()
    Xh = X.float().cpu().numpy()
    Wh = W.float().cpu().numpy()
    th = t.cpu().numpy()
    cwh = cw.double().cpu().numpy()
    st = O.forward_stats(Xh, Wh, None, th, "mean", row_block=512, class_weight=cwh)
    tol = TOL[torch.float16]
    assert rel_scalar(loss.item(), st["loss"]) < tol["loss"]
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(w.N, 256, replace=False))
    _, dXr = O.grad_rows(Xh, Wh, None, th, st["lse"], st["w"], rows)
    assert rel_max(dX[torch.from_numpy(rows).cuda()].double().cpu().numpy(), dXr) < tol["grad"]
    cls = _sample_classes(th, w.C, rng)
    dWc, _ = O.dw_rows(Xh, Wh, None, th, st["lse"], st["w"], cls)
    assert rel_max(dW[torch.from_numpy(cls).cuda()].double().cpu().numpy(), dWc) < tol["grad"]
    assert torch.isfinite(dX).all() and torch.isfinite(dW).all()
