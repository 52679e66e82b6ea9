"""A seeded random sweep over the option space of the fused call against the
float64 oracle: input dtype (fp32 / bf16 / fp16), reduction, bias, ignored
rows, class weights, chunk size, gradient dtype, the subset of gradients
wanted, target distribution, and shapes with ragged tails on every
dimension (including row counts that take the row-slab path); and the same
for cross entropy on given logits (dtype, reduction, ignored rows, class
weights, logit scale, and class counts on both sides of the resident /
streaming kernel boundary); and the bounded backward (small gradient-buffer
budgets so that classes are recomputed, sometimes with batch chunks too,
through both gradient entry points). Each case is drawn from its own seed,
so a failure names a reproducible configuration."""

import random

import numpy as np
import pytest
import torch

from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs, make_logits_inputs
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu

N_CASES = 80


def _case(i):
    r = random.Random(1000 + i)
    dtype = r.choice([torch.float32, torch.bfloat16, torch.float16])
    sixteen = dtype != torch.float32
    N = r.choice([1, 7, 130, 777, 1100, 2300])
    D = r.choice([8, 24, 64, 136]) if sixteen else r.choice([5, 33, 64, 130])
    C = r.choice([1, 3, 255, 257, 1000, 3001])
    red = r.choice(["mean", "sum", "none"])
    n_ign = r.choice([0, 0, 1, N // 7, N // 2])
    if red == "mean":
        n_ign = min(n_ign, N - 1)
    case = dict(
        dtype=dtype, N=N, D=D, C=C, reduction=red, bias=r.random() < 0.5, n_ignored=n_ign,
        class_weight=r.random() < 0.3, chunk_rows=r.choice([0, 0, 128, 512]),
        grad_dtype=(torch.float32 if r.random() < 0.2 else
                    (r.choice([torch.bfloat16, torch.float16]) if dtype == torch.float32 and r.random() < 0.25
                     else None)),
        want=(tuple(r.random() < 0.7 for _ in range(3)) if r.random() < 0.2 else (True, True, True)),
        zipf=r.random() < 0.3, w_std=r.choice([0.05, 0.3, 1.0]), seed=r.randrange(1 << 30))
    return case


def _describe(c):
    return (f"{str(c['dtype']).split('.')[-1]} N={c['N']} D={c['D']} C={c['C']} {c['reduction']} "
            f"bias={c['bias']} ign={c['n_ignored']} cw={c['class_weight']} chunk={c['chunk_rows']} "
            f"gdt={c['grad_dtype']} want={c['want']} zipf={c['zipf']}")


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(cuda_lib, i):
    c = _case(i)
    inp = make_linear_inputs(c["N"], c["D"], c["C"], c["dtype"], "cuda", seed=c["seed"], bias=c["bias"],
                             w_std=c["w_std"], b_std=0.2, n_ignored=c["n_ignored"],
                             target_dist="zipf" if c["zipf"] else "uniform")
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    N, C = c["N"], c["C"]
    g = None
    if c["reduction"] == "none":
        g = torch.randn(N, generator=torch.Generator(device="cuda").manual_seed(c["seed"]), device="cuda")
    elif c["reduction"] == "sum":
        g = torch.tensor(0.75, device="cuda")
    cw = None
    if c["class_weight"]:
        cw = torch.rand(C, generator=torch.Generator(device="cuda").manual_seed(c["seed"] + 1),
                        device="cuda") * 1.8 + 0.2
    want_dx, want_dw, want_db = c["want"]
    loss, dX, dW, db = cuda_lib.lce_forward_backward(
        X, W, b, t, c["reduction"], -100, g, want_dx=want_dx, want_dw=want_dw, want_db=want_db,
        grad_dtype=c["grad_dtype"], chunk_rows=c["chunk_rows"], class_weight=cw)
    torch.cuda.synchronize()
    rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), c["reduction"], -100,
                                            to64(g), class_weight=to64(cw))
    tol = TOL[c["dtype"]]
    gtol = tol["grad"]
    if c["grad_dtype"] in (torch.bfloat16, torch.float16):  # 16-bit gradient storage
        gtol = max(gtol, TOL[c["grad_dtype"]]["grad"])
    what = _describe(c)
    if c["reduction"] == "none":
        assert rel_max(to64(loss), rl) < tol["loss"], what
    else:
        assert rel_scalar(loss.item(), rl) < tol["loss"], what
    for on, got, ref, name in ((want_dx, dX, rX, "dX"), (want_dw, dW, rW, "dW"),
                               (want_db and b is not None, db, rb, "db")):
        if on:
            assert got is not None and np.isfinite(to64(got)).all(), (name, what)
            assert rel_max(to64(got), ref) < gtol, (name, rel_max(to64(got), ref), what)
        else:
            assert got is None, (name, what)


N_BOUNDED = 60


def _bounded_case(i):
    r = random.Random(3000 + i)
    dtype = r.choice([torch.bfloat16, torch.float16])
    N = r.choice([9, 200, 777, 1100, 2300])
    D = r.choice([8, 64, 136, 264])
    C = r.choice([700, 1500, 3001, 5000])
    red = r.choice(["mean", "sum", "none"])
    n_ign = r.choice([0, 1, N // 7])
    if red == "mean":
        n_ign = min(n_ign, N - 1)
    cmin = max(256, -(-D // 256) * 256)
    cols = r.choice([cmin, cmin + 256, 1024])
    # mostly all rows with a narrow buffer; sometimes a budget below D classes
    # of all rows, which also splits the rows into batch chunks
    budget = N * cols * 2 if r.random() < 0.8 else max(256 * cmin * 2, N * cmin)
    return dict(dtype=dtype, N=N, D=D, C=C, reduction=red, bias=r.random() < 0.5, n_ignored=n_ign,
                class_weight=r.random() < 0.3, budget=budget, given_lse=r.random() < 0.4,
                grad_dtype=torch.float32 if r.random() < 0.25 else None,
                want=(tuple(r.random() < 0.7 for _ in range(3)) if r.random() < 0.2 else (True, True, True)),
                zipf=r.random() < 0.3, w_std=r.choice([0.05, 0.3, 1.0]), seed=r.randrange(1 << 30))


@pytest.mark.parametrize("i", range(N_BOUNDED))
def test_random_bounded_case(cuda_lib, i):
    """The bounded backward (classes recomputed beyond a small gradient
    buffer, sometimes with batch chunks too), through lce_forward_backward or
    lce_backward from the forward's lse."""
    c = _bounded_case(i)
    what = (f"{str(c['dtype']).split('.')[-1]} N={c['N']} D={c['D']} C={c['C']} {c['reduction']} "
            f"bias={c['bias']} ign={c['n_ignored']} cw={c['class_weight']} budget={c['budget']} "
            f"lse={c['given_lse']} gdt={c['grad_dtype']} want={c['want']}")
    inp = make_linear_inputs(c["N"], c["D"], c["C"], c["dtype"], "cuda", seed=c["seed"], bias=c["bias"],
                             w_std=c["w_std"], b_std=0.2, n_ignored=c["n_ignored"],
                             target_dist="zipf" if c["zipf"] else "uniform")
    X, W, b, t = inp["X"], inp["W"], inp["b"], inp["target"]
    N, C = c["N"], c["C"]
    g = None
    if c["reduction"] == "none":
        g = torch.randn(N, generator=torch.Generator(device="cuda").manual_seed(c["seed"]), device="cuda")
    elif c["reduction"] == "sum":
        g = torch.tensor(0.75, device="cuda")
    cw = None
    if c["class_weight"]:
        cw = torch.rand(C, generator=torch.Generator(device="cuda").manual_seed(c["seed"] + 1),
                        device="cuda") * 1.8 + 0.2
    want_dx, want_dw, want_db = c["want"]
    kw = dict(want_dx=want_dx, want_dw=want_dw, want_db=want_db, grad_dtype=c["grad_dtype"],
              class_weight=cw, buffer_bytes=c["budget"])
    loss = None
    if c["given_lse"]:
        _, lse = cuda_lib.lce_forward(X, W, b, t, c["reduction"], -100, want_lse=True, class_weight=cw)
        dX, dW, db = cuda_lib.lce_backward(X, W, b, t, lse, c["reduction"], -100, g, **kw)
    else:
        loss, dX, dW, db = cuda_lib.lce_forward_backward(X, W, b, t, c["reduction"], -100, g, **kw)
    torch.cuda.synchronize()
    rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), c["reduction"], -100,
                                            to64(g), class_weight=to64(cw))
    tol = TOL[c["dtype"]]
    gtol = tol["grad"]
    if loss is not None:
        if c["reduction"] == "none":
            assert rel_max(to64(loss), rl) < tol["loss"], what
        else:
            assert rel_scalar(loss.item(), rl) < tol["loss"], what
    for on, got, ref, name in ((want_dx, dX, rX, "dX"), (want_dw, dW, rW, "dW"),
                               (want_db and b is not None, db, rb, "db")):
        if on:
            assert got is not None and np.isfinite(to64(got)).all(), (name, what)
            assert rel_max(to64(got), ref) < gtol, (name, rel_max(to64(got), ref), what)
        else:
            assert got is None, (name, what)


def _ce_case(i):
    r = random.Random(5000 + i)
    dtype = r.choice([torch.float32, torch.bfloat16, torch.float16])
    N = r.choice([1, 5, 64, 300])
    V = r.choice([1, 2, 31, 1000, 16384, 16385, 40000, 131072, 140000])
    red = r.choice(["mean", "sum", "none"])
    n_ign = r.choice([0, 1, N // 3])
    if red == "mean":
        n_ign = min(n_ign, N - 1)
    return dict(dtype=dtype, N=N, V=V, reduction=red, n_ignored=n_ign, class_weight=r.random() < 0.3,
                std=r.choice([0.5, 2.0, 8.0]), seed=r.randrange(1 << 30))


@pytest.mark.parametrize("i", range(48))
def test_random_ce_case(cuda_lib, i):
    c = _ce_case(i)
    inp = make_logits_inputs(c["N"], c["V"], c["dtype"], "cuda", seed=c["seed"], std=c["std"],
                             n_ignored=c["n_ignored"])
    logits, t = inp["logits"], inp["target"]
    N, V = c["N"], c["V"]
    g = None
    if c["reduction"] == "none":
        g = torch.randn(N, generator=torch.Generator(device="cuda").manual_seed(c["seed"]), device="cuda")
    elif c["reduction"] == "sum":
        g = torch.tensor(1.5, device="cuda")
    cw = None
    if c["class_weight"]:
        cw = torch.rand(V, generator=torch.Generator(device="cuda").manual_seed(c["seed"] + 1),
                        device="cuda") * 1.8 + 0.2
    snap = to64(logits)
    loss = cuda_lib.lce_cross_entropy_from_logits(logits, t, c["reduction"], -100, g, class_weight=cw)
    torch.cuda.synchronize()
    rl, rg = O.ce_from_logits(snap, t.cpu().numpy(), c["reduction"], -100, to64(g), class_weight=to64(cw))
    tol = TOL[c["dtype"]]
    what = str(c)
    if c["reduction"] == "none":
        assert rel_max(to64(loss), rl) < tol["loss"], what
    else:
        assert rel_scalar(loss.item(), rl) < tol["loss"], what
    assert rel_max(to64(logits), rg) < tol["grad"], what
