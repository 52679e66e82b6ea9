"""The fused call is capturable in a CUDA graph: the library allocates
nothing, never synchronizes and issues only stream work, so one capture of
lce_forward_backward replays with new inputs written into the captured
buffers. Each replay is checked against the float64 oracle."""

import pytest
import torch

from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs
from oracle import lce_oracle as O
from tests.util import TOL, rel_max, rel_scalar, to64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,N,D,C", [(torch.float32, 300, 96, 1500), (torch.bfloat16, 1300, 128, 2500)])
def test_capture_and_replay(cuda_lib, dtype, N, D, C):
    src = [make_linear_inputs(N, D, C, dtype, "cuda", seed=s, bias=True, w_std=0.2, b_std=0.1, n_ignored=N // 20)
           for s in (1, 2)]
    X = src[0]["X"].clone()
    W = src[0]["W"].clone()
    b = src[0]["b"].clone()
    t = src[0]["target"].clone()
    nbytes = cuda_lib.lce_workspace_size(cuda_lib.LCE_OP_FORWARD_BACKWARD, N, D, C,
                                         cuda_lib.LCE_F32 if dtype == torch.float32 else cuda_lib.LCE_BF16,
                                         cuda_lib.LCE_RED_MEAN,
                                         cuda_lib.LCE_F32 if dtype == torch.float32 else cuda_lib.LCE_BF16, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    # one eager call first: per-kernel attributes are set on first use
    with torch.cuda.stream(stream):
        cuda_lib.lce_forward_backward(X, W, b, t, "mean", workspace=ws, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        out = cuda_lib.lce_forward_backward(X, W, b, t, "mean", workspace=ws, stream=stream)
    for s in src:
        X.copy_(s["X"])
        W.copy_(s["W"])
        b.copy_(s["b"])
        t.copy_(s["target"])
        graph.replay()
        torch.cuda.synchronize()
        loss, dX, dW, db = out
        rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), "mean")
        tol = TOL[dtype]
        assert rel_scalar(loss.item(), rl) < tol["loss"]
        for got, ref in ((dX, rX), (dW, rW), (db, rb)):
            assert rel_max(to64(got), ref) < tol["grad"]


@pytest.mark.parametrize("entry", ["forward_backward", "backward"])
def test_capture_and_replay_bounded(cuda_lib, entry):
    """The bounded plan (classes recomputed beyond a 512-class buffer, row
    slabs, the fp32 dX accumulator) and the backward from a given lse are
    capturable too: one capture, replayed on two sets of inputs."""
    N, D, C, dtype = 1100, 64, 2000, torch.bfloat16
    red = "none" if entry == "backward" else "mean"
    src = [make_linear_inputs(N, D, C, dtype, "cuda", seed=s, bias=True, w_std=0.4, b_std=0.2, n_ignored=N // 20)
           for s in (3, 4)]
    X, W, b, t = (src[0][k].clone() for k in ("X", "W", "b", "target"))
    g = torch.randn(N, device="cuda") if red == "none" else None
    op = cuda_lib.LCE_OP_BACKWARD if entry == "backward" else cuda_lib.LCE_OP_FORWARD_BACKWARD
    nbytes = cuda_lib.lce_workspace_size_for_buffer(op, N, D, C, cuda_lib.LCE_BF16, cuda_lib._REDUCTION[red],
                                                    cuda_lib.LCE_BF16, N * 512 * 2)
    plan = cuda_lib.plan_of(op, N, D, C, cuda_lib.LCE_BF16, cuda_lib.LCE_BF16, nbytes)
    assert plan["nvc"] >= 2, plan
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    lse = torch.empty(N, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def call():
        if entry == "backward":
            return cuda_lib.lce_backward(X, W, b, t, lse, red, -100, g, workspace=ws, stream=stream)
        return cuda_lib.lce_forward_backward(X, W, b, t, red, -100, g, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        call()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        out = call()
    for s in src:
        for dst, key in ((X, "X"), (W, "W"), (b, "b"), (t, "target")):
            dst.copy_(s[key])
        if entry == "backward":  # the lse of these inputs, outside the graph
            _, l2 = cuda_lib.lce_forward(X, W, b, t, red, -100, want_lse=True)
            lse.copy_(l2)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        rl, rX, rW, rb = O.lce_forward_backward(to64(X), to64(W), to64(b), t.cpu().numpy(), red, -100,
                                                None if g is None else to64(g))
        tol = TOL[dtype]
        if entry == "backward":
            dX, dW, db = out
        else:
            loss, dX, dW, db = out
            assert rel_scalar(loss.item(), rl) < tol["loss"]
        for got, ref in ((dX, rX), (dW, rW), (db, rb)):
            assert rel_max(to64(got), ref) < tol["grad"]
