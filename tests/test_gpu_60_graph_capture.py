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
