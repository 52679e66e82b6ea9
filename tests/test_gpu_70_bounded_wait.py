"""The failure path of the bounded waits, on the GPU without a fault: the
CTA-pair GEMM in its dX form is launched with a side-job dependency that
nothing will satisfy (no unit can be claimed, the finished count stays 0).
The producer's wait gives up after its limit (about 2 s), every role of
the kernel unwinds through its own bounded waits, the status word carries
the timeout bit, and the context still runs a correct GEMM afterwards."""

import time

import torch
import pytest

from tests.util import rel_max

pytestmark = pytest.mark.gpu


def test_unmet_dependency_times_out_and_context_survives(cuda_lib):
    M, N, K = 512, 256, 256
    g = torch.Generator(device="cuda").manual_seed(3)
    A = torch.randn(M, K, generator=g, device="cuda").bfloat16()
    B = torch.randn(K, N, generator=g, device="cuda").bfloat16()  # MN-major B: [K, N]
    counters = torch.tensor([1 << 20, 0], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    cuda_lib.test_gemm_bf16_unmet_dependency(A, B, M, N, K, counters, status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(status.item()) & 2, "the timeout bit is set"
    assert int(counters[1].item()) == 0
    assert elapsed < 60.0
    # the context is intact: the same layout without the dependency is exact
    ref = A.double().cpu().numpy() @ B.double().cpu().numpy()
    ok_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = cuda_lib.test_gemm_bf16(A, B, M, N, K, 0, 1, status=ok_status, cta_pair=True)
    torch.cuda.synchronize()
    assert int(ok_status.item()) == 0
    assert rel_max(out.double().cpu().numpy(), ref) < 1e-5
