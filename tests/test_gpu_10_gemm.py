"""The GEMM engines on their own: tcgen05 (bf16, TMA + tensor memory),
3xTF32 on the tensor cores (fp32) and SIMT (fp32), in the four operand
layouts, against a float64 matmul of the same values."""

import numpy as np
import pytest
import torch

from tests.util import rel_max

pytestmark = pytest.mark.gpu

LAYOUTS = [(0, 0), (0, 1), (1, 0), (1, 1)]
SHAPES = [(128, 256, 64), (296, 520, 200), (1024, 768, 1000), (8, 16, 8)]


def _operands(M, N, K, a_mn, b_mn, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn(K, M, generator=g, device="cuda") if a_mn else torch.randn(M, K, generator=g, device="cuda")
    B = torch.randn(K, N, generator=g, device="cuda") if b_mn else torch.randn(N, K, generator=g, device="cuda")
    A = A.to(dtype).contiguous()
    B = B.to(dtype).contiguous()
    A64 = A.double().cpu().numpy()
    B64 = B.double().cpu().numpy()
    Am = A64.T if a_mn else A64  # [M, K]
    Bm = B64.T if b_mn else B64  # [N, K]
    return A, B, Am @ Bm.T


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("a_mn,b_mn", LAYOUTS)
@pytest.mark.parametrize("M,N,K", SHAPES + [(600, 800, 136)])
def test_tcgen05_gemm(cuda_lib, a_mn, b_mn, M, N, K, pair):
    A, B, ref = _operands(M, N, K, a_mn, b_mn, torch.bfloat16, 11 + M + N + K)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = cuda_lib.test_gemm_bf16(A, B, M, N, K, a_mn, b_mn, status=status, cta_pair=pair)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert rel_max(out.double().cpu().numpy(), ref) < 1e-5


@pytest.mark.parametrize("a_mn,b_mn", LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 16), (300, 517, 203), (7, 3, 5)])
def test_simt_gemm(cuda_lib, a_mn, b_mn, M, N, K):
    A, B, ref = _operands(M, N, K, a_mn, b_mn, torch.float32, 5 + M + N + K)
    out = cuda_lib.test_gemm_f32(A, B, M, N, K, a_mn, b_mn)
    torch.cuda.synchronize()
    assert rel_max(out.double().cpu().numpy(), ref) < 1e-5


@pytest.mark.parametrize("a_mn,b_mn", LAYOUTS)
@pytest.mark.parametrize("M,N,K,splits", [(256, 256, 32, 1), (300, 517, 203, 1), (7, 3, 5, 1),
                                          (1000, 600, 3000, 1), (520, 260, 4100, 5)])
def test_tf32x3_gemm(cuda_lib, a_mn, b_mn, M, N, K, splits):
    """Three TF32 products reach fp32 accuracy: the error bound of the split
    (about 2^-21 of |A||B| per product) keeps the result within 1e-5 of the
    float64 matmul relative to its largest entry."""
    A, B, ref = _operands(M, N, K, a_mn, b_mn, torch.float32, 17 + M + N + K)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = cuda_lib.test_gemm_tf32x3(A, B, M, N, K, a_mn, b_mn, k_splits=splits, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert rel_max(out.double().cpu().numpy(), ref) < 1e-5


def test_tf32x3_beats_one_tf32_product(cuda_lib):
    """The lo parts matter: a single TF32 product per element (relative
    error about 2^-11 each) leaves about 1e-4 of the largest entry at this
    K; the three products with folded partial sums stay below 1e-5."""
    M, N, K = 512, 512, 1024
    A, B, ref = _operands(M, N, K, 0, 0, torch.float32, 99)
    out = cuda_lib.test_gemm_tf32x3(A, B, M, N, K, 0, 0)
    torch.cuda.synchronize()
    err = np.abs(out.double().cpu().numpy() - ref).max() / np.abs(ref).max()
    assert err < 1e-5
