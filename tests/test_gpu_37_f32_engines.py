"""Engine switches against the float64 oracle. fp32 inputs run on the
3xTF32 tensor-core engine by default (shapes only its TF32 operand copies
see: D not a multiple of 4, a K tail inside one 32-wide block, split-K on
dX) and on the SIMT fp32 engine with LCE_F32_SIMT=1; bf16 inputs run on the
one-CTA tcgen05 kernel with LCE_TC_PAIR=0. The switches are read once per
process, so those cases run in child processes."""

import os
import subprocess
import sys

import pytest
import torch

from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs
from tests.test_gpu_30_lce_small import _check

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("N,D,C", [(37, 37, 613), (300, 130, 2049), (513, 5, 700), (1100, 264, 9000)])
@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_tf32x3_shapes(cuda_lib, N, D, C, reduction):
    inp = make_linear_inputs(N, D, C, torch.float32, "cuda", seed=N + D + C, bias=True, w_std=0.5, b_std=0.3,
                             n_ignored=N // 10)
    cuda_lib.profile_reset()
    cuda_lib.profile_enable(True)
    try:
        _check(cuda_lib, inp, reduction)
    finally:
        cuda_lib.profile_enable(False)
    names = cuda_lib.profile_summary()
    assert "gemm_logits_3xtf32" in names and "gemm_dw_3xtf32" in names and "gemm_dx_3xtf32" in names
    assert "gemm_logits_simt" not in names


_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import linear_cross_entropy_lce_gb300 as L
from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs, make_workload
from tests.test_gpu_30_lce_small import _check
L.profile_enable(True)
_check(L, make_workload("tiny_fp32", "cuda"), "mean")
_check(L, make_linear_inputs(300, 130, 2049, torch.float32, "cuda", seed=4, bias=True, n_ignored=7), "sum")
_check(L, make_linear_inputs(600, 64, 1000, torch.float32, "cuda", seed=5), "mean", chunk_rows=128)
names = L.profile_summary()
assert "gemm_logits_simt" in names and "gemm_logits_3xtf32" not in names, names
print("SIMT-OK")
"""


def test_simt_engine_in_child_process():
    env = dict(os.environ, LCE_F32_SIMT="1")
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "SIMT-OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


_CHILD_ONE_CTA = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import linear_cross_entropy_lce_gb300 as L
from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs
from tests.test_gpu_30_lce_small import _check
L.profile_enable(True)
_check(L, make_linear_inputs(700, 64, 1000, torch.bfloat16, "cuda", seed=6, bias=True, w_std=0.2, n_ignored=9),
       "mean")
_check(L, make_linear_inputs(1300, 128, 2500, torch.bfloat16, "cuda", seed=7, bias=False, w_std=0.1), "sum")
_check(L, make_linear_inputs(300, 32, 600, torch.bfloat16, "cuda", seed=8, bias=True), "none")
print("ONE-CTA-OK")
"""


def test_one_cta_tensor_core_engine_in_child_process():
    """LCE_TC_PAIR=0 runs the bf16 path on the one-CTA tcgen05 kernel (128 x 256
    tiles) instead of CTA pairs; its logits and store epilogues against the
    oracle."""
    env = dict(os.environ, LCE_TC_PAIR="0")
    r = subprocess.run([sys.executable, "-c", _CHILD_ONE_CTA, ROOT], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "ONE-CTA-OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
