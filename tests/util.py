"""Helpers shared by the GPU parity tests (no method arithmetic here)."""

import numpy as np
import torch

# Tolerances: fp32 inputs, loss rel 1e-5 and gradients rel 1e-4; bf16
# inputs, loss rel 2e-3 and gradients max|diff| / max|ref| <= 2e-2; fp16
# inputs (10-bit mantissa: the 16-bit G tile and 16-bit outputs each round at
# 2^-11 relative), loss rel 1e-3 and gradients 1e-2.
TOL = {
    torch.float32: {"loss": 1e-5, "grad": 1e-4},
    torch.bfloat16: {"loss": 2e-3, "grad": 2e-2},
    torch.float16: {"loss": 1e-3, "grad": 1e-2},
}


def to64(t):
    """Exact float64 copy of a device tensor (bf16 and fp32 upcast exactly)."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def rel_max(got, ref):
    """max |got - ref| / max |ref| (0/0 -> 0)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.max(np.abs(got - ref)) if got.size else 0.0
    s = np.max(np.abs(ref)) if ref.size else 0.0
    if s == 0.0:
        return float(d)
    return float(d / s)


def rel_scalar(got, ref):
    got = float(got)
    ref = float(ref)
    if ref == 0.0:
        return abs(got)
    return abs(got - ref) / abs(ref)
