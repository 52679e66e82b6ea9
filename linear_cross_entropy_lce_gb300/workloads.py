"""Seeded synthetic workloads for the fused linear + cross-entropy loss.

This module only draws random inputs; it holds none of the method's
arithmetic, so both the CUDA path and the float64 oracle can be fed from it.
The five named workloads follow the shapes and value distributions of the
source pages' workloads:

* ``tiny_fp32``        N=64, D=32, C=512; X, W ~ N(0,1)/sqrt(D); bias ~ N(0, 0.1);
                       uniform targets with 4 rows set to ignore_index; mean.
* ``fp32_mid``         N=2048, D=512, C=8192; X ~ N(0,1); W ~ N(0, 1/D) (variance);
                       no bias; uniform targets; sum.
* ``bf16_llm_head``    N=8192, D=4096, C=128256; X ~ N(0,1); W ~ N(0, 0.02);
                       no bias; Zipf(1.1) targets, 5 % ignored; mean.
* ``ce_logits_fp32``   logits [16384, 131072] ~ N(0,1) (B=8 x T=2048, the shape
                       profiled in Liger-Kernel issue #343); uniform targets; mean.
* ``bf16_large_head``  N=16384, D=4096, C=131072; X ~ N(0,1); W ~ N(0, 0.02);
                       bias ~ N(0, 0.01); uniform targets; reduction none with a
                       per-row upstream gradient ~ N(0,1).

Readings: "N(0, s)" with a literal s is a standard deviation, "N(0, 1/D)" a
variance; Zipf(s) is p(k) ~ k^-s over k = 1..C, class id k-1, drawn by
inverse CDF; "k rows ignored" are the first k of a seeded permutation.
Seeds: 0..4 in the order above. Random numbers come from torch.Generator on
the requested device, so a CUDA run and its host copy see the same values.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

IGNORE_INDEX = -100


@dataclasses.dataclass
class Workload:
    name: str
    N: int
    D: int  # 0 for the logits-given workload
    C: int  # number of classes (V for the logits-given workload)
    dtype: torch.dtype
    reduction: str
    bias: bool
    seed: int
    x_std: float = 1.0
    w_std: float = 1.0
    b_std: float = 0.0
    scale_by_sqrt_d: bool = False
    target_dist: str = "uniform"  # or "zipf"
    zipf_s: float = 1.1
    n_ignored: int = 0
    grad_out_std: Optional[float] = None  # per-row upstream gradient for 'none'
    kind: str = "linear"  # "linear" or "logits"

    @property
    def flops_fwd_bwd(self) -> float:
        """Algorithmic flops of one forward+backward: 2NDC for the logits and
        2NDC each for dX and dW (reduction='none' adds a 2NDC forward)."""
        base = 6.0 * self.N * self.D * self.C
        return base + (2.0 * self.N * self.D * self.C if self.reduction == "none" else 0.0)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 64, 32, 512, torch.float32, "mean", True, 0,
                          x_std=1.0, w_std=1.0, b_std=0.1, scale_by_sqrt_d=True, n_ignored=4),
    "fp32_mid": Workload("fp32_mid", 2048, 512, 8192, torch.float32, "sum", False, 1,
                         x_std=1.0, w_std=1.0 / math.sqrt(512)),
    "bf16_llm_head": Workload("bf16_llm_head", 8192, 4096, 128256, torch.bfloat16, "mean", False, 2,
                              x_std=1.0, w_std=0.02, target_dist="zipf", n_ignored=410),
    "ce_logits_fp32": Workload("ce_logits_fp32", 16384, 0, 131072, torch.float32, "mean", False, 3,
                               x_std=1.0, kind="logits"),
    "bf16_large_head": Workload("bf16_large_head", 16384, 4096, 131072, torch.bfloat16, "none", True, 4,
                                x_std=1.0, w_std=0.02, b_std=0.01, grad_out_std=1.0),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_targets(N, C, gen, device, dist="uniform", zipf_s=1.1, n_ignored=0,
                 ignore_index=IGNORE_INDEX):
    """int64 targets in [0, C); the first n_ignored rows of a seeded
    permutation are set to ignore_index."""
    if N == 0:
        return torch.empty(0, dtype=torch.int64, device=device)
    if dist == "uniform":
        t = torch.randint(0, C, (N,), generator=gen, device=device, dtype=torch.int64)
    elif dist == "zipf":
        k = torch.arange(1, C + 1, device=device, dtype=torch.float64)
        p = k.pow(-zipf_s)
        cdf = torch.cumsum(p, 0)
        cdf = cdf / cdf[-1]
        u = torch.rand(N, generator=gen, device=device, dtype=torch.float64)
        t = torch.searchsorted(cdf, u).clamp_(max=C - 1).to(torch.int64)
    else:
        raise ValueError(dist)
    if n_ignored:
        perm = torch.randperm(N, generator=gen, device=device)
        t[perm[:n_ignored]] = ignore_index
    return t


def make_linear_inputs(N, D, C, dtype=torch.float32, device="cpu", seed=0, bias=False,
                       x_std=1.0, w_std=1.0, b_std=0.1, scale_by_sqrt_d=False,
                       target_dist="uniform", zipf_s=1.1, n_ignored=0,
                       grad_out_std=None, ignore_index=IGNORE_INDEX):
    """Draw X [N, D], W [C, D], b [C] or None, target [N] int64 and an optional
    per-row upstream gradient [N] fp32, all on ``device``."""
    gen = _gen(device, seed)
    X = torch.randn(N, D, generator=gen, device=device, dtype=torch.float32) * x_std
    W = torch.randn(C, D, generator=gen, device=device, dtype=torch.float32) * w_std
    if scale_by_sqrt_d:
        X = X / math.sqrt(D)
        W = W / math.sqrt(D)
    b = None
    if bias:
        b = torch.randn(C, generator=gen, device=device, dtype=torch.float32) * b_std
    t = draw_targets(N, C, gen, device, target_dist, zipf_s, n_ignored, ignore_index)
    g = None
    if grad_out_std is not None:
        g = torch.randn(N, generator=gen, device=device, dtype=torch.float32) * grad_out_std
    X = X.to(dtype).contiguous()
    W = W.to(dtype).contiguous()
    if b is not None:
        b = b.to(dtype).contiguous()
    return {"X": X, "W": W, "b": b, "target": t, "grad_out": g}


def make_logits_inputs(N, V, dtype=torch.float32, device="cpu", seed=0, std=1.0,
                       target_dist="uniform", n_ignored=0, ignore_index=IGNORE_INDEX):
    """Draw logits [N, V] ~ N(0, std) and int64 targets [N]."""
    gen = _gen(device, seed)
    logits = (torch.randn(N, V, generator=gen, device=device, dtype=torch.float32) * std).to(dtype)
    t = draw_targets(N, V, gen, device, target_dist, 1.1, n_ignored, ignore_index)
    return {"logits": logits.contiguous(), "target": t}


def make_workload(name: str, device="cpu"):
    """Inputs of one named workload on ``device``."""
    w = WORKLOADS[name]
    if w.kind == "logits":
        return make_logits_inputs(w.N, w.C, w.dtype, device, w.seed, w.x_std,
                                  w.target_dist, w.n_ignored)
    return make_linear_inputs(w.N, w.D, w.C, w.dtype, device, w.seed, w.bias,
                              w.x_std, w.w_std, w.b_std, w.scale_by_sqrt_d,
                              w.target_dist, w.zipf_s, w.n_ignored, w.grad_out_std)
