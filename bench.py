"""Benchmark of the fused linear + cross-entropy forward+backward on GB300.

Default: the bf16 LLM-head workload (N=8192 tokens, D=4096, C=128256, Zipf
targets, 5% ignored, mean), one step = one lce_forward_backward call (loss,
dX, dW) on inputs resident in HBM, with the library's default workspace
plan (gradient buffer bounded by 1 GiB). Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl reference] [--dtype f16] [--class-weights]
                  [--api autograd]

--dtype f16 runs a bf16 workload's inputs in fp16, --class-weights adds
per-class cross-entropy weights (the _ex entry points), --api autograd
times the step through linear_cross_entropy(...).backward(); each prints
the same JSON line for that variant of the workload.

--impl reference times the float64 CPU oracle on the host cores on a
bounded sample of the same workload (the method has no other reference
implementation). With torchrun (N > 1) every rank runs an independent
replica (the step does not shard); rank 0 prints.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_cross_entropy_lce_gb300.workloads import WORKLOADS, make_workload  # noqa: E402

METRIC = "fused linear-CE fwd+bwd tokens/s and TFLOP/s at 1 GB300; % bf16 tensor peak"


# DRAM bytes (read + write) per launch of a kernel, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum): {(workload, kernel):
# (bytes, commit of the capture, hash of the kernel's sources at the
# capture)}. The bench reports an entry only while those sources hash the
# same, so a capture never outlives a change of the kernel it measured.
MEASURED_TRAFFIC = {
    # full-size one-pass captures (gpu__time_duration.sum, dram__bytes_read.sum,
    # dram__bytes_write.sum) of one step after one warm-up step
    ("bf16_llm_head", "gemm_logits_tc"): (1710572416, "f97684c", "08ce547b25b2a1b7"),  # mean of 4 launches
    ("bf16_llm_head", "gemm_dx_tc"): (5836620416, "f97684c", "08ce547b25b2a1b7"),  # mean of 2 launches
    ("bf16_llm_head", "gemm_dw_tc"): (4515026816, "f97684c", "08ce547b25b2a1b7"),  # mean of 2 launches
    ("bf16_llm_head", "gemm_recompute_tc"): (2388614144, "f97684c", "08ce547b25b2a1b7"),  # mean of 1 launches
    ("bf16_large_head", "gemm_logits_tc"): (4606856448, "f97684c", "08ce547b25b2a1b7"),  # mean of 1 launches
    ("bf16_large_head", "gemm_recompute_tc"): (2726271488, "f97684c", "08ce547b25b2a1b7"),  # mean of 4 launches
    ("bf16_large_head", "gemm_dx_tc"): (6234672448, "f97684c", "08ce547b25b2a1b7"),  # mean of 4 launches
    ("bf16_large_head", "gemm_dw_tc"): (5786866944, "f97684c", "08ce547b25b2a1b7"),  # mean of 4 launches
    ("ce_logits_fp32", "ce_resident"): (17415280640, "3a95670", "cbc8eadfcfbde878"),
    ("tiny_fp32", "gemm_logits_3xtf32"): (301312, "acaef4c", "f5ad3eb2b57b7737"),
    ("tiny_fp32", "gemm_dx_3xtf32"): (507392, "acaef4c", "f5ad3eb2b57b7737"),
    ("tiny_fp32", "gemm_dw_3xtf32"): (392192, "acaef4c", "f5ad3eb2b57b7737"),
    ("fp32_mid", "gemm_logits_3xtf32"): (52630528, "acaef4c", "f5ad3eb2b57b7737"),
    ("fp32_mid", "gemm_dx_3xtf32"): (179888384, "acaef4c", "f5ad3eb2b57b7737"),
    ("fp32_mid", "gemm_dw_3xtf32"): (143001344, "acaef4c", "f5ad3eb2b57b7737"),
}

CSRC = os.path.join(ROOT, "linear_cross_entropy_lce_gb300", "csrc")
# the sources each kernel is built from
_GEMM_SOURCES = ("common.cuh", "ptx.cuh", "epilogues.cuh", "tc2_gemm.cuh", "combine_unit.cuh", "grad_unit.cuh",
                 "gemm_tc.cu", "internal.h")
KERNEL_SOURCES = {
    "gemm_logits_tc": _GEMM_SOURCES, "gemm_recompute_tc": _GEMM_SOURCES, "gemm_dx_tc": _GEMM_SOURCES,
    "gemm_dw_tc": _GEMM_SOURCES,
    "ce_resident": ("common.cuh", "ptx.cuh", "ce_logits.cu", "internal.h"),
    "ce_stream": ("common.cuh", "ptx.cuh", "ce_logits.cu", "internal.h"),
    "gemm_logits_3xtf32": ("common.cuh", "ptx.cuh", "epilogues.cuh", "tc2x3_gemm.cuh", "gemm_tf32.cu", "internal.h"),
    "gemm_dx_3xtf32": ("common.cuh", "ptx.cuh", "epilogues.cuh", "tc2x3_gemm.cuh", "gemm_tf32.cu", "internal.h"),
    "gemm_dw_3xtf32": ("common.cuh", "ptx.cuh", "epilogues.cuh", "tc2x3_gemm.cuh", "gemm_tf32.cu", "internal.h"),
}


def kernel_sources_hash(kernel):
    """sha256 (16 hex digits) over the CUDA sources the kernel is built from
    (every source file for a kernel not in KERNEL_SOURCES)."""
    import hashlib

    files = KERNEL_SOURCES.get(kernel)
    if files is None:
        files = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h")))
    h = hashlib.sha256()
    for fn in sorted(files):
        with open(os.path.join(CSRC, fn), "rb") as f:
            h.update(fn.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload, kernel):
    """(bytes per launch or None, note)."""
    e = MEASURED_TRAFFIC.get((workload, kernel))
    if e is None:
        return None, "no ncu capture recorded for this kernel and workload"
    nbytes, commit, src = e
    if src != kernel_sources_hash(kernel):
        return None, f"stale: captured at {commit}, the kernel's sources changed since"
    return nbytes, f"ncu capture at {commit}"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return ws, rank


def _oracle_sample_seconds(name, rows, device_inputs=None, seed=0, class_weight=None):
    """Time the float64 oracle on `rows` rows of the workload (host cores)."""
    from oracle import lce_oracle as O

    w = WORKLOADS[name]
    inp = device_inputs if device_inputs is not None else make_workload(name, "cpu")
    if w.kind == "logits":
        z = inp["logits"][:rows].float().cpu().numpy()
        t = inp["target"][:rows].cpu().numpy()
        t0 = time.perf_counter()
        O.ce_from_logits(z, t, w.reduction, -100)
        return time.perf_counter() - t0
    X = inp["X"][:rows].float().cpu().numpy()
    W = inp["W"].float().cpu().numpy()
    b = None if inp["b"] is None else inp["b"].double().cpu().numpy()
    t = inp["target"][:rows].cpu().numpy()
    g = None if inp["grad_out"] is None else inp["grad_out"][:rows].double().cpu().numpy()
    cw = None if class_weight is None else class_weight.double().cpu().numpy()
    t0 = time.perf_counter()
    O.lce_forward_backward(X, W, b, t, w.reduction, -100, g, class_weight=cw)
    return time.perf_counter() - t0


def _workload(args):
    """The named workload, or a copy resized by --rows / --dim / --classes
    (smaller cases of the same kernels, e.g. for profiler captures)."""
    import dataclasses

    w = WORKLOADS[args.workload]
    if not (args.rows or args.dim or args.classes):
        return w
    N = args.rows or w.N
    D = args.dim or w.D
    C = args.classes or w.C
    n_ign = int(round(w.n_ignored * N / w.N))
    return dataclasses.replace(w, name=f"{w.name}[N={N},D={D},C={C}]", N=N, D=D, C=C, n_ignored=n_ign)


def _make_resized(w):
    from linear_cross_entropy_lce_gb300.workloads import make_linear_inputs, make_logits_inputs

    if w.kind == "logits":
        return make_logits_inputs(w.N, w.C, w.dtype, "cuda", w.seed, w.x_std, w.target_dist, w.n_ignored)
    return make_linear_inputs(w.N, w.D, w.C, w.dtype, "cuda", w.seed, w.bias, w.x_std, w.w_std, w.b_std,
                              w.scale_by_sqrt_d, w.target_dist, w.zipf_s, w.n_ignored, w.grad_out_std)


def aggregate_ms(ms, dist=None, device=None):
    """Per-step time of the whole job: the maximum over ranks."""
    if dist is None:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


L2_BYTES = 129 * 2 ** 20  # GB300 L2; the box's own figure is used when a device is present


def input_bytes(w):
    """Bytes of one step's inputs (X and W, or the logits)."""
    esz = 2 if w.dtype in (torch.bfloat16, torch.float16) else 4
    if w.kind == "logits":
        return w.N * w.C * esz
    return (w.N + w.C) * w.D * esz


def flushes_l2(w, l2_bytes=L2_BYTES):
    """Whether the bench flushes L2 between timed steps: when the step's
    inputs are not well larger than L2, they would stay resident across
    steps and time as cache hits."""
    return input_bytes(w) < 2 * l2_bytes


def _config(w, ws, l2_bytes=L2_BYTES):
    """The workload description both arms print."""
    if flushes_l2(w, l2_bytes):
        l2 = ("L2 flushed between timed steps (a %d MB write, outside each step's timing); inputs %.1f MB"
              % (4 * l2_bytes // 2 ** 20, input_bytes(w) / 1e6))
    else:
        l2 = "inputs larger than L2, not flushed (%.2f GB of X and W, or logits)" % (input_bytes(w) / 1e9)
    return {"workload": w.name, "N": w.N, "D": w.D, "C": w.C, "reduction": w.reduction,
            "bias": w.bias, "targets": w.target_dist, "parallelism": "replicas" if ws > 1 else "single",
            "l2": l2}


def run_reference(args):
    ws, rank = _dist()
    if rank != 0:
        return 0
    name = args.workload
    w = WORKLOADS[name]
    rows = args.ref_rows
    inp = make_workload(name, "cuda" if torch.cuda.is_available() else "cpu")
    for _ in range(args.warmup if args.warmup < 1 else 1):
        _oracle_sample_seconds(name, rows, inp)
    times = [_oracle_sample_seconds(name, rows, inp) for _ in range(args.steps)]
    sec = float(np.mean(times))
    value = rows / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w, ws),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
                         "sample": f"{rows} of {w.N} rows per step, full method (loss and all gradients "
                                   f"for those rows) in float64 numpy"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_gpu(args):
    import linear_cross_entropy_lce_gb300 as lce

    ws, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl")
        dist = dist_mod
    lce.load_library()
    name = args.workload
    w = _workload(args)
    inp = make_workload(name, "cuda") if w is WORKLOADS[name] else _make_resized(w)
    if w is not WORKLOADS[name]:
        name = w.name
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peaks = _peaks()
    variant = []  # departures from the named workload (--dtype, --class-weights, --api)
    cw = None
    if args.api == "autograd":
        if w.kind == "logits":
            raise SystemExit("bench: --api autograd applies to the linear workloads")
        variant.append("autograd")

    if w.kind == "logits":
        logits, t = inp["logits"], inp["target"]
        N, V = logits.shape
        nbytes = lce.lce_workspace_size(lce.LCE_OP_CE_FROM_LOGITS, N, 1, V, lce.LCE_F32, lce.LCE_RED_MEAN,
                                        lce.LCE_F32, 0)
        wsbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        status_acc = torch.zeros(1, dtype=torch.int32, device=dev)
        status_word = wsbuf[:4].view(torch.int32)

        def step():
            out = lce.lce_cross_entropy_from_logits(logits, t, w.reduction, -100, workspace=wsbuf)
            status_acc.bitwise_or_(status_word)
            return out

        dt = lce.LCE_F32
        flops = 0.0
    else:
        X, W, b, t, g = inp["X"], inp["W"], inp["b"], inp["target"], inp["grad_out"]
        N, D = X.shape
        C = W.shape[0]
        if args.dtype == "f16":
            if X.dtype != torch.bfloat16:
                raise SystemExit("bench: --dtype f16 applies to the bf16 workloads")
            X, W = X.half(), W.half()
            b = None if b is None else b.half()
            inp = dict(inp, X=X, W=W, b=b)
            variant.append("f16")
        if args.class_weights:
            gen = torch.Generator(device=dev).manual_seed(7)
            cw = torch.rand(C, generator=gen, device=dev) + 0.5
            variant.append("class_weights")
        dt = {torch.bfloat16: lce.LCE_BF16, torch.float16: lce.LCE_F16}.get(X.dtype, lce.LCE_F32)
        red = {"none": 0, "sum": 1, "mean": 2}[w.reduction]
        # reduction none: forward (loss, lse), then the backward from that lse
        # (the page's none op); else one forward+backward call
        bw_op = lce.LCE_OP_BACKWARD if red == 0 else lce.LCE_OP_FORWARD_BACKWARD
        if args.buffer_mib is not None:
            nbytes = lce.lce_workspace_size_for_buffer(bw_op, N, D, C, dt, red, dt, args.buffer_mib << 20)
        else:
            nbytes = lce.lce_workspace_size(bw_op, N, D, C, dt, red, dt, 0)
        if red == 0:
            nbytes = max(nbytes, lce.lce_workspace_size(lce.LCE_OP_FORWARD, N, D, C, dt, red, dt, 0))
        wsbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        status_acc = torch.zeros(1, dtype=torch.int32, device=dev)
        status_word = wsbuf[:4].view(torch.int32)
        plan = lce.plan_of(bw_op, N, D, C, dt, dt, nbytes, want_db=b is not None)
        dX = torch.empty_like(X)
        dW = torch.empty_like(W)
        db = torch.empty_like(b) if b is not None else None
        loss = torch.empty(N if red == 0 else 1, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        lib = lce.load_library()
        import ctypes

        P = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())

        def calls(Xi, Wi, bi, ti, gi, li, dXi, dWi, dbi, mark=None):
            st = ctypes.c_void_p(stream.cuda_stream)
            if red == 0:
                if cw is None:
                    e = lib.lce_forward(P(Xi), P(Wi), P(bi), P(ti), N, D, C, dt, 0, red, -100, P(li), P(lse),
                                        P(wsbuf), nbytes, st)
                else:
                    e = lib.lce_forward_ex(P(Xi), P(Wi), P(bi), P(ti), P(cw), None, N, D, C, dt, 0, red, -100,
                                           P(li), P(lse), P(wsbuf), nbytes, st)
                lce._check(e, "fwd")
                status_acc.bitwise_or_(status_word)
                if mark is not None:
                    mark()  # CUDA event between the two parts
                if cw is None:
                    e = lib.lce_backward(P(Xi), P(Wi), P(bi), P(ti), P(lse), N, D, C, dt, 0, red, -100, P(gi),
                                         P(dXi), P(dWi), P(dbi), dt, P(wsbuf), nbytes, st)
                else:
                    e = lib.lce_backward_ex(P(Xi), P(Wi), P(bi), P(ti), P(cw), None, P(lse), N, D, C, dt, 0, red,
                                            -100, P(gi), P(dXi), P(dWi), P(dbi), dt, P(wsbuf), nbytes, st)
                lce._check(e, "bwd")
            elif cw is None:
                lce._check(lib.lce_forward_backward(P(Xi), P(Wi), P(bi), P(ti), N, D, C, dt, 0, red, -100, P(gi),
                                                    P(li), P(dXi), P(dWi), P(dbi), dt, P(wsbuf), nbytes, st),
                           "fwd+bwd")
            else:
                lce._check(lib.lce_forward_backward_ex(P(Xi), P(Wi), P(bi), P(ti), P(cw), None, N, D, C, dt, 0,
                                                       red, -100, P(gi), P(li), P(dXi), P(dWi), P(dbi), dt,
                                                       P(wsbuf), nbytes, st), "fwd+bwd")
            status_acc.bitwise_or_(status_word)

        if args.api == "autograd":
            # the public autograd function: its own workspace (the library's
            # default plan) and gradient buffers from torch's caching
            # allocator; after the timed steps its gradients are compared
            # with the C-ABI call's (a pipeline that gave up would not match)
            from linear_cross_entropy_lce_gb300.autograd import linear_cross_entropy

            leaves = [x.detach().requires_grad_() if x is not None else None for x in (X, W, b)]

            def step(mark=None):
                for p in leaves:
                    if p is not None:
                        p.grad = None
                out = linear_cross_entropy(leaves[0], leaves[1], t, bias=leaves[2], reduction=w.reduction,
                                           ignore_index=-100, class_weight=cw)
                if mark is not None:
                    mark()
                out.backward(None if g is None else g.reshape(out.shape))
                return out
        else:
            def step(mark=None):
                calls(X, W, b, t, g, loss, dX, dW, db, mark)
                return loss

        flops = w.flops_fwd_bwd

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def check_status(where):
        """Every kernel wait in the library is bounded; one that gave up sets a
        bit in the workspace's status word, and a step whose pipeline gave up
        did not do its work. Each call clears the word, so every step ORs it
        into status_acc on the device right after its calls; any bit there
        means the run is not a measurement."""
        torch.cuda.synchronize()
        st = int(status_acc.item())
        status_acc.zero_()
        if st != 0:
            raise SystemExit(f"bench: device status bits {st} after the {where}; the run is not a measurement")

    for _ in range(args.warmup):
        step()
    barrier()
    check_status("warm-up steps")

    # ---- device-timed region
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    launches0 = lce.launch_count()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    part_events = []  # reduction none: (start, between, end) per step
    split_parts = w.kind == "linear" and w.reduction == "none"
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", L2_BYTES) or L2_BYTES
    flush = flushes_l2(w, l2_bytes)
    if flush:
        # inputs that fit in L2: write a buffer of 4x L2 before every step and
        # time each step on its own, so no step starts with its inputs cached
        scrub = torch.empty(4 * l2_bytes, dtype=torch.uint8, device=dev)
        step_events = []
        for _ in range(args.steps):
            scrub.fill_(1)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            step(mark=lambda: ev[1].record(stream)) if split_parts else step()
            ev[2].record(stream)
            step_events.append(ev)
            if split_parts:
                part_events.append(ev)
        barrier()
        per_step = sum(ev[0].elapsed_time(ev[2]) for ev in step_events) / args.steps
        del scrub
    else:
        e0.record(stream)
        for _ in range(args.steps):
            if split_parts:
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                ev[0].record(stream)
                step(mark=lambda: ev[1].record(stream))
                ev[2].record(stream)
                part_events.append(ev)
            else:
                step()
        e1.record(stream)
        barrier()
        per_step = e0.elapsed_time(e1) / args.steps
    check_status("timed steps")
    launches = lce.launch_count() - launches0
    clocks = sampler.stop()
    ms = aggregate_ms(per_step, dist, dev)
    if args.api == "autograd":
        # the autograd function's workspace is its own, so its status word is
        # not visible here: check its gradients against the C-ABI call instead
        step()
        calls(X, W, b, t, g, loss, dX, dW, db)
        barrier()
        check_status("C-ABI comparison call")
        for got, ref, what in ((leaves[0].grad, dX, "dX"), (leaves[1].grad, dW, "dW")):
            err = float((got.float() - ref.float()).abs().max() / ref.float().abs().max().clamp_min(1e-30))
            if not err <= 1e-3:
                raise SystemExit(f"bench: autograd {what} differs from the C-ABI call ({err:.2e}); not a measurement")

    # ---- context for the memory bound: the same step with the plan that
    # keeps every class of every row in the gradient buffer (no
    # recomputation), a few steps, outside the timed region
    whole = None
    if w.kind != "logits" and dist is None and args.api == "abi":
        wbytes = lce.lce_workspace_size_for_buffer(bw_op, N, D, C, dt, red, dt, (1 << 63) - 1)
        if red == 0:
            wbytes = max(wbytes, lce.lce_workspace_size(lce.LCE_OP_FORWARD, N, D, C, dt, red, dt, 0))
        wplan = lce.plan_of(bw_op, N, D, C, dt, dt, wbytes, want_db=b is not None)
        free_b, _ = torch.cuda.mem_get_info(dev)
        if (wplan["Cb"], wplan["Bc"]) != (plan["Cb"], plan["Bc"]) and wbytes + (1 << 30) < free_b:
            main_ws, main_n = wsbuf, nbytes
            wsbuf = torch.empty(wbytes, dtype=torch.uint8, device=dev)
            status_word = wsbuf[:4].view(torch.int32)
            nbytes = wbytes
            for _ in range(3):
                step()
            barrier()
            k = min(args.steps, 10)
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(k):
                step()
            a1.record(stream)
            barrier()
            check_status("whole-buffer steps")
            wms = a0.elapsed_time(a1) / k
            whole = {"ms_per_step": wms, "tflops": flops / (wms / 1e3) / 1e12, "workspace_bytes": int(wbytes),
                     "steps": k, "note": "every class of every row stored in the gradient buffer; not the "
                                         "headline (timed after it, outside the timed region)"}
            del wsbuf
            wsbuf, nbytes = main_ws, main_n
            status_word = wsbuf[:4].view(torch.int32)

    # ---- the same step captured once in a CUDA graph and replayed (the
    # library allocates and synchronizes nothing, so its calls capture):
    # reported for short steps, where launch overhead is visible
    graph_ms = None
    if ms < 5.0 and dist is None and args.api == "abi":
        cap_stream = torch.cuda.Stream()
        cap_stream.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        prev = stream
        stream = cap_stream  # step() launches on `stream`
        with torch.cuda.graph(graph, stream=cap_stream):
            step()
        stream = prev
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(args.steps):
            graph.replay()
        g1.record()
        torch.cuda.synchronize()
        graph_ms = g0.elapsed_time(g1) / args.steps
        del graph

    # ---- per-kernel times: a separate pass with the library's CUDA-event
    # profiler (its events would add to the timed region on small steps)
    prof_steps = min(args.steps, 10)
    lce.profile_reset()
    scrub = torch.empty(4 * l2_bytes, dtype=torch.uint8, device=dev) if flush else None
    for _ in range(prof_steps):
        if scrub is not None:
            scrub.fill_(1)  # outside the profiled launches, which are timed one by one
        lce.profile_enable(True)
        step()
        lce.profile_enable(False)
    barrier()
    del scrub
    check_status("profiled steps")
    lce.profile_enable(False)
    prof = lce.profile_summary()
    lce.profile_reset()

    # ---- end to end through the public API with host buffers: every step
    # copies its inputs from pinned host memory and copies its results (the
    # loss and every gradient) back to pinned host memory. Inputs and outputs
    # are double-buffered on the device; inputs go in on one copy stream and
    # results come out on another, so step k+1's input copy and step k-1's
    # result copy overlap step k's kernels, as a training input pipeline
    # and an optimizer on the host would.
    if w.kind != "logits":
        in_sets = [[X, W, t, b, g]]
        in_sets.append([None if x is None else torch.empty_like(x) for x in in_sets[0]])
        out_sets = [[loss, dX, dW, db]]
        out_sets.append([None if x is None else torch.empty_like(x) for x in out_sets[0]])

        def run_on(i):
            Xi, Wi, ti, bi, gi = in_sets[i]
            if args.api == "autograd":
                # fresh gradient tensors each step: they are handed to the
                # result copy's stream so their memory is not reused early
                lv = [x.detach().requires_grad_() if x is not None else None for x in (Xi, Wi, bi)]
                out = linear_cross_entropy(lv[0], lv[1], ti, bias=lv[2], reduction=w.reduction, ignore_index=-100,
                                           class_weight=cw)
                out.backward(None if gi is None else gi.reshape(out.shape))
                res = [out.detach(), lv[0].grad, lv[1].grad, None if lv[2] is None else lv[2].grad]
                for r in res:
                    if r is not None:
                        r.record_stream(out_stream)
                out_sets[i] = res
                return
            li, dXi, dWi, dbi = out_sets[i]
            calls(Xi, Wi, bi, ti, gi, li, dXi, dWi, dbi)
    else:
        # the gradient replaces the logits: the step's result is the loss and
        # the whole logits buffer
        e2e_loss = [torch.empty(1, dtype=torch.float32, device=dev) for _ in range(2)]
        in_sets = [[logits, t], [torch.empty_like(logits), torch.empty_like(t)]]
        out_sets = [[e2e_loss[0], in_sets[0][0]], [e2e_loss[1], in_sets[1][0]]]

        def run_on(i):
            li, ti = in_sets[i]
            e2e_loss[i].copy_(lce.lce_cross_entropy_from_logits(li, ti, w.reduction, -100,
                                                                workspace=wsbuf).reshape(1))
            status_acc.bitwise_or_(status_word)

    host_in = [None if x is None else x.cpu().pin_memory() for x in in_sets[0]]
    host_out = [None if x is None else torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in out_sets[0]]
    h2d = sum(x.numel() * x.element_size() for x in host_in if x is not None)
    d2h = sum(x.numel() * x.element_size() for x in host_out if x is not None)
    in_stream = torch.cuda.Stream(device=dev)
    out_stream = torch.cuda.Stream(device=dev)
    ready = [torch.cuda.Event(), torch.cuda.Event()]     # inputs of set i on the device
    in_free = [torch.cuda.Event(), torch.cuda.Event()]   # kernels done reading input set i
    done = [torch.cuda.Event(), torch.cuda.Event()]      # results of set i written
    out_free = [torch.cuda.Event(), torch.cuda.Event()]  # results of set i copied to the host
    for e in in_free + out_free:
        e.record(stream)

    def h2d_into(i, after=None):
        with torch.cuda.stream(in_stream):
            in_stream.wait_event(in_free[i])
            if after is not None:
                in_stream.wait_event(after)
            for d, h in zip(in_sets[i], host_in):
                if d is not None:
                    d.copy_(h, non_blocking=True)
            ready[i].record(in_stream)

    def d2h_from(i):
        with torch.cuda.stream(out_stream):
            out_stream.wait_event(done[i])
            for d, h in zip(out_sets[i], host_out):
                if d is not None:
                    h.copy_(d, non_blocking=True)
            out_free[i].record(out_stream)

    def e2e_steps(k_steps, start_ev):
        h2d_into(0, start_ev)
        for k in range(k_steps):
            i = k % 2
            if k + 1 < k_steps:
                h2d_into(1 - i)
            stream.wait_event(ready[i])
            stream.wait_event(out_free[i])  # results of step k - 2 have left this set
            run_on(i)
            in_free[i].record(stream)
            done[i].record(stream)
            d2h_from(i)
        stream.wait_event(out_free[(k_steps - 1) % 2])  # the last results are on the host
        stream.wait_event(out_free[k_steps % 2])

    s0 = torch.cuda.Event()
    s0.record(stream)
    e2e_steps(2, s0)  # warm-up
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    e2e_steps(args.steps, f0)
    f1.record(stream)
    barrier()
    check_status("end-to-end steps")
    ems = aggregate_ms(f0.elapsed_time(f1) / args.steps, dist, dev)
    e2e = {"value": ws * N / (ems / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "ms_per_step": ems,
           "pipelined": "inputs and results double-buffered; host-to-device and device-to-host copies on "
                        "two more streams, overlapping the neighbouring steps' kernels"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel (the one with the most device time)
    roofline = None
    if prof:
        dominant = max(prof, key=lambda k: prof[k][1])
        n_l, tot_ms, work = prof[dominant]
        avg_s = tot_ms / n_l / 1e3
        per_launch = work / n_l
        # captures are of the named workloads as given: a variant has none
        traffic, traffic_note = measured_traffic("+".join([name] + variant), dominant)
        common = {"traffic": traffic, "traffic_note": traffic_note, "kernel": dominant,
                  "launches_per_step": n_l / prof_steps}
        if dominant.startswith("gemm_") and (dominant.endswith("_tc") or dominant.endswith("_3xtf32")):
            # bf16 / fp16 contractions against the measured cuBLAS bf16 peak;
            # the fp32 product as three TF32 tensor-core products against the
            # TF32 peak / 3, TF32 peak = measured bf16 x the nominal dense
            # TF32 / bf16 ratio (1.1 / 2.25: no measured TF32 peak exists)
            ratio = 1.0 if dominant.endswith("_tc") else (1.1 / 2.25) / 3.0
            achieved = per_launch / avg_s / 1e12
            peak = peaks["bf16_tflops"] * ratio
            peak_s = peaks["bf16_tflops_sustained"] * ratio
            how = "" if ratio == 1.0 else " x 1.1/2.25 (nominal TF32/bf16) / 3 (TF32 products per fp32 product)"
            roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                        "frac": achieved / peak, "peak_sustained": peak_s, "frac_sustained": achieved / peak_s,
                        "peak_source": f"{peaks['source']} bf16_tflops (burst){how}; frac_sustained uses "
                                       f"bf16_tflops_sustained{how}",
                        "algorithmic_flops_per_launch": per_launch, **common}
        elif dominant.startswith("gemm_"):
            # exact fp32 FMA on the CUDA cores: SMs x 128 FP32 lanes x 2 flop x max SM clock
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            peak = sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
            achieved = per_launch / avg_s / 1e12
            roofline = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                        "frac": achieved / peak,
                        "peak_source": f"derived: {sms} SMs x 128 FP32 FMA lanes x 2 flop x "
                                       f"{peaks['sm_max_mhz']:.0f} MHz",
                        "algorithmic_flops_per_launch": per_launch, **common}
        else:
            achieved = per_launch / avg_s / 1e9
            roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"] + " hbm_gbs (copy)",
                        "algorithmic_bytes_per_launch": per_launch, **common}

    # ---- CPU baseline: the oracle on a bounded sample, rank 0, N=1 only
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        rows = args.cpu_rows
        sec = _oracle_sample_seconds(args.workload, rows, inp, class_weight=cw)
        cpu = {"value": rows / sec, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
               "sample": f"{rows} of {w.N} rows, full method (loss and all gradients for those rows) in "
                         f"float64 numpy, {sec:.1f} s"}

    tokens_per_s = ws * w.N / (ms / 1e3)
    cfg = _config(w, ws, l2_bytes)
    cfg["workspace_bytes"] = int(nbytes)
    if variant:
        cfg["variant"] = {"input_dtype": "f16" if "f16" in variant else None,
                          "class_weights": "uniform [0.5, 1.5), seed 7" if cw is not None else None,
                          "api": "autograd: linear_cross_entropy(...).backward()" if args.api == "autograd"
                                 else "C ABI"}
    executed = None
    if w.kind != "logits":
        esz = X.element_size()
        cfg["gradient_buffer"] = {
            "rows": plan["Bc"], "classes": plan["Cb"], "bytes": plan["Bc"] * plan["Cb"] * esz,
            "stored_classes": min(plan["Cs"], w.C), "recomputed_class_chunks": plan["nvc"],
            "batch_chunks": plan["nchunks"],
            "whole_logits_bytes": w.N * w.C * esz,
            "budget": f"{args.buffer_mib} MiB (--buffer-mib)" if args.buffer_mib is not None
                      else "library default (1 GiB)"}
        # tensor-core work actually run: the algorithmic 6NDC (8NDC for none),
        # plus the logits of every class recomputed after the forward sweep
        recomputed = max(0, w.C - min(plan["Cs"], w.C)) if red != 0 else 0
        executed = flops + 2.0 * w.N * w.D * recomputed
    line = {
        "metric": METRIC,
        "value": tokens_per_s,
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {lce.LCE_BF16: "bf16", lce.LCE_F16: "f16"}.get(dt, "f32"),
        "data": "synthetic",
        "config": cfg,
        "gpu_launches": launches,
        "clocks": clocks,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "kernels_ms_per_step": {k: v[1] / prof_steps for k, v in sorted(prof.items(), key=lambda kv: -kv[1][1])},
        "kernels_launches_per_step": {k: v[0] / prof_steps for k, v in prof.items()},
    }
    if graph_ms is not None:
        line["graph_replay_ms_per_step"] = graph_ms
    if whole is not None:
        line["whole_buffer_plan"] = whole
    if part_events:
        fwd_ms = sum(ev[0].elapsed_time(ev[1]) for ev in part_events) / len(part_events)
        fb_ms = sum(ev[1].elapsed_time(ev[2]) for ev in part_events) / len(part_events)
        ndc2 = 2.0 * w.N * w.D * w.C
        line["parts"] = {"forward_ms": fwd_ms, "forward_tflops": ndc2 / (fwd_ms / 1e3) / 1e12,
                         "backward_ms": fb_ms, "backward_tflops": 3 * ndc2 / (fb_ms / 1e3) / 1e12}
    if executed is not None:
        line["executed_tflops"] = executed * ws / (ms / 1e3) / 1e12
    if flops:
        line["tflops"] = flops * ws / (ms / 1e3) / 1e12
        line["pct_bf16_peak"] = 100.0 * line["tflops"] / ws / peaks["bf16_tflops"]
        line["pct_bf16_peak_sustained"] = 100.0 * line["tflops"] / ws / peaks["bf16_tflops_sustained"]
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="bf16_llm_head", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--ref-rows", type=int, default=32, help="rows per step of the --impl reference arm")
    ap.add_argument("--cpu-rows", type=int, default=256, help="rows of the oracle sample in cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", type=int, default=0, help="override N (profiling a smaller case)")
    ap.add_argument("--dim", type=int, default=0, help="override D")
    ap.add_argument("--classes", type=int, default=0, help="override C (or V)")
    ap.add_argument("--print-source-hashes", action="store_true",
                    help="print the source hash of every kernel in KERNEL_SOURCES and exit")
    ap.add_argument("--buffer-mib", type=int, default=None,
                    help="gradient-buffer budget of the workspace plan (default: the library's 1 GiB)")
    ap.add_argument("--dtype", default="input", choices=["input", "f16"],
                    help="f16: a bf16 workload's X, W and bias in fp16 instead")
    ap.add_argument("--class-weights", action="store_true",
                    help="per-class cross-entropy weights, uniform in [0.5, 1.5) (seed 7)")
    ap.add_argument("--api", default="abi", choices=["abi", "autograd"],
                    help="autograd: the step is linear_cross_entropy(...).backward() on the same inputs")
    args = ap.parse_args()
    if args.print_source_hashes:
        print(json.dumps({k: kernel_sources_hash(k) for k in KERNEL_SOURCES}))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
