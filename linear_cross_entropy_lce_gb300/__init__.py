"""Fused linear + cross-entropy loss for GB300 (sm_103a).

A thin ctypes binding over liblce.so (see include/lce.h). Every step of the
computation runs in the library's CUDA kernels; this module only marshals
arguments: it allocates outputs and the workspace with torch, takes the data
pointers and the current CUDA stream, and raises ``LceError`` on a nonzero
status. There is no CPU fallback: without the built library every call
raises.

Functions (same names as the C ABI):
  lce_workspace_size(op, N, D, C, dtype, reduction, grad_dtype, chunk_rows=0)
  lce_forward(X, W, b, target, reduction="mean", ignore_index=-100, ...)
  lce_forward_backward(X, W, b, target, reduction="mean", ignore_index=-100,
                       grad_out=None, ...)
  lce_backward(X, W, b, target, lse, reduction="mean", ...)
  lce_workspace_size_for_buffer(op, N, D, C, dtype, reduction, grad_dtype, buffer_bytes)
  lce_cross_entropy_from_logits(logits, target, reduction="mean",
                                ignore_index=-100, grad_out=None, ...)
  lce_status_string(code), lce_read_device_status(workspace)
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblce.so")

LCE_F32, LCE_BF16, LCE_F16 = 0, 1, 2
LCE_RED_NONE, LCE_RED_SUM, LCE_RED_MEAN = 0, 1, 2
LCE_OP_FORWARD, LCE_OP_FORWARD_BACKWARD, LCE_OP_CE_FROM_LOGITS, LCE_OP_BACKWARD = 0, 1, 2, 3
LCE_NOALLOC_MAX_ROWS = 1 << 20
LCE_ERR_WORKSPACE = 6
STATUS = {
    0: "LCE_OK", 1: "LCE_ERR_NULL", 2: "LCE_ERR_SHAPE", 3: "LCE_ERR_DTYPE", 4: "LCE_ERR_REDUCTION",
    5: "LCE_ERR_GRAD_OUT", 6: "LCE_ERR_WORKSPACE", 7: "LCE_ERR_CUDA", 8: "LCE_ERR_TARGET_RANGE",
    9: "LCE_ERR_ALIGN", 10: "LCE_ERR_TIMEOUT", 11: "LCE_ERR_DEVICE",
}
_REDUCTION = {"none": LCE_RED_NONE, "sum": LCE_RED_SUM, "mean": LCE_RED_MEAN}
_DTYPE = {torch.float32: LCE_F32, torch.bfloat16: LCE_BF16, torch.float16: LCE_F16}
_TORCH_DTYPE = {LCE_F32: torch.float32, LCE_BF16: torch.bfloat16, LCE_F16: torch.float16}

_lib = None

c_void_p, c_int, c_int64, c_size_t, c_double = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                                 ctypes.c_size_t, ctypes.c_double)

_SIGNATURES = {
    "lce_workspace_size": (c_size_t, [c_int, c_int64, c_int64, c_int64, c_int, c_int, c_int, c_int64]),
    "lce_workspace_size_for_buffer": (c_size_t, [c_int, c_int64, c_int64, c_int64, c_int, c_int, c_int, c_size_t]),
    "lce_aspect_ratio_chunk_rows": (c_int64, [c_int64, c_int64, c_int64, c_int64]),
    "lce_backward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int,
                             c_int, c_int, c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p,
                             c_size_t, c_void_p]),
    "lce_backward_ex": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64,
                                c_int64, c_int64, c_int, c_int, c_int, c_int64, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_int, c_void_p, c_size_t, c_void_p]),
    "lce_forward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int, c_int,
                            c_int, c_int64, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "lce_forward_backward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int,
                                     c_int, c_int, c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_int, c_void_p, c_size_t, c_void_p]),
    "lce_cross_entropy_from_logits": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_int, c_int, c_int64,
                                              c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "lce_forward_ex": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64,
                               c_int, c_int, c_int, c_int64, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "lce_forward_backward_ex": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64,
                                        c_int64, c_int, c_int, c_int, c_int64, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_int, c_void_p, c_size_t, c_void_p]),
    "lce_cross_entropy_from_logits_ex": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int,
                                                 c_int, c_int64, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "lce_mean_denominator": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_int64, c_void_p, c_void_p, c_size_t,
                                     c_void_p]),
    "lce_cross_entropy_from_logits_noalloc": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_int, c_int,
                                                      c_int64, c_void_p, c_void_p, c_void_p, c_void_p]),
    "lce_scale_gradients": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int64, c_int, c_void_p,
                                    c_void_p]),
    "lce_status_string": (ctypes.c_char_p, [c_int]),
    "lce_read_device_status": (c_int, [c_void_p, c_void_p]),
    "lce_launch_count": (c_int64, []),
    "lce_profile_enable": (c_int, [c_int]),
    "lce_profile_reset": (c_int, []),
    "lce_profile_query": (c_int, [c_int, ctypes.POINTER(c_int64), ctypes.POINTER(c_double),
                                  ctypes.POINTER(c_double)]),
    "lce_kernel_name": (ctypes.c_char_p, [c_int]),
    "lce_num_kernel_ids": (c_int, []),
    "lce_test_gemm_bf16": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int, c_int,
                                   c_int, c_void_p, c_void_p]),
    "lce_test_gemm_f32": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int, c_int,
                                  c_void_p]),
    "lce_test_gemm_bf16_unmet_dependency": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64,
                                                    c_void_p, c_void_p, c_void_p]),
    "lce_test_gemm_tf32x3": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int, c_int,
                                     c_int, c_void_p, c_size_t, c_void_p, c_void_p]),
}


class LceError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({status_string(code)})")


def load_library(path: Optional[str] = None):
    """Load liblce.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -m linear_cross_entropy_lce_gb300._build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    if _lib is None:
        return STATUS.get(code, "unknown")
    return _lib.lce_status_string(code).decode()


lce_status_string = status_string


def _check(code: int, where: str):
    if code != 0:
        raise LceError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPE:
        raise TypeError(f"unsupported dtype {t.dtype}: use float32, bfloat16 or float16")
    return _DTYPE[t.dtype]


def lce_workspace_size(op: int, N: int, D: int, C: int, dtype: int, reduction: int, grad_dtype: int,
                       chunk_rows: int = 0) -> int:
    lib = load_library()
    return int(lib.lce_workspace_size(op, N, D, C, dtype, reduction, grad_dtype, chunk_rows))


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]):
    if workspace is not None:
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _class_weight(cw, C, device):
    if cw is None:
        return None
    cw = torch.as_tensor(cw, dtype=torch.float32, device=device).reshape(-1).contiguous()
    if cw.numel() != C:
        raise ValueError(f"class_weight must have {C} entries")
    return cw


def _denom(d, device):
    """A given mean denominator as a device fp32 scalar tensor (or None)."""
    if d is None:
        return None
    return torch.as_tensor(d, dtype=torch.float32, device=device).reshape(-1)[:1].contiguous()


def lce_mean_denominator(target, C, ignore_index=-100, class_weight=None, stream=None):
    """Device fp32 [1]: the mean's denominator of these rows (valid-row count,
    or the sum of their class weights). Data-parallel shards sum it."""
    lib = load_library()
    if target.dtype != torch.int64 or not target.is_contiguous():
        raise TypeError("target must be a contiguous int64 tensor")
    dev = target.device
    out = torch.empty(1, dtype=torch.float32, device=dev)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    cw = _class_weight(class_weight, C, dev)
    _check(lib.lce_mean_denominator(_ptr(target), _ptr(cw), target.numel(), C, ignore_index, _ptr(out), _ptr(ws), 256,
                                    _stream(stream)), "lce_mean_denominator")
    return out


def _check_inputs(X, W, b, target):
    if X.dim() != 2 or W.dim() != 2 or X.shape[1] != W.shape[1]:
        raise ValueError("expected X [N, D] and W [C, D]")
    if X.dtype != W.dtype or (b is not None and b.dtype != X.dtype):
        raise TypeError("X, W and b must share one dtype")
    if target.dtype != torch.int64:
        raise TypeError("target must be int64")
    if b is not None and b.shape != (W.shape[0],):
        raise ValueError(f"expected bias shape ({W.shape[0]},), got {tuple(b.shape)}")
    for t in (X, W, b, target):
        if t is not None and not t.is_contiguous():
            raise ValueError("inputs must be contiguous")


def lce_forward(X, W, b, target, reduction="mean", ignore_index=-100, want_lse=False,
                workspace=None, stream=None, class_weight=None, denominator=None):
    """Loss (fp32 scalar, or [N] for 'none') and optionally lse [N].
    class_weight: optional per-class weights [C] (fp32). denominator:
    optional device fp32 scalar replacing the mean's denominator (a
    data-parallel shard passes the whole batch's; see lce.h)."""
    lib = load_library()
    _check_inputs(X, W, b, target)
    N, D = X.shape
    C = W.shape[0]
    red = _REDUCTION[reduction]
    dt = _dtype_code(X)
    dev = X.device
    loss = torch.empty(N if red == LCE_RED_NONE else 1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev) if want_lse else None
    nbytes = lib.lce_workspace_size(LCE_OP_FORWARD, N, D, C, dt, red, LCE_F32, 0)
    ws = _workspace(nbytes, dev, workspace)
    cw = _class_weight(class_weight, C, dev)
    _check(lib.lce_forward_ex(_ptr(X), _ptr(W), _ptr(b), _ptr(target), _ptr(cw), _ptr(_denom(denominator, dev)), N,
                              D, C, dt, LCE_F32, red,
                              ignore_index, _ptr(loss), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)),
           "lce_forward")
    loss = loss if red == LCE_RED_NONE else loss[0]
    return (loss, lse) if want_lse else loss


def lce_workspace_size_for_buffer(op: int, N: int, D: int, C: int, dtype: int, reduction: int, grad_dtype: int,
                                  buffer_bytes: int) -> int:
    lib = load_library()
    return int(lib.lce_workspace_size_for_buffer(op, N, D, C, dtype, reduction, grad_dtype, buffer_bytes))


def lce_aspect_ratio_chunk_rows(N: int, D: int, C: int, divisor: int = 1) -> int:
    """The page's "aspect_ratio[:divisor]" batch chunk size (see lce.h)."""
    return int(load_library().lce_aspect_ratio_chunk_rows(N, D, C, divisor))


def _grad_ws_bytes(lib, op, N, D, C, dt, red, gdt, chunk_rows, buffer_bytes):
    if buffer_bytes is not None:
        if chunk_rows:
            raise ValueError("give chunk_rows or buffer_bytes, not both")
        return lib.lce_workspace_size_for_buffer(op, N, D, C, dt, red, gdt, buffer_bytes)
    return lib.lce_workspace_size(op, N, D, C, dt, red, gdt, chunk_rows)


def lce_forward_backward(X, W, b, target, reduction="mean", ignore_index=-100, grad_out=None,
                         want_dx=True, want_dw=True, want_db=True, grad_dtype=None, chunk_rows=0,
                         workspace=None, stream=None, class_weight=None, buffer_bytes=None, denominator=None):
    """Loss and (dX, dW, db); a gradient not wanted (or db without bias) is None.

    grad_out: None (= 1) or a scalar / 1-element tensor for sum and mean; a
    float32 [N] tensor for 'none'. The workspace (unless given) is sized for
    the default plan, for batch chunks of chunk_rows rows, or for a gradient
    buffer of at most buffer_bytes (see lce_workspace_size_for_buffer).
    """
    lib = load_library()
    _check_inputs(X, W, b, target)
    N, D = X.shape
    C = W.shape[0]
    red = _REDUCTION[reduction]
    dt = _dtype_code(X)
    gdt = dt if grad_dtype is None else _DTYPE[grad_dtype]
    gtype = _TORCH_DTYPE[gdt]
    dev = X.device
    g = None
    if grad_out is not None:
        g = torch.as_tensor(grad_out, dtype=torch.float32, device=dev).reshape(-1).contiguous()
        if red != LCE_RED_NONE and g.numel() != 1:
            raise ValueError("grad_out must be a scalar for sum / mean")
    loss = torch.empty(N if red == LCE_RED_NONE else 1, dtype=torch.float32, device=dev)
    dX = torch.empty(N, D, dtype=gtype, device=dev) if want_dx else None
    dW = torch.empty(C, D, dtype=gtype, device=dev) if want_dw else None
    db = torch.empty(C, dtype=gtype, device=dev) if (want_db and b is not None) else None
    nbytes = _grad_ws_bytes(lib, LCE_OP_FORWARD_BACKWARD, N, D, C, dt, red, gdt, chunk_rows, buffer_bytes)
    ws = _workspace(nbytes, dev, workspace)
    cw = _class_weight(class_weight, C, dev)
    _check(lib.lce_forward_backward_ex(_ptr(X), _ptr(W), _ptr(b), _ptr(target), _ptr(cw),
                                       _ptr(_denom(denominator, dev)), N, D, C, dt, LCE_F32,
                                       red, ignore_index, _ptr(g), _ptr(loss), _ptr(dX), _ptr(dW), _ptr(db), gdt,
                                       _ptr(ws), ws.numel(), _stream(stream)), "lce_forward_backward")
    return (loss if red == LCE_RED_NONE else loss[0]), dX, dW, db


def lce_backward(X, W, b, target, lse, reduction="mean", ignore_index=-100, grad_out=None,
                 want_dx=True, want_dw=True, want_db=True, grad_dtype=None, chunk_rows=0,
                 workspace=None, stream=None, class_weight=None, buffer_bytes=None, denominator=None):
    """(dX, dW, db) from the row lse [N] (float32) of lce_forward(..., want_lse=True)."""
    lib = load_library()
    _check_inputs(X, W, b, target)
    N, D = X.shape
    C = W.shape[0]
    red = _REDUCTION[reduction]
    dt = _dtype_code(X)
    gdt = dt if grad_dtype is None else _DTYPE[grad_dtype]
    gtype = _TORCH_DTYPE[gdt]
    dev = X.device
    if lse.dtype != torch.float32 or lse.shape != (N,) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [N] tensor")
    g = None
    if grad_out is not None:
        g = torch.as_tensor(grad_out, dtype=torch.float32, device=dev).reshape(-1).contiguous()
        if red != LCE_RED_NONE and g.numel() != 1:
            raise ValueError("grad_out must be a scalar for sum / mean")
    dX = torch.empty(N, D, dtype=gtype, device=dev) if want_dx else None
    dW = torch.empty(C, D, dtype=gtype, device=dev) if want_dw else None
    db = torch.empty(C, dtype=gtype, device=dev) if (want_db and b is not None) else None
    nbytes = _grad_ws_bytes(lib, LCE_OP_BACKWARD, N, D, C, dt, red, gdt, chunk_rows, buffer_bytes)
    ws = _workspace(nbytes, dev, workspace)
    cw = _class_weight(class_weight, C, dev)
    _check(lib.lce_backward_ex(_ptr(X), _ptr(W), _ptr(b), _ptr(target), _ptr(cw), _ptr(_denom(denominator, dev)),
                               _ptr(lse), N, D, C, dt, LCE_F32,
                               red, ignore_index, _ptr(g), _ptr(dX), _ptr(dW), _ptr(db), gdt, _ptr(ws), ws.numel(),
                               _stream(stream)), "lce_backward")
    return dX, dW, db


def lce_cross_entropy_from_logits(logits, target, reduction="mean", ignore_index=-100, grad_out=None,
                                  workspace=None, stream=None, class_weight=None, denominator=None):
    """Loss; the gradient overwrites ``logits`` in place."""
    lib = load_library()
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("expected contiguous logits [N, V]")
    if target.dtype != torch.int64:
        raise TypeError("target must be int64")
    N, V = logits.shape
    red = _REDUCTION[reduction]
    dt = _dtype_code(logits)
    dev = logits.device
    g = None
    if grad_out is not None:
        g = torch.as_tensor(grad_out, dtype=torch.float32, device=dev).reshape(-1).contiguous()
    loss = torch.empty(N if red == LCE_RED_NONE else 1, dtype=torch.float32, device=dev)
    nbytes = lib.lce_workspace_size(LCE_OP_CE_FROM_LOGITS, N, 1, V, dt, red, dt, 0)
    ws = _workspace(nbytes, dev, workspace)
    cw = _class_weight(class_weight, V, dev)
    _check(lib.lce_cross_entropy_from_logits_ex(_ptr(logits), _ptr(target), _ptr(cw), _ptr(_denom(denominator, dev)),
                                                N, V, dt, red, ignore_index,
                                                _ptr(g), _ptr(loss), _ptr(ws), ws.numel(), _stream(stream)),
           "lce_cross_entropy_from_logits")
    return loss if red == LCE_RED_NONE else loss[0]


def lce_scale_gradients(dX, dW, db, grad_out, stream=None):
    """dX, dW, db (any may be None; one dtype) *= grad_out (a device fp32
    scalar tensor), in place; nothing is touched when grad_out == 1."""
    lib = load_library()
    ts = [t for t in (dX, dW, db) if t is not None]
    if not ts:
        return
    gdt = _dtype_code(ts[0])
    for t in ts:
        if _dtype_code(t) != gdt or not t.is_contiguous():
            raise ValueError("gradients must be contiguous and share one dtype")
    g = grad_out.to(torch.float32).reshape(-1)[:1].contiguous()
    n = lambda t: 0 if t is None else t.numel()
    _check(lib.lce_scale_gradients(_ptr(dX), n(dX), _ptr(dW), n(dW), _ptr(db), n(db), gdt, _ptr(g), _stream(stream)),
           "lce_scale_gradients")


def plan_of(op: int, N: int, D: int, C: int, dtype: int, grad_dtype: int, ws_bytes: int, want_dx=True, want_dw=True,
            want_db=True) -> dict:
    """The workspace plan a call makes for ws_bytes (host-only; see
    lce_test_plan in lce_testing.h): rows per batch chunk Bc, chunk count,
    total bytes, gradient-buffer columns Cb, classes stored by the forward
    sweep Cs and recomputed class chunks nvc."""
    lib = load_library()
    fn = lib.lce_test_plan
    fn.argtypes = [c_int, c_int64, c_int64, c_int64, c_int, c_int, c_int, c_int, c_int, c_size_t,
                   ctypes.POINTER(c_int64), c_int]
    fn.restype = c_int
    nf = 28  # LCE_TEST_PLAN_FIELDS
    out = (c_int64 * nf)()
    r = fn(op, N, D, C, dtype, grad_dtype, int(want_dx), int(want_dw), int(want_db), ws_bytes, out, nf)
    if r != nf:
        raise LceError(LCE_ERR_WORKSPACE if r == 0 else 1, "plan_of")
    v = list(out)
    return {"Bc": v[0], "nchunks": v[1], "total": v[2], "C_pad": v[3], "Cb": v[nf - 3], "Cs": v[nf - 2],
            "nvc": v[nf - 1]}


def lce_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    lib = load_library()
    return int(lib.lce_read_device_status(_ptr(workspace), _stream(stream)))


# ---- kernel accounting (benchmark support)

def launch_count() -> int:
    return int(load_library().lce_launch_count())


def profile_enable(on: bool = True):
    load_library().lce_profile_enable(1 if on else 0)


def profile_reset():
    load_library().lce_profile_reset()


def profile_summary() -> dict:
    """{kernel name: (launches, total ms, total algorithmic work)} for the
    recorded launches; work is flop for gemm_* kernels, HBM bytes otherwise."""
    lib = load_library()
    out = {}
    for k in range(lib.lce_num_kernel_ids()):
        n = c_int64(0)
        ms = c_double(0.0)
        work = c_double(0.0)
        _check(lib.lce_profile_query(k, ctypes.byref(n), ctypes.byref(ms), ctypes.byref(work)),
               "lce_profile_query")
        if n.value:
            out[lib.lce_kernel_name(k).decode()] = (int(n.value), float(ms.value), float(work.value))
    return out


# ---- building-block checks (include/lce_testing.h)

def test_gemm_bf16(A, B, M, N, K, a_mn_major, b_mn_major, status=None, cta_pair=False, stream=None):
    """lce_test_gemm_bf16: fp32 [M, N] = A B^T on the tcgen05 engine (layouts as in lce_testing.h)."""
    lib = load_library()
    out = torch.empty(M, N, dtype=torch.float32, device=A.device)
    _check(lib.lce_test_gemm_bf16(_ptr(A), _ptr(B), _ptr(out), M, N, K, int(a_mn_major), int(b_mn_major),
                                  int(cta_pair), _ptr(status), _stream(stream)), "lce_test_gemm_bf16")
    return out


def test_gemm_bf16_unmet_dependency(A, B, M, N, K, counters, status, stream=None):
    """lce_test_gemm_bf16_unmet_dependency: the failure path of the bounded waits (see lce_testing.h)."""
    lib = load_library()
    out = torch.empty(M, N, dtype=torch.float32, device=A.device)
    _check(lib.lce_test_gemm_bf16_unmet_dependency(_ptr(A), _ptr(B), _ptr(out), M, N, K, _ptr(counters),
                                                   _ptr(status), _stream(stream)),
           "lce_test_gemm_bf16_unmet_dependency")
    return out


def test_gemm_tf32x3(A, B, M, N, K, a_mn_major, b_mn_major, k_splits=1, status=None, stream=None):
    """lce_test_gemm_tf32x3: fp32 [M, N] = A B^T as three TF32 products on the tensor cores."""
    lib = load_library()
    out = torch.empty(M, N, dtype=torch.float32, device=A.device)
    def part(rows, cols):  # one hi or lo copy of an operand stored [rows, cols], 256-byte aligned
        return ((rows * ((cols + 3) // 4 * 4) * 4) + 255) // 256 * 256

    ws_bytes = 2 * (part(K, M) if a_mn_major else part(M, K)) + 2 * (part(K, N) if b_mn_major else part(N, K))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=A.device)
    _check(lib.lce_test_gemm_tf32x3(_ptr(A), _ptr(B), _ptr(out), M, N, K, int(a_mn_major), int(b_mn_major),
                                    int(k_splits), _ptr(ws), ws_bytes, _ptr(status), _stream(stream)),
           "lce_test_gemm_tf32x3")
    return out


def test_gemm_f32(A, B, M, N, K, a_mn_major, b_mn_major, stream=None):
    """lce_test_gemm_f32: fp32 [M, N] = A B^T with fp32 FMA on the CUDA cores."""
    lib = load_library()
    out = torch.empty(M, N, dtype=torch.float32, device=A.device)
    _check(lib.lce_test_gemm_f32(_ptr(A), _ptr(B), _ptr(out), M, N, K, int(a_mn_major), int(b_mn_major),
                                 _stream(stream)), "lce_test_gemm_f32")
    return out
