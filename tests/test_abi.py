"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks return their status codes without touching a GPU."""

import ctypes
import os
import re

import pytest

import linear_cross_entropy_lce_gb300 as lce
from linear_cross_entropy_lce_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return lce.load_library()


def _declared_symbols():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"LCE_API\s+[\w\s\*]+?\b(lce_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert len(names) >= 14
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(12):
        s = lce.status_string(code)
        assert s and s != "unknown status"
    assert lce.status_string(99) == "unknown status"


def test_workspace_size(lib):
    ws = lce.lce_workspace_size
    a = ws(lce.LCE_OP_FORWARD_BACKWARD, 8192, 4096, 128256, lce.LCE_BF16, lce.LCE_RED_MEAN, lce.LCE_BF16)
    # the default plan: a 1 GiB gradient buffer (half the classes of all
    # rows), the fp32 [N, D] dX accumulator and small per-row arrays
    assert 1 << 30 <= a < (1 << 30) + 8192 * 4096 * 4 + (64 << 20)
    # every class stored: the whole [8192, 128256] bf16 buffer
    full = ws(lce.LCE_OP_FORWARD_BACKWARD, 8192, 4096, 128256, lce.LCE_BF16, lce.LCE_RED_MEAN, lce.LCE_BF16, 8192)
    assert 8192 * 128256 * 2 <= full < 8192 * 128256 * 2 * 1.05
    # batch chunks with every class: 8 chunks need the fp32 [C, D] dW accumulator
    eight = ws(lce.LCE_OP_FORWARD_BACKWARD, 8192, 4096, 128256, lce.LCE_BF16, lce.LCE_RED_MEAN,
               lce.LCE_BF16, 1024)
    assert eight > a and eight >= 128256 * 4096 * 4
    # many rows, narrow head: chunks bound the memory
    big = ws(lce.LCE_OP_FORWARD_BACKWARD, 65536, 1024, 32000, lce.LCE_BF16, lce.LCE_RED_MEAN, lce.LCE_BF16, 65536)
    small = ws(lce.LCE_OP_FORWARD_BACKWARD, 65536, 1024, 32000, lce.LCE_BF16, lce.LCE_RED_MEAN,
               lce.LCE_BF16, 1024)
    assert small < big / 10
    fwd = ws(lce.LCE_OP_FORWARD, 8192, 4096, 128256, lce.LCE_BF16, lce.LCE_RED_MEAN, lce.LCE_BF16)
    assert fwd < 100 << 20
    assert ws(lce.LCE_OP_CE_FROM_LOGITS, 16384, 1, 131072, lce.LCE_F32, lce.LCE_RED_MEAN, lce.LCE_F32) > 0
    # invalid arguments give 0
    assert ws(lce.LCE_OP_FORWARD, -1, 4, 4, lce.LCE_F32, 0, 0) == 0
    assert ws(lce.LCE_OP_FORWARD, 4, 4, 4, 7, 0, 0) == 0
    assert ws(lce.LCE_OP_FORWARD, 4, 4, 4, 0, 9, 0) == 0
    assert ws(9, 4, 4, 4, 0, 0, 0) == 0


FAKE = ctypes.c_void_p(4096)  # never dereferenced: every call below fails its host checks


def _fwd(lib, **kw):
    a = dict(X=FAKE, W=FAKE, b=None, t=FAKE, N=16, D=8, C=32, dtype=lce.LCE_F32, acc=lce.LCE_F32,
             red=lce.LCE_RED_MEAN, ign=-100, loss=FAKE, lse=None, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return lib.lce_forward(a["X"], a["W"], a["b"], a["t"], a["N"], a["D"], a["C"], a["dtype"], a["acc"],
                           a["red"], a["ign"], a["loss"], a["lse"], a["ws"], a["wsb"], None)


def _fb(lib, **kw):
    a = dict(X=FAKE, W=FAKE, b=None, t=FAKE, N=16, D=8, C=32, dtype=lce.LCE_F32, acc=lce.LCE_F32,
             red=lce.LCE_RED_MEAN, ign=-100, g=None, loss=FAKE, dX=FAKE, dW=FAKE, db=None,
             gdt=lce.LCE_F32, ws=FAKE, wsb=1 << 20)
    a.update(kw)
    return lib.lce_forward_backward(a["X"], a["W"], a["b"], a["t"], a["N"], a["D"], a["C"], a["dtype"],
                                    a["acc"], a["red"], a["ign"], a["g"], a["loss"], a["dX"], a["dW"],
                                    a["db"], a["gdt"], a["ws"], a["wsb"], None)


def test_host_argument_errors(lib):
    assert _fwd(lib, X=None) == 1  # LCE_ERR_NULL
    assert _fwd(lib, t=None) == 1
    assert _fwd(lib, loss=None) == 1
    assert _fwd(lib, N=-1) == 2  # LCE_ERR_SHAPE
    assert _fwd(lib, D=0) == 2
    assert _fwd(lib, C=0) == 2
    assert _fwd(lib, dtype=5) == 3  # LCE_ERR_DTYPE
    assert _fwd(lib, acc=lce.LCE_BF16) == 3
    assert _fwd(lib, red=3) == 4  # LCE_ERR_REDUCTION
    assert _fwd(lib, ws=None) == 6  # LCE_ERR_WORKSPACE
    assert _fwd(lib, wsb=64) == 6
    assert _fwd(lib, ws=ctypes.c_void_p(4100)) == 9  # LCE_ERR_ALIGN (workspace)
    assert _fwd(lib, dtype=lce.LCE_BF16, D=12) == 9  # bf16 needs D % 8 == 0
    assert _fwd(lib, dtype=lce.LCE_BF16, X=ctypes.c_void_p(4098)) == 9
    assert _fb(lib, red=lce.LCE_RED_NONE, g=None) == 5  # LCE_ERR_GRAD_OUT
    assert _fb(lib, gdt=4) == 3
    assert _fb(lib, dtype=lce.LCE_BF16, dX=ctypes.c_void_p(4098)) == 9
    ce = lib.lce_cross_entropy_from_logits
    assert ce(None, FAKE, 4, 8, lce.LCE_F32, lce.LCE_RED_MEAN, -100, None, FAKE, FAKE, 1 << 20, None) == 1
    assert ce(FAKE, FAKE, 4, 0, lce.LCE_F32, lce.LCE_RED_MEAN, -100, None, FAKE, FAKE, 1 << 20, None) == 2
    assert ce(FAKE, FAKE, 4, 8, 3, lce.LCE_RED_MEAN, -100, None, FAKE, FAKE, 1 << 20, None) == 3
    assert ce(FAKE, FAKE, 4, 8, lce.LCE_F32, 5, -100, None, FAKE, FAKE, 1 << 20, None) == 4
    assert ce(FAKE, FAKE, 4, 8, lce.LCE_F32, lce.LCE_RED_NONE, -100, None, FAKE, FAKE, 1 << 20, None) == 5
    assert ce(FAKE, FAKE, 4, 8, lce.LCE_F32, lce.LCE_RED_MEAN, -100, None, FAKE, FAKE, 16, None) == 6
    assert lib.lce_read_device_status(None, None) == 1
    assert lib.lce_test_gemm_bf16(FAKE, FAKE, FAKE, 8, 8, 12, 0, 0, 0, None, None) == 9
    assert lib.lce_test_gemm_bf16(None, FAKE, FAKE, 8, 8, 8, 0, 0, 1, None, None) == 1
    ud = lib.lce_test_gemm_bf16_unmet_dependency
    assert ud(FAKE, FAKE, FAKE, 8, 8, 8, None, FAKE, None) == 1
    assert ud(FAKE, FAKE, FAKE, 0, 8, 8, FAKE, FAKE, None) == 2
    assert ud(FAKE, FAKE, FAKE, 8, 8, 12, FAKE, FAKE, None) == 9
    tx = lib.lce_test_gemm_tf32x3
    assert tx(FAKE, FAKE, FAKE, 8, 8, 8, 0, 0, 1, None, 1 << 20, None, None) == 1
    assert tx(FAKE, FAKE, FAKE, 0, 8, 8, 0, 0, 1, FAKE, 1 << 20, None, None) == 2
    assert tx(FAKE, FAKE, FAKE, 8, 8, 8, 0, 0, 1, ctypes.c_void_p(4100), 1 << 20, None, None) == 9
    assert tx(FAKE, FAKE, FAKE, 8, 8, 8, 0, 0, 1, FAKE, 1000, None, None) == 6


def test_profile_api_without_launches(lib):
    lce.profile_reset()
    assert lce.profile_summary() == {}
    assert lib.lce_num_kernel_ids() >= 10
    assert lib.lce_kernel_name(0) == b"prep"
