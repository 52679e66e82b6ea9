"""Host-side planning of the loss calls, on the CPU through the C ABI's
host-only test entry points: the row slabs of the CTA-pair backward, and
the workspace plan (batch chunk, region offsets) at sizes far beyond what
the GPU tests run. Nothing here touches a GPU."""

import ctypes

import pytest

import linear_cross_entropy_lce_gb300 as lce
from linear_cross_entropy_lce_gb300 import _build

NF = 28  # LCE_TEST_PLAN_FIELDS
I64 = ctypes.c_int64


@pytest.fixture(scope="module")
def lib():
    _build.build()
    L = lce.load_library()
    L.lce_test_row_slabs.argtypes = [I64, ctypes.POINTER(I64)]
    L.lce_test_row_slabs.restype = ctypes.c_int
    L.lce_test_plan.argtypes = [ctypes.c_int, I64, I64, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(I64), ctypes.c_int]
    L.lce_test_plan.restype = ctypes.c_int
    L.lce_workspace_size.argtypes = [ctypes.c_int, I64, I64, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int, I64]
    L.lce_workspace_size.restype = ctypes.c_size_t
    return L


def _slabs(lib, rows):
    off = (I64 * 5)()
    n = lib.lce_test_row_slabs(rows, off)
    return n, list(off)


@pytest.mark.parametrize("rows", [1024, 1025, 1100, 1229, 1500, 1638, 2047, 2048, 3000, 4096, 8192, 8193, 16384,
                                  65536, 1 << 20])
def test_row_slabs_cover_the_chunk(lib, rows):
    n, off = _slabs(lib, rows)
    assert 1 <= n <= 4
    assert off[0] == 0 and off[n] == rows
    sizes = [off[k + 1] - off[k] for k in range(n)]
    assert all(s > 0 for s in sizes)
    # every slab but the last starts and ends on a 256-row boundary (the
    # CTA-pair tile height), so only the last one has a ragged tail
    assert all(off[k] % 256 == 0 for k in range(n))
    assert sizes == sorted(sizes)
    if rows >= 8192:
        # four strictly growing slabs near 4 : 7 : 9 : 12 of the rows
        assert n == 4
        assert all(a < b for a, b in zip(sizes, sizes[1:]))
        for s, wgt in zip(sizes, (4, 7, 9, 12)):
            assert abs(s / rows - wgt / 32) < 256 / rows + 1e-9


def test_row_slabs_never_shrink(lib):
    """Each slab's side job runs beside the next slab's GEMM, so no slab may
    be larger than the one after it, at any row count the slabbed path takes
    (every count from 1024 to 8192, then a stride beyond)."""
    for rows in list(range(1024, 8193)) + list(range(8193, 70000, 97)):
        n, off = _slabs(lib, rows)
        sizes = [off[k + 1] - off[k] for k in range(n)]
        assert n >= 2 and sizes == sorted(sizes) and off[n] == rows, (rows, sizes)


def test_row_slabs_arguments(lib):
    assert lib.lce_test_row_slabs(-1, (I64 * 5)()) == -1
    assert lib.lce_test_row_slabs(100, None) == -1
    n, off = _slabs(lib, 0)
    assert n == 0 and off[0] == 0


def _plan(lib, op, N, D, C, dtype, grad_dtype, ws, want=(1, 1, 1)):
    out = (I64 * NF)()
    r = lib.lce_test_plan(op, N, D, C, dtype, grad_dtype, *want, ws, out, NF)
    return r, list(out)


def _ws(lib, op, N, D, C, dtype, grad_dtype, chunk_rows=0):
    return lib.lce_workspace_size(op, N, D, C, dtype, lce.LCE_RED_MEAN, grad_dtype, chunk_rows)


SHAPES = [
    # (N, D, C, dtype): the five workloads' shapes and ragged / extreme ones
    (64, 32, 512, lce.LCE_F32),
    (2048, 512, 8192, lce.LCE_F32),
    (8192, 4096, 128256, lce.LCE_BF16),
    (16384, 4096, 131072, lce.LCE_BF16),
    (777, 136, 3001, lce.LCE_F16),
    (1, 8, 1, lce.LCE_BF16),
    (1 << 20, 1024, 32000, lce.LCE_BF16),
    (300000, 64, 262144, lce.LCE_F32),
]


@pytest.mark.parametrize("N,D,C,dtype", SHAPES)
@pytest.mark.parametrize("op", [lce.LCE_OP_FORWARD, lce.LCE_OP_FORWARD_BACKWARD])
def test_plan_regions_fit_and_do_not_overlap(lib, op, N, D, C, dtype):
    for grad_dtype in (dtype, lce.LCE_F32):
        ws = _ws(lib, op, N, D, C, dtype, grad_dtype)
        assert ws > 0
        r, v = _plan(lib, op, N, D, C, dtype, grad_dtype, ws)
        assert r == NF
        Bc, nchunks, total, C_pad, nseg = v[:5]
        offs = v[5:]
        # the plan the calls choose for the queried size is the one it was sized for
        assert total <= ws
        assert 1 <= Bc <= N and nchunks == -(-N // Bc)
        assert Bc == N or (Bc % 128 == 0 and Bc & (Bc - 1) == 0)
        assert C_pad >= C and C_pad % 128 == 0 and nseg >= 1
        # regions in order, 256-byte aligned, inside the total
        assert all(o % 256 == 0 for o in offs)
        assert offs == sorted(offs) and offs[0] > 0 and offs[-1] <= total
        # the regions the pages' method needs have room for their arrays
        off_cnt, off_loss, off_zt, off_tcol, off_gt, off_partial, off_L, off_dw = offs[:8]
        assert off_zt - off_loss >= 4 * N               # per-row losses, fp32
        assert off_L - off_partial >= 8 * nseg * Bc     # (max, sum-exp) pairs of a chunk
        if op == lce.LCE_OP_FORWARD_BACKWARD:
            esz = 4 if dtype == lce.LCE_F32 else 2
            assert off_dw - off_L >= Bc * C_pad * esz  # the chunk's P~ / G buffer
        else:
            assert off_dw == off_L                      # no P~ buffer in the forward


def test_plan_smaller_workspace_gives_smaller_chunks(lib):
    op, N, D, C, dt = lce.LCE_OP_FORWARD_BACKWARD, 65536, 1024, 32000, lce.LCE_BF16
    full = _ws(lib, op, N, D, C, dt, dt)
    r, v = _plan(lib, op, N, D, C, dt, dt, full)
    prev_bc = v[0]
    for chunk in (8192, 2048, 512, 128):
        ws = _ws(lib, op, N, D, C, dt, dt, chunk)
        r, v = _plan(lib, op, N, D, C, dt, dt, ws)
        assert r == NF and v[2] <= ws and v[0] <= min(prev_bc, chunk)
        prev_bc = v[0]
    # below the smallest chunk's plan nothing fits
    r, _ = _plan(lib, op, N, D, C, dt, dt, 4096)
    assert r == 0


def test_plan_arguments(lib):
    out = (I64 * NF)()
    assert lib.lce_test_plan(7, 10, 8, 8, lce.LCE_BF16, lce.LCE_BF16, 1, 1, 1, 1 << 30, out, NF) == -1
    assert lib.lce_test_plan(lce.LCE_OP_FORWARD, 10, 0, 8, lce.LCE_BF16, lce.LCE_BF16, 1, 1, 1, 1 << 30,
                             out, NF) == -1
    assert lib.lce_test_plan(lce.LCE_OP_FORWARD, 10, 8, 8, lce.LCE_BF16, lce.LCE_BF16, 1, 1, 1, 1 << 30,
                             out, NF - 1) == -1
