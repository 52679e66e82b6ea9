"""Host-side planning of the loss calls, on the CPU through the C ABI's
host-only test entry points: the row slabs of the CTA-pair backward, and
the workspace plan (batch chunk, region offsets) at sizes far beyond what
the GPU tests run. Nothing here touches a GPU."""

import ctypes
import os

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
    L.lce_workspace_size_for_buffer.argtypes = [ctypes.c_int, I64, I64, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_size_t]
    L.lce_workspace_size_for_buffer.restype = ctypes.c_size_t
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


GIB = 1 << 30


def _esz(dtype):
    return 4 if dtype == lce.LCE_F32 else 2


@pytest.mark.parametrize("N,D,C,dtype", SHAPES)
@pytest.mark.parametrize("op", [lce.LCE_OP_FORWARD, lce.LCE_OP_FORWARD_BACKWARD, lce.LCE_OP_BACKWARD])
def test_plan_regions_fit_and_do_not_overlap(lib, op, N, D, C, dtype):
    for grad_dtype in (dtype, lce.LCE_F32):
        ws = _ws(lib, op, N, D, C, dtype, grad_dtype)
        assert ws > 0
        r, v = _plan(lib, op, N, D, C, dtype, grad_dtype, ws)
        assert r == NF
        Bc, nchunks, total, C_pad, nseg = v[:5]
        offs = v[5:25]
        Cb, Cs, nvc = v[25:28]
        # the plan the calls choose for the queried size is the one it was sized for (or a faster one)
        assert total <= ws
        assert 1 <= Bc <= N and nchunks == -(-N // Bc)
        assert Bc == N or Bc % 128 == 0
        assert C_pad >= C and C_pad % 128 == 0 and nseg >= 1
        # regions in order, 256-byte aligned, inside the total
        assert all(o % 256 == 0 for o in offs)
        assert offs == sorted(offs) and offs[0] > 0 and offs[-1] <= total
        off_cnt, off_loss, off_zt, off_tcol, off_gt, off_partial, off_L, off_dw, off_db = offs[:9]
        off_lse, off_wv, off_dx = offs[12:15]
        backward = op != lce.LCE_OP_FORWARD
        given_lse = op == lce.LCE_OP_BACKWARD and dtype != lce.LCE_F32
        if not given_lse:
            assert off_zt - off_loss >= 4 * N               # per-row losses, fp32
            assert off_L - off_partial >= 8 * nseg * Bc     # (max, sum-exp) pairs of a chunk
        if backward:
            # the gradient buffer, within the default budget
            assert off_dw - off_L >= Bc * Cb * _esz(dtype)
            assert Bc * Cb * _esz(dtype) <= GIB or (dtype == lce.LCE_F32)
            # every class is covered: stored [0, Cs), then nvc chunks of Cb
            assert Cs + nvc * Cb >= C and (nvc == 0 or Cs + (nvc - 1) * Cb < C)
            assert Cs == (0 if given_lse else Cb)
            if nvc:  # recomputed classes keep the rows' lse and weights
                assert off_wv - off_lse >= 4 * Bc and off_dx - off_wv >= 4 * Bc
        else:
            assert off_dw == off_L                      # no P~ buffer in the forward
        if dtype == lce.LCE_F32 and os.environ.get("LCE_F32_SIMT") != "1":
            # 3xTF32: hi / lo of W and of the chunk's X in their own layout,
            # and G's lo part beside the buffer; no transposed copies
            off_wh, off_wl, off_xh, off_xl, off_gl = offs[15:20]
            ldD = -(-D // 4) * 4
            assert off_wl - off_wh >= C * ldD * 4 and off_xh - off_wl >= C * ldD * 4
            assert off_xl - off_xh >= Bc * ldD * 4 and off_gl - off_xl >= Bc * ldD * 4
            if backward:
                assert total - off_gl >= Bc * C_pad * 4


@pytest.mark.parametrize("N,D,C,Bc,Cb,nvc", [
    (8192, 4096, 128256, 8192, 65536, 1),     # the LLM head: half the vocabulary stored, the rest recomputed
    (16384, 4096, 131072, 16384, 32768, 3),   # the large head
    (1 << 20, 1024, 32000, 524288, 1024, 31),  # so many rows that 1024 classes of all rows exceed 1 GiB
    (2048, 512, 8192, 2048, 8192, 0),          # everything fits: nothing recomputed
])
def test_default_plan_bounds_the_gradient_buffer(lib, N, D, C, Bc, Cb, nvc):
    dt = lce.LCE_BF16
    ws = _ws(lib, lce.LCE_OP_FORWARD_BACKWARD, N, D, C, dt, dt)
    r, v = _plan(lib, lce.LCE_OP_FORWARD_BACKWARD, N, D, C, dt, dt, ws)
    assert r == NF
    assert (v[0], v[25], v[27]) == (Bc, Cb, nvc)
    assert v[0] * v[25] * 2 <= GIB
    # no [C, D] fp32 scratch unless the rows are split into batch chunks
    assert (v[13] - v[12] > 0) == (v[1] > 1)
    # lce_workspace_size_for_buffer with 0 is the default; a huge budget stores every class
    assert lib.lce_workspace_size_for_buffer(lce.LCE_OP_FORWARD_BACKWARD, N, D, C, dt, lce.LCE_RED_MEAN, dt, 0) == ws
    big = lib.lce_workspace_size_for_buffer(lce.LCE_OP_FORWARD_BACKWARD, N, D, C, dt, lce.LCE_RED_MEAN, dt,
                                            ctypes.c_size_t(-1).value)
    r, v = _plan(lib, lce.LCE_OP_FORWARD_BACKWARD, N, D, C, dt, dt, big)
    assert v[27] == 0 and v[25] == v[3]


def test_plan_smaller_workspace_recomputes_more(lib):
    """Shrinking the workspace first narrows the stored classes (more of them
    recomputed), then splits the rows; every plan fits what it was given."""
    op, N, D, C, dt = lce.LCE_OP_FORWARD_BACKWARD, 65536, 1024, 32000, lce.LCE_BF16
    prev = None
    for mib in (8192, 2048, 1024, 512, 256, 128, 64):
        ws = lib.lce_workspace_size_for_buffer(op, N, D, C, dt, lce.LCE_RED_MEAN, dt, mib << 20)
        r, v = _plan(lib, op, N, D, C, dt, dt, ws)
        assert r == NF and v[2] <= ws
        Bc, Cb = v[0], v[25]
        if prev is not None:
            assert (Bc, Cb) <= prev or Bc < prev[0]
        prev = (Bc, Cb)
    # below the smallest plan nothing fits
    r, _ = _plan(lib, op, N, D, C, dt, dt, 4096)
    assert r == 0


def test_chunk_rows_plan(lib):
    """chunk_rows sizes batch chunks with every class stored; chunk_rows >= N
    stores the whole [N, C] buffer."""
    op, N, D, C, dt = lce.LCE_OP_FORWARD_BACKWARD, 8192, 4096, 128256, lce.LCE_BF16
    ws = _ws(lib, op, N, D, C, dt, dt, N)
    r, v = _plan(lib, op, N, D, C, dt, dt, ws)
    assert (v[0], v[25], v[27]) == (N, v[3], 0)
    assert ws >= N * 128256 * 2  # the whole [N, C] buffer (2.1 GB)


def test_aspect_ratio_chunk_rows(lib):
    """The page's "aspect_ratio[:k]" rule: next_pow2(ceil(N / ceil(C / D))) / k."""
    f = lib.lce_aspect_ratio_chunk_rows
    f.argtypes = [I64, I64, I64, I64]
    f.restype = I64
    assert f(8192, 4096, 128256, 1) == 256          # ceil(128256 / 4096) = 32 -> 8192 / 32 = 256
    assert f(8192, 4096, 128256, 4) == 64
    assert f(16384, 4096, 131072, 1) == 512
    assert f(2048, 512, 8192, 1) == 128
    assert f(1000, 64, 700, 1) == 128               # ceil(1000 / 11) = 91 -> 128
    assert f(100, 4096, 1000, 1) == 128             # C <= D: one chunk covers all rows
    assert f(8, 4096, 128256, 64) == 1              # never below one row
    assert f(0, 8, 8, 1) == 0 and f(8, 8, 8, 0) == 0
    # the plan for that chunk size: batch chunks with every class stored
    op, dt = lce.LCE_OP_FORWARD_BACKWARD, lce.LCE_BF16
    ws = _ws(lib, op, 8192, 4096, 128256, dt, dt, 256)
    r, v = _plan(lib, op, 8192, 4096, 128256, dt, dt, ws)
    assert r == NF and v[25] == v[3] and v[27] == 0


def test_budget_below_the_smallest_block(lib):
    """A budget below one block of 256 rows x the minimum class chunk gets
    that block (the smallest plan), with batch chunks of 256 rows."""
    f = lib.lce_workspace_size_for_buffer
    op, N, D, C, dt = lce.LCE_OP_FORWARD_BACKWARD, 100000, 1024, 50000, lce.LCE_BF16
    tiny = f(op, N, D, C, dt, lce.LCE_RED_MEAN, dt, 4096)
    r, v = _plan(lib, op, N, D, C, dt, dt, tiny)
    assert r == NF and v[0] == 256 and v[25] == 1024
    assert v[2] <= tiny
