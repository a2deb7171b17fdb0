"""The bucketed two-phase scheme: the deterministic misaligned product without a
transpose for matrices that keep no per-(run, tile) offsets ("Add CUDA transfer
and matmul kernels for the normalized views", "The kernels"; the two-phase
scheme chosen over atomic adds).

Each call sorts the entries stably into (tile of output rows, group of blocks)
buckets and sums every bucket's records in entry order; the groups are the
block-stream scheme's, so every element's sum runs in the same order as there.
The tests check the products against the oracle, bit for bit against the
allocation-free entry point (which runs the block-stream scheme), on repeats and
for a single column against the batch, with many tiles and several groups.
"""
import ctypes

import numpy as np
import pytest
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import _lib as L
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import TOL, assert_close, dense_operand, gpu_out_rows, oracle_product, oracle_triples

pytestmark = pytest.mark.gpu

MISALIGNED = [("vcs", "col", "A@B"), ("vcs", "row", "B@A"), ("csr", "row", "B@A"),
              ("csr", "col", "A@B")]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def _build(coo, layout, major, **kw):
    c = coo.to("cuda")
    fn = vs.build_vcs if layout == "vcs" else vs.build_csr
    return fn(c.rows, c.cols, c.vals, (coo.n_rows, coo.n_cols), major, **kw)


def _block_stream(A, B, direction):
    """The same product through vs_spmm_noalloc (the block-stream scheme here)."""
    out = vs.empty_out(A, B.shape[1] if direction == "A@B" else B.shape[0], direction, B.dtype)
    bd, od = vs.api._dense(B), vs.api._dense(out)
    L.check(L.load().vs_spmm_noalloc(A.handle, ctypes.byref(bd), ctypes.byref(od),
                                     L.A_B if direction == "A@B" else L.B_A,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    return out


def _check(coo, A, layout, major, direction, widths, dtype=torch.float32):
    tri = oracle_triples(coo, layout, major)
    for w in widths:
        B, Bt = dense_operand(coo, direction, w, dtype, seed=w)
        want, D = oracle_product(coo, tri, direction, Bt)
        out = vs.spmm(A, B, direction, "two_phase")
        torch.cuda.synchronize()
        assert_close(gpu_out_rows(out, direction), want, D, TOL[dtype],
                     f"bucketed {layout}/{major} {direction} w={w}")
        assert torch.equal(vs.spmm(A, B, direction, "two_phase"), out), "repeat"
        assert torch.equal(_block_stream(A, B, direction), out), "block-stream order"
        col = w - 1
        Bc = B[:, col:col + 1].contiguous() if direction == "A@B" else \
            B[col:col + 1, :].t().contiguous().t()
        oc = vs.spmm(A, Bc, direction, "two_phase")
        ref = out[:, col:col + 1] if direction == "A@B" else out[col:col + 1, :]
        assert torch.equal(oc, ref), "a column alone"
    stream = torch.cuda.current_stream().cuda_stream
    L.check(L.load().vs_device_status(A.handle, ctypes.c_void_p(stream)))


@pytest.mark.parametrize("layout,major,direction", MISALIGNED)
def test_bucketed_matches_oracle_and_the_block_stream_order(layout, major, direction):
    """Sorted matrices built without the tiled arrays (two_phase_tile_rows = -1):
    3,000 x 2,600 with duplicates and empty rows, outputs of two tiles."""
    coo = W.random_coo(3000, 2600, 120_000, seed=61, values="counts", duplicates=True,
                       empty_rows=0.05)
    A = _build(coo, layout, major, two_phase_tile_rows=-1)
    assert A.info()["two_phase_tiles"] == 0
    _check(coo, A, layout, major, direction, (1, 4, 16, 33, 64))
    A.destroy()


@pytest.mark.parametrize("layout", ["vcs", "csr"])
def test_bucketed_many_tiles_and_groups(layout):
    """An output of 130,000 rows: 64 tiles and two groups of blocks (the
    partials are combined), including long columns cut into chunks."""
    coo = W.random_coo(130_000, 400, 600_000, seed=62, values="counts", duplicates=False)
    A = _build(coo, layout, "col", two_phase_tile_rows=-1)
    _check(coo, A, layout, "col", "A@B", (16, 5))
    A.destroy()


def test_bucketed_unsorted_slices_and_float64():
    """A CSR whose slices keep COO order (no tiled arrays: its output spans several
    tiles), float32 and float64."""
    for dtype, vals in ((torch.float32, "counts"), (torch.float64, "normal")):
        un = W.random_coo(2500, 5000, 80_000, seed=63, values=vals, duplicates=True, sort=False,
                          dtype=dtype)
        for major, direction in (("row", "B@A"), ("col", "A@B")):
            A = _build(un, "csr", major)
            assert A.info()["two_phase_tiles"] == 0
            _check(un, A, "csr", major, direction, (8, 17), dtype)
            A.destroy()
