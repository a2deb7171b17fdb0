"""The tiled two-phase scheme: the deterministic misaligned product without a
transpose ("Add CUDA transfer and matmul kernels for the normalized views",
"The kernels"; the two-phase scheme chosen over atomic adds).

The output rows are cut into tiles; the matrix keeps, per (run, tile), where
the run's entries inside the tile start, so each CTA reads only its own
entries.  Every element's sum runs over its group's entries in entry order,
then over the groups in order, so the result depends on the matrix alone: the
tests check it against the oracle, bit for bit on repeats and across tile
sizes (the build option two_phase_tile_rows), and a column computed alone
against the batch; the kernels' failure flag stays clear.
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

TILE = 2048  # default output rows per tile

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


def _flags_clear(A):
    stream = torch.cuda.current_stream().cuda_stream
    L.check(L.load().vs_device_status(A.handle, ctypes.c_void_p(stream)))


def _n_out(coo, major):
    return coo.n_cols if major == "row" else coo.n_rows


def _coo(seed=81, dtype=torch.float32, values="counts", sort=True):
    """3,000 x 2,600 with duplicates, empty rows and two long rows and columns:
    both output sizes span two default tiles."""
    base = W.random_coo(3000, 2600, 90_000, seed=seed, values=values, duplicates=True,
                        empty_rows=0.05, sort=sort, dtype=dtype)
    g = torch.Generator().manual_seed(seed + 1)
    rows, cols = [base.rows], [base.cols]
    for r, k in ((7, 2500), (1500, 2000)):
        rows.append(torch.full((k,), r, dtype=torch.int32))
        cols.append(torch.randperm(2600, generator=g)[:k].sort().values.to(torch.int32))
    for c, k in ((11, 2900), (2599, 2400)):
        cols.append(torch.full((k,), c, dtype=torch.int32))
        rows.append(torch.randperm(3000, generator=g)[:k].sort().values.to(torch.int32))
    extra = sum(x.numel() for x in rows) - base.nnz
    if values == "counts":
        v = torch.empty(extra, dtype=torch.float64).geometric_(0.5, generator=g)
    else:
        v = torch.randn(extra, dtype=torch.float64, generator=g)
    r, c = torch.cat(rows), torch.cat(cols)
    vals = torch.cat([base.vals, v.to(dtype)])
    if sort:
        o = torch.argsort(r.to(torch.int64) * 2600 + c, stable=True)
        r, c, vals = r[o], c[o], vals[o]
    return W.Coo(3000, 2600, r, c, vals)


@pytest.mark.parametrize("layout,major,direction", MISALIGNED)
def test_tiled_matches_oracle_and_is_fixed_by_the_matrix(layout, major, direction):
    coo = _coo()
    A = _build(coo, layout, major)
    tiles = A.info()["two_phase_tiles"]
    assert tiles == (_n_out(coo, major) + TILE - 1) // TILE == 2, A.info()
    small = _build(coo, layout, major, two_phase_tile_rows=100)
    odd = _build(coo, layout, major, two_phase_tile_rows=1)
    assert small.info()["two_phase_tiles"] == (_n_out(coo, major) + 99) // 100
    assert odd.info()["two_phase_tiles"] == _n_out(coo, major)
    tri = oracle_triples(coo, layout, major)
    for w in (1, 4, 16, 33):
        B, Bt = dense_operand(coo, direction, w, torch.float32, seed=w)
        want, D = oracle_product(coo, tri, direction, Bt)
        out = vs.spmm(A, B, direction, "two_phase")
        torch.cuda.synchronize()
        assert_close(gpu_out_rows(out, direction), want, D, TOL[torch.float32],
                     f"tiled {layout}/{major} {direction} w={w}")
        assert torch.equal(vs.spmm(A, B, direction, "two_phase"), out), "repeat"
        # the tiling changes no bit
        assert torch.equal(vs.spmm(small, B, direction, "two_phase"), out), "tile rows 100"
        if w <= 4:
            assert torch.equal(vs.spmm(odd, B, direction, "two_phase"), out), "tile rows 1"
        # a column alone equals the same column of the batch
        for col in {0, w - 1}:
            Bc = B[:, col:col + 1].contiguous() if direction == "A@B" else \
                B[col:col + 1, :].t().contiguous().t()
            oc = vs.spmm(A, Bc, direction, "two_phase")
            ref = out[:, col:col + 1] if direction == "A@B" else out[col:col + 1, :]
            assert torch.equal(oc, ref), f"column {col} alone"
    for h in (A, small, odd):
        _flags_clear(h)
        h.destroy()


@pytest.mark.parametrize("major,direction", [("row", "B@A"), ("col", "A@B")])
def test_tiled_float64_and_unsorted_slices(major, direction):
    """float64 CSR (sorted: tiled over several tiles); and a CSR whose slices are
    not sorted, which keeps the tiled scheme while its output fits one tile and
    the block-stream scheme otherwise."""
    coo = _coo(seed=91, dtype=torch.float64, values="normal")
    A = _build(coo, "csr", major)
    assert A.info()["two_phase_tiles"] == 2
    tri = oracle_triples(coo, "csr", major)
    for w in (3, 8, 17):
        B, Bt = dense_operand(coo, direction, w, torch.float64, seed=w)
        want, D = oracle_product(coo, tri, direction, Bt)
        out = vs.spmm(A, B, direction, "two_phase")
        assert_close(gpu_out_rows(out, direction), want, D, TOL[torch.float64], f"f64 w={w}")
        assert torch.equal(vs.spmm(A, B, direction, "two_phase"), out)
    A.destroy()
    # unsorted slices
    un = W.random_coo(1000, 900, 40_000, seed=92, values="counts", duplicates=True, sort=False)
    for tile_rows, expect in ((0, 1), (500, 0)):
        U = _build(un, "csr", major, two_phase_tile_rows=tile_rows or None)
        assert U.info()["two_phase_tiles"] == expect, U.info()
        tri = oracle_triples(un, "csr", major)
        B, Bt = dense_operand(un, direction, 16, torch.float32, seed=5)
        want, D = oracle_product(un, tri, direction, Bt)
        out = vs.spmm(U, B, direction, "two_phase")
        assert_close(gpu_out_rows(out, direction), want, D, TOL[torch.float32],
                     f"unsorted tile_rows={tile_rows}")
        assert torch.equal(vs.spmm(U, B, direction, "two_phase"), out)
        U.destroy()


def test_tiled_skewed_rows_and_tiny_matrices():
    """Output rows of very different popularity (the owners are balanced by
    entry counts, a single row can hold most entries), a one-entry matrix, a
    one-row output and an output smaller than a warp's share."""
    n_rows, n_cols = 4000, 3000
    g = torch.Generator().manual_seed(7)
    k = torch.arange(1, n_cols + 1, dtype=torch.float64)
    cdf = torch.cumsum(k.pow(-1.5), 0)
    u = torch.rand(120_000, generator=g, dtype=torch.float64) * cdf[-1]
    cols = torch.searchsorted(cdf, u).clamp_(max=n_cols - 1).to(torch.int32)
    rows = torch.randint(0, n_rows, (120_000,), generator=g).to(torch.int32)
    o = torch.argsort(rows.to(torch.int64) * n_cols + cols, stable=True)
    vals = torch.empty(120_000, dtype=torch.float64).geometric_(0.5, generator=g).float()
    coo = W.Coo(n_rows, n_cols, rows[o], cols[o], vals[o])
    for layout in ("vcs", "csr"):
        A = _build(coo, layout, "row")
        assert A.info()["two_phase_tiles"] == 2
        tri = oracle_triples(coo, layout, "row")
        B, Bt = dense_operand(coo, "B@A", 16, torch.float32, seed=3)
        want, D = oracle_product(coo, tri, "B@A", Bt)
        out = vs.spmm(A, B, "B@A", "two_phase")
        assert_close(gpu_out_rows(out, "B@A"), want, D, TOL[torch.float32], f"skewed {layout}")
        assert torch.equal(vs.spmm(A, B, "B@A", "two_phase"), out)
        A.destroy()
    for (nr, nc, nnz) in ((1, 1, 1), (5, 1, 9), (1, 3000, 2500), (40, 7, 300)):
        tiny = W.random_coo(nr, nc, nnz, seed=nr + nc, values="small_int", duplicates=True)
        for layout, major, direction in MISALIGNED:
            A = _build(tiny, layout, major, two_phase_tile_rows=3)
            tri = oracle_triples(tiny, layout, major)
            B, Bt = dense_operand(tiny, direction, 5, torch.float32, seed=1, kind="small_int")
            want, D = oracle_product(tiny, tri, direction, Bt)
            out = vs.spmm(A, B, direction, "two_phase")
            got = gpu_out_rows(out, direction)
            assert np.array_equal(got, want), (nr, nc, layout, major, direction)  # exact: small ints
            A.destroy()


def test_tiled_main_workload_two_phase_vs_oracle_sampled():
    """The main workload's three misaligned products by the tiled scheme, every
    output row checked against the oracle's per-row product."""
    import oracle
    from gpu_helpers import workload
    coo = workload("main")
    for layout, major, direction in (("vcs", "col", "A@B"), ("vcs", "row", "B@A"),
                                     ("csr", "row", "B@A")):
        A = _build(coo, layout, major)
        assert A.info()["two_phase_tiles"] >= 1
        tri = oracle_triples(coo, layout, major)
        B, Bt = dense_operand(coo, direction, 16, torch.float32, seed=11)
        want, D = oracle_product(coo, tri, direction, Bt)
        out = vs.spmm(A, B, direction, "two_phase")
        assert_close(gpu_out_rows(out, direction), want, D, TOL[torch.float32],
                     f"main {layout}/{major} {direction}")
        assert torch.equal(vs.spmm(A, B, direction, "two_phase"), out)
        A.destroy()
    del oracle
