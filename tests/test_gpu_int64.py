"""64-bit slice pointers with 32-bit indices ("Regridder", "Why not cuSPARSE").

Handles built with pointer_bits=64 store int64 slice pointers (CSR ptr, VCS
major_ptr and value_ptr) and run the kernels over consecutive slice segments;
segment_entries forces many small segments, so a 50,000-entry matrix takes the
path a matrix of more than 2^31 entries takes.  Checked against the oracle:
the exported arrays bit for bit, every product and variant within the
tolerance, and the gathers bit for bit against the int32 build of the same
matrix (every slice keeps its summation tree).
"""
import os

import numpy as np
import pytest
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

import oracle
from gpu_helpers import (PRODUCTS, TOL, aligned, assert_close, dense_operand, gpu_out_rows,
                         oracle_arrays, oracle_product, oracle_triples)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def _coo(dtype=torch.float32, values="counts"):
    """900 x 1,300 with ~45 entries per row, some empty rows, duplicates, and three
    rows (and, for the column layouts, columns) far longer than a segment."""
    base = W.random_coo(900, 1300, 40_000, seed=51, values=values, duplicates=True,
                        empty_rows=0.05, sort=False, dtype=dtype)
    g = torch.Generator().manual_seed(52)
    rows, cols = [base.rows], [base.cols]
    for r, k in ((3, 1300), (450, 1200), (899, 1250)):
        rows.append(torch.full((k,), r, dtype=torch.int32))
        cols.append(torch.randperm(1300, generator=g)[:k].to(torch.int32))
    extra = sum(x.numel() for x in rows) - base.nnz
    v = torch.empty(extra, dtype=torch.float64).geometric_(0.5, generator=g).to(dtype)
    return W.permute(W.Coo(900, 1300, torch.cat(rows), torch.cat(cols), torch.cat([base.vals, v])),
                     seed=53)


def _build(coo, layout, major, **kw):
    c = coo.to("cuda")
    fn = vs.build_vcs if layout == "vcs" else vs.build_csr
    return fn(c.rows, c.cols, c.vals, (coo.n_rows, coo.n_cols), major, **kw)


SEG = 3000  # entries per segment: ~15 segments, and slices of 1,200+ entries cross no segment


@pytest.mark.parametrize("layout,major", [("csr", "row"), ("csr", "col"), ("vcs", "row"),
                                          ("vcs", "col")])
def test_wide_arrays_match_oracle(layout, major):
    coo = _coo()
    A = _build(coo, layout, major, pointer_bits=64, segment_entries=SEG)
    info = A.info()
    assert info["pointer_bits"] == 64 and info["n_segments"] > 10, info
    want = oracle_arrays(coo, layout, major)
    got = A.arrays()
    assert got["ptr"].dtype == torch.int64
    assert np.array_equal(got["ptr"].cpu().numpy(), want["ptr"].astype(np.int64))
    assert np.array_equal(got["indices"].cpu().numpy(), want["indices"])
    gv, wv = got["values"].cpu().numpy(), want["values"]
    assert np.array_equal(gv.view(np.uint32 if gv.itemsize == 4 else np.uint64),
                          wv.view(np.uint32 if wv.itemsize == 4 else np.uint64))
    if layout == "vcs":
        assert got["value_ptr"].dtype == torch.int64
        assert np.array_equal(got["value_ptr"].cpu().numpy(), want["value_ptr"].astype(np.int64))
    # bytes: 8-byte slice pointers
    lb, _ = A.nbytes()
    n_major = coo.n_rows if major == "row" else coo.n_cols
    if layout == "vcs":
        R = info["n_runs"]
        assert lb == 8 * (n_major + 1) + 4 * coo.nnz + 4 * R + 8 * (R + 1)
    else:
        assert lb == 8 * (n_major + 1) + 8 * coo.nnz
    A.destroy()


@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
def test_wide_products_match_oracle_and_int32_build(layout, major, direction):
    coo = _coo()
    A = _build(coo, layout, major, pointer_bits=64, segment_entries=SEG)
    N = _build(coo, layout, major)  # int32 pointers, one piece
    assert N.info()["pointer_bits"] == 32 and N.info()["n_segments"] == 1
    tri = oracle_triples(coo, layout, major)
    variants = ["deterministic"] if aligned(major, direction) else \
        ["two_phase", "atomic", "transposed"]
    for w in (1, 16, 33):
        B, Bt = dense_operand(coo, direction, w, torch.float32, seed=w)
        want, D = oracle_product(coo, tri, direction, Bt)
        for variant in variants:
            if variant == "transposed":
                A.attach_transpose()
                N.attach_transpose()
            out = vs.spmm(A, B, direction, variant)
            torch.cuda.synchronize()
            assert_close(gpu_out_rows(out, direction), want, D, TOL[torch.float32],
                         f"wide {layout}/{major} {direction} {variant} w={w}")
            if variant == "atomic":
                continue
            assert torch.equal(vs.spmm(A, B, direction, variant), out)
            if variant in ("deterministic", "transposed"):  # the gathers: the same trees
                assert torch.equal(vs.spmm(N, B, direction, variant), out)
    A.destroy()
    N.destroy()


def test_wide_float64_and_derived_handles():
    coo = _coo(torch.float64, "normal")
    A = _build(coo, "csr", "row", pointer_bits=64, segment_entries=SEG)
    tri = oracle_triples(coo, "csr", "row")
    B, Bt = dense_operand(coo, "A@B", 7, torch.float64, seed=3)
    want, D = oracle_product(coo, tri, "A@B", Bt)
    assert_close(gpu_out_rows(vs.spmm(A, B, "A@B"), "A@B"), want, D, TOL[torch.float64], "f64")
    # the exact transpose as a handle of its own (wide too)
    T = A.transpose()
    assert T.info()["pointer_bits"] == 64
    Bl, Blt = dense_operand(coo, "B@A", 5, torch.float64, seed=4)
    want_t, D_t = oracle_product(coo, tri, "B@A", Blt)
    # B @ A == (A^T @ B^T)^T: the transpose handle's A@B with B^T rows
    got_t = gpu_out_rows(vs.spmm(T, Bl.t(), "A@B"), "A@B")
    assert_close(got_t, want_t, D_t, TOL[torch.float64], "transpose handle")
    # entries scaled by factors in storage order, sharing the indices
    f = torch.linspace(0.5, 2.0, coo.nnz, dtype=torch.float64, device="cuda")
    S = A.scale_entries(f)
    a = A.arrays()
    ti, tj, _ = tri
    sv = (a["values"] * f).cpu().numpy()
    want_s, D_s = oracle.spmm_ab(coo.n_rows, coo.n_cols, ti, tj, sv, Bt)
    assert_close(gpu_out_rows(vs.spmm(S, B, "A@B"), "A@B"), want_s, D_s, TOL[torch.float64], "scaled")
    S.destroy()
    A.destroy()
    assert_close(gpu_out_rows(vs.spmm(T, Bl.t(), "A@B"), "A@B"), want_t, D_t,
                 TOL[torch.float64], "transpose outlives its source")
    T.destroy()


def test_wide_views_host_operands_group_size():
    coo = _coo()
    A = _build(coo, "vcs", "row", pointer_bits=64, segment_entries=SEG)
    A.attach_transpose()
    gen = torch.Generator().manual_seed(5)
    r = 0.5 + torch.rand(coo.n_rows, generator=gen)
    c = 0.5 + torch.rand(coo.n_cols, generator=gen)
    ti, tj, ta = oracle_triples(coo, "vcs", "row")
    vtri = oracle.view_triples(ti, tj, ta, "sqrt", r.double().numpy(), c.double().numpy())
    for direction in ("A@B", "B@A"):
        B, Bt = dense_operand(coo, direction, 16, torch.float32, seed=6)
        want, D = oracle_product(coo, vtri, direction, Bt)
        out = vs.spmm(A, B, direction, map="sqrt", row_scale=r.cuda(), col_scale=c.cuda())
        assert_close(gpu_out_rows(out, direction), want, D, TOL[torch.float32], f"view {direction}")
        # host operands, pinned
        want_p, D_p = oracle_product(coo, (ti, tj, ta), direction, Bt)
        Bh = B.cpu().pin_memory() if direction == "A@B" else B.t().cpu().pin_memory().t()
        got = vs.spmm_host(A, Bh, direction, "deterministic")
        assert_close(gpu_out_rows(got, direction), want_p, D_p, TOL[torch.float32], "host")
    for g in (1, 8, 32):
        A.force_group_size(g)
        B, Bt = dense_operand(coo, "A@B", 16, torch.float32, seed=7)
        want, D = oracle_product(coo, (ti, tj, ta), "A@B", Bt)
        out = vs.spmm(A, B, "A@B")
        assert_close(gpu_out_rows(out, "A@B"), want, D, TOL[torch.float32], f"g={g}")
        assert torch.equal(vs.spmm(A, B, "A@B"), out)
    A.destroy()


def test_wide_edge_cases_and_bad_options():
    z = torch.empty(0, dtype=torch.int32, device="cuda")
    A = vs.build_csr(z, z, torch.empty(0, device="cuda"), (5, 4), pointer_bits=64)
    assert A.info()["pointer_bits"] == 64
    out = vs.spmm(A, torch.ones(4, 3, device="cuda"), "A@B")
    assert torch.equal(out.cpu(), torch.zeros(5, 3))
    assert A.arrays()["ptr"].cpu().tolist() == [0] * 6
    A.destroy()
    coo = _coo().to("cuda")
    for bad in ({"pointer_bits": 16}, {"segment_entries": -5}):
        with pytest.raises(vs.VsError) as e:
            vs.build_csr(coo.rows, coo.cols, coo.vals, (coo.n_rows, coo.n_cols), **bad)
        assert e.value.status == 1


@pytest.mark.skipif(os.environ.get("VS_TEST_HUGE") != "1",
                    reason="builds a matrix of more than 2^31 entries (about 100 GB); "
                           "set VS_TEST_HUGE=1")
def test_more_than_2_31_entries():
    """2,200,000,000 entries: rows of 1,100 consecutive columns (mod 20,000),
    value 1 + (row mod 3).  Spot-checked against the definition."""
    n_rows, per_row, n_cols = 2_000_000, 1_100, 20_000
    nnz = n_rows * per_row
    assert nnz > 2 ** 31
    dev = torch.device("cuda")
    rows = (torch.arange(nnz, device=dev, dtype=torch.int64) // per_row).to(torch.int32)
    cols = ((rows.to(torch.int64) * 7 + torch.arange(nnz, device=dev, dtype=torch.int64) % per_row)
            % n_cols).to(torch.int32)
    vals = (1 + rows % 3).to(torch.float32)
    A = vs.build_csr(rows, cols, vals, (n_rows, n_cols))
    del rows, cols, vals
    torch.cuda.empty_cache()
    info = A.info()
    assert info["pointer_bits"] == 64 and info["n_segments"] >= 2 and info["nnz"] == nnz
    ptr = A.arrays()["ptr"]
    assert int(ptr[-1]) == nnz and int(ptr[n_rows // 2]) == (n_rows // 2) * per_row
    del ptr
    B = torch.randn(n_cols, 4, device=dev, dtype=torch.float64).float()
    out = vs.spmm(A, B, "A@B")
    Bd = B.double().cpu().numpy()
    for r in (0, 1, 976_000, 1_952_000, n_rows - 1):  # rows on both sides of the 2^31 boundary
        c = (r * 7 + np.arange(per_row)) % n_cols
        want = (1 + r % 3) * Bd[c].sum(axis=0)
        D = (1 + r % 3) * np.abs(Bd[c]).sum(axis=0)
        assert np.all(np.abs(out[r].double().cpu().numpy() - want) <= 1e-5 * D), r
    A.destroy()
