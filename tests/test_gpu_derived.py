"""Matrices derived from a built one: the exact transpose as a matrix of its own
("Regridder", "API": .T) and the per-entry scaled copy that shares its indices
(the hook of the conservative transpose).  Arrays bit-exact against the
oracle's builds, products against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import _lib as L
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import TOL, assert_arrays_equal, assert_close, build, oracle_triples

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def _coo(dtype=torch.float32):
    return W.random_coo(700, 1300, 40_000, seed=17, values="counts", duplicates=True,
                        sort=False, dtype=dtype)


def _product(A: vs.SparseMatrix, n_rows: int, n_cols: int, ti, tj, ta, w: int, dtype):
    X = W.dense(n_cols, w, seed=4, dtype=dtype)
    got = vs.spmm(A, X.cuda(), "A@B").double().cpu().numpy()
    want, D = oracle.spmm_ab(n_rows, n_cols, ti, tj, ta, X.double().numpy())
    return got, want, D


@pytest.mark.parametrize("layout", ["csr", "vcs"])
@pytest.mark.parametrize("major", ["row", "col"])
def test_transpose_is_a_matrix_of_its_own(layout, major):
    coo = _coo()
    A = build(coo, layout, major)
    ti, tj, ta = oracle_triples(coo, layout, major)   # A's entries in storage order
    T = A.transpose()
    assert T.shape == (coo.n_cols, coo.n_rows) and T.layout == layout and T.major == major
    # the oracle's layout of A^T built from A's entries in A's storage order
    maj, mnr = (tj, ti) if major == "row" else (ti, tj)
    nm, nn = (coo.n_cols, coo.n_rows) if major == "row" else (coo.n_rows, coo.n_cols)
    if layout == "vcs":
        mp, vals, vp, ind = oracle.vcs_build(nm, nn, maj, mnr, ta.astype(np.float32))
        want = {"ptr": mp, "values": vals, "value_ptr": vp, "indices": ind}
    else:
        p, i, v = oracle.csr_build(nm, nn, maj, mnr, ta.astype(np.float32))
        want = {"ptr": p, "indices": i, "values": v}
    assert_arrays_equal(T, want)
    got, ref, D = _product(T, coo.n_cols, coo.n_rows, tj, ti, ta, 16, torch.float32)
    assert_close(got, ref, D, TOL[torch.float32], f"A^T @ B {layout}/{major}")
    A.destroy()                      # T owns its arrays
    got2, _, _ = _product(T, coo.n_cols, coo.n_rows, tj, ti, ta, 16, torch.float32)
    assert np.array_equal(got, got2)
    T.destroy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.float64])
@pytest.mark.parametrize("major", ["row", "col"])
def test_scaled_entries_share_indices(dtype, major):
    coo = _coo(dtype)
    A = build(coo, "csr", major)
    a = A.arrays()
    nnz = a["indices"].numel()
    g = torch.Generator().manual_seed(3)
    f = (0.5 + 1.5 * torch.rand(nnz, generator=g, dtype=torch.float64)).to(dtype)
    S = A.scale_entries(f.cuda())
    s = S.arrays()
    assert torch.equal(s["ptr"], a["ptr"]) and torch.equal(s["indices"], a["indices"])
    want_vals = (a["values"].cpu() * f)           # one rounding in the dtype, as on the GPU
    assert torch.equal(s["values"].cpu().view(torch.int64 if dtype == torch.float64 else torch.int32),
                       want_vals.view(torch.int64 if dtype == torch.float64 else torch.int32))
    # the product with the scaled values, against the oracle on the same triples
    ti, tj, _ = oracle_triples(coo, "csr", major)
    ta = want_vals.double().numpy()
    X = W.dense(coo.n_cols, 8, seed=5, dtype=dtype)
    want, D = oracle.spmm_ab(coo.n_rows, coo.n_cols, ti, tj, ta, X.double().numpy())
    direction = "A@B"
    if major == "col":
        S.attach_transpose()
    got = vs.spmm(S, X.cuda(), direction).double().cpu().numpy()
    assert_close(got, want, D, TOL[dtype], f"scaled {major} {dtype}")
    # the shared index arrays outlive the handle that built them
    A.destroy()
    again = vs.spmm(S, X.cuda(), direction).double().cpu().numpy()
    assert np.array_equal(got, again)
    S.destroy()


def test_scaled_entries_then_original_still_intact():
    coo = _coo()
    A = build(coo, "csr", "row")
    X = W.dense(coo.n_cols, 4, seed=6).cuda()
    before = vs.spmm(A, X, "A@B").clone()
    S = A.scale_entries(torch.full((coo.nnz,), 2.0, device="cuda"))
    S.destroy()
    assert torch.equal(vs.spmm(A, X, "A@B"), before)
    A.destroy()


def test_scale_entries_rejects_vcs():
    coo = _coo()
    A = build(coo, "vcs", "row")
    with pytest.raises(L.VsError) as e:
        A.scale_entries(torch.ones(coo.nnz, device="cuda"))
    assert L.STATUS[e.value.status] == "VS_ERR_LAYOUT"
    A.destroy()
