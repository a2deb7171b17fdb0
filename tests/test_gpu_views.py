"""Normalized views: products with diag(r) g(A) diag(c) in place of A, for the
value maps and scalings of vs_spmm_view, every layout and direction, against
the float64 oracle's view of the matrix (oracle.view_triples) and its
products."""
import pytest
import torch

import oracle
import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import (PRODUCTS, TOL, aligned, assert_close, build, dense_operand, gpu_out_rows,
                         oracle_product, oracle_triples)

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def _scales(coo, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    r = (0.25 + torch.rand(coo.n_rows, generator=g, dtype=torch.float64)).to(dtype)
    c = (0.25 + torch.rand(coo.n_cols, generator=g, dtype=torch.float64)).to(dtype)
    return r, c


def _view_triples(tri, gname, r, c):
    ti, tj, ta = tri
    return oracle.view_triples(ti, tj, ta, gname, None if r is None else r.double().numpy(),
                               None if c is None else c.double().numpy())


@pytest.mark.parametrize("gname", ["identity", "log1p", "sqrt"])
@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
def test_view_products(layout, major, direction, gname):
    coo = W.random_coo(900, 700, 60_000, seed=23, values="counts", duplicates=True, sort=False)
    A = build(coo, layout, major)
    r, c = _scales(coo, torch.float32, 9)
    tri = oracle_triples(coo, layout, major)
    B, Bt = dense_operand(coo, direction, 16, torch.float32, seed=2)
    variants = ["deterministic"] if aligned(major, direction) else \
        ["two_phase", "atomic", "transposed"]
    for rs, cs in ((r, c), (r, None), (None, c)):
        want, D = oracle_product(coo, _view_triples(tri, gname, rs, cs), direction, Bt)
        for variant in variants:
            if variant == "transposed":
                A.attach_transpose()
            kw = dict(map=gname, row_scale=None if rs is None else rs.cuda(),
                      col_scale=None if cs is None else cs.cuda())
            out = vs.spmm(A, B, direction, variant, **kw)
            got = gpu_out_rows(out, direction)
            assert_close(got, want, D, TOL[torch.float32],
                         f"{layout}/{major} {direction} {variant} g={gname}")
            if variant != "atomic":
                assert torch.equal(vs.spmm(A, B, direction, variant, **kw), out)
    A.destroy()


def test_view_identity_without_scales_equals_plain_product():
    coo = W.random_coo(500, 400, 20_000, seed=29, values="counts", sort=False)
    A = build(coo, "vcs", "row")
    B, _ = dense_operand(coo, "A@B", 8, torch.float32)
    plain = vs.spmm(A, B, "A@B")
    viewed = vs.spmm(A, B, "A@B", map="identity",
                     row_scale=torch.ones(coo.n_rows, device="cuda"))
    assert torch.equal(plain, viewed)
    A.destroy()


def test_view_float64_csr_long_rows():
    coo = W.random_coo(40, 3000, 60_000, seed=31, values="normal", dtype=torch.float64,
                       sort=False)
    A = build(coo, "csr", "row")
    assert A.info()["n_long_slices"] > 0          # the share combine applies the row scale
    r, c = _scales(coo, torch.float64, 11)
    B, Bt = dense_operand(coo, "A@B", 5, torch.float64, seed=3)
    tri = oracle_triples(coo, "csr", "row")
    want, D = oracle_product(coo, _view_triples(tri, "identity", r, c), "A@B", Bt)
    got = gpu_out_rows(vs.spmm(A, B, "A@B", row_scale=r.cuda(), col_scale=c.cuda()), "A@B")
    assert_close(got, want, D, TOL[torch.float64], "f64 view")
    A.destroy()
