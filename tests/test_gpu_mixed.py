"""Mixed precision: a float32 CSR or VCS matrix with float64 operands; products
and sums in float64 ("Regridder", "Why not cuSPARSE": a float32 matrix
applied to float64 data).  Against the float64 oracle at the float64
tolerance: the stored values are exact in float64, so only the summation
order differs."""
import pytest
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import _lib as L
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import (PRODUCTS, TOL, aligned, assert_close, build, dense_operand, gpu_out_rows,
                         oracle_product, oracle_triples)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


CASES = {
    # name: (coo, widths) -- a small X (shared-memory slab) and a long-slice matrix
    "small": (lambda: W.random_coo(1500, 800, 50_000, seed=41, values="counts", sort=False),
              (1, 8, 33)),
    "long": (lambda: W.random_coo(60, 9000, 120_000, seed=43, values="normal", sort=False),
             (4, 16)),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
def test_float32_matrix_float64_operands(case, layout, major, direction):
    make, widths = CASES[case]
    coo = make()
    A = build(coo, layout, major)
    tri = oracle_triples(coo, layout, major)
    if not aligned(major, direction):
        for variant in ("two_phase", "atomic"):
            B, _ = dense_operand(coo, direction, 4, torch.float64)
            with pytest.raises(L.VsError) as e:
                vs.spmm(A, B, direction, variant)
            assert L.STATUS[e.value.status] == "VS_ERR_UNSUPPORTED"
        A.attach_transpose()
    for w in widths:
        B, Bt = dense_operand(coo, direction, w, torch.float64, seed=w)
        want, D = oracle_product(coo, tri, direction, Bt)
        out = vs.spmm(A, B, direction)
        assert out.dtype == torch.float64
        got = gpu_out_rows(out, direction)
        assert_close(got, want, D, TOL[torch.float64], f"{case} {layout}/{major} {direction} w={w}")
        assert torch.equal(vs.spmm(A, B, direction), out)
    A.destroy()


def test_float64_matrix_rejects_float32_operands():
    coo = W.random_coo(100, 80, 1000, seed=3, dtype=torch.float64)
    A = build(coo, "csr", "row")
    B, _ = dense_operand(coo, "A@B", 4, torch.float32)
    with pytest.raises(L.VsError) as e:
        vs.spmm(A, B, "A@B")
    assert L.STATUS[e.value.status] == "VS_ERR_INVALID"
    A.destroy()
