"""vs_spmm_noalloc: the deterministic product for callers that must not
allocate device memory when they run it (stream capture, foreign allocators).

It is called here through the C ABI directly and checked against vs_spmm
(VS_DETERMINISTIC) on the same handle, within the parity tolerance of the
other GPU tests (|a - b| <= 1e-5 * sum|a||b| per element, float64 oracle for
the scale) and bit for bit, on two calls in a row -- the second one reuses the
static scratch array the first one left behind.  The file sorts last so that a
run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import _lib as L
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import (TOL, build, dense_operand, gpu_out_rows, oracle_product, oracle_triples,
                         workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def _noalloc(A, B, out, direction):
    lib = L.load()
    bd, od = vs.api._dense(B), vs.api._dense(out)
    stream = torch.cuda.current_stream().cuda_stream
    L.check(lib.vs_spmm_noalloc(A.handle, ctypes.byref(bd), ctypes.byref(od),
                                L.A_B if direction == "A@B" else L.B_A, ctypes.c_void_p(stream)))
    torch.cuda.synchronize()
    return out


CASES = [
    # (workload, layout, major, direction, width): misaligned products whose
    # two-phase scheme keeps several group partials, i.e. uses the scratch
    ("random", "vcs", "row", "B@A", 16),
    ("random", "csr", "row", "B@A", 33),
    ("random", "vcs", "col", "A@B", 8),
    ("main", "vcs", "col", "A@B", 16),
    ("main", "vcs", "row", "B@A", 64),   # partials need a narrower column block
    ("main", "csr", "row", "B@A", 16),
    ("main", "vcs", "row", "A@B", 16),   # aligned: the gather, no scratch at all
]


@pytest.mark.parametrize("name,layout,major,direction,w", CASES)
def test_noalloc_matches_vs_spmm_twice(name, layout, major, direction, w):
    if name == "random":
        coo = W.random_coo(3000, 2500, 200_000, seed=21, values="counts", duplicates=True,
                           sort=False)
    else:
        coo = workload(name)
    A = build(coo, layout, major)
    B, Bt = dense_operand(coo, direction, w, torch.float32, seed=5)
    ref = vs.spmm(A, B, direction, "deterministic")
    torch.cuda.synchronize()
    want, D = oracle_product(coo, oracle_triples(coo, layout, major), direction, Bt)
    ref_rows = gpu_out_rows(ref, direction)
    for call in range(2):
        out = vs.empty_out(A, w, direction)
        out.fill_(float("nan"))
        got = gpu_out_rows(_noalloc(A, B, out, direction), direction)
        err = np.abs(got - ref_rows)
        assert np.all(err <= TOL[torch.float32] * D), f"call {call}: beyond tolerance"
        assert np.array_equal(got, ref_rows), f"call {call}: bits differ from vs_spmm"
        assert np.all(np.abs(got - want) <= TOL[torch.float32] * D)
    A.destroy()
