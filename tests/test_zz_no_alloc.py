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


def test_noalloc_on_a_fresh_handle_allocates_nothing():
    """On a handle that has never run vs_spmm, two vs_spmm_noalloc calls of a
    two-phase product leave the handle's scratch and the device's free memory
    unchanged, and match vs_spmm on a second handle of the same matrix bit for
    bit (and the oracle within the tolerance)."""
    coo = W.random_coo(3000, 2500, 200_000, seed=22, values="counts", duplicates=True,
                       sort=False)
    direction, w = "B@A", 16
    B, Bt = dense_operand(coo, direction, w, torch.float32, seed=6)
    # a first call on another handle loads the library's module (and its
    # static array) before anything is measured
    warm = build(coo, "vcs", "row")
    _noalloc(warm, B, vs.empty_out(warm, w, direction), direction)
    warm.destroy()
    A = build(coo, "vcs", "row")
    outs = [vs.empty_out(A, w, direction) for _ in range(2)]
    torch.cuda.synchronize()
    _, scratch0 = A.nbytes()
    free0, _ = torch.cuda.mem_get_info()
    for out in outs:
        _noalloc(A, B, out, direction)
    torch.cuda.synchronize()
    _, scratch1 = A.nbytes()
    free1, _ = torch.cuda.mem_get_info()
    assert scratch1 == scratch0, (scratch0, scratch1)
    assert free1 == free0, (free0, free1)
    R = build(coo, "vcs", "row")
    ref = gpu_out_rows(vs.spmm(R, B, direction, "deterministic"), direction)
    want, D = oracle_product(coo, oracle_triples(coo, "vcs", "row"), direction, Bt)
    for out in outs:
        got = gpu_out_rows(out, direction)
        assert np.array_equal(got, ref)
        assert np.all(np.abs(got - want) <= TOL[torch.float32] * D)
    A.destroy()
    R.destroy()


def test_noalloc_on_a_matrix_with_64_bit_pointers():
    """Wide matrices: the gathers (aligned, and misaligned over the transpose)
    run allocation-free and equal vs_spmm; the two-phase route, which adds the
    segments through a temporary, answers VS_ERR_UNSUPPORTED."""
    coo = W.random_coo(2000, 1500, 80_000, seed=23, values="counts", duplicates=True, sort=False)
    c = coo.to("cuda")
    A = vs.build_vcs(c.rows, c.cols, c.vals, (coo.n_rows, coo.n_cols), "row", pointer_bits=64,
                     segment_entries=9_000)
    assert A.info()["n_segments"] > 5
    B, Bt = dense_operand(coo, "A@B", 16, torch.float32, seed=7)
    want, D = oracle_product(coo, oracle_triples(coo, "vcs", "row"), "A@B", Bt)
    for _ in range(2):
        got = gpu_out_rows(_noalloc(A, B, vs.empty_out(A, 16, "A@B"), "A@B"), "A@B")
        assert np.array_equal(got, gpu_out_rows(vs.spmm(A, B, "A@B"), "A@B"))
        assert np.all(np.abs(got - want) <= TOL[torch.float32] * D)
    Bl, _ = dense_operand(coo, "B@A", 16, torch.float32, seed=8)
    with pytest.raises(L.VsError) as e:
        _noalloc(A, Bl, vs.empty_out(A, 16, "B@A"), "B@A")
    assert e.value.status == 8
    A.attach_transpose()
    got = gpu_out_rows(_noalloc(A, Bl, vs.empty_out(A, 16, "B@A"), "B@A"), "B@A")
    assert np.array_equal(got, gpu_out_rows(vs.spmm(A, Bl, "B@A"), "B@A"))
    A.destroy()
