"""GPU parity: libvs assembly and products against the float64 oracle.

Assembly must be bit-exact (integer arrays equal, value arrays equal bit for
bit).  Products must satisfy |gpu - oracle| <= 1e-5 * sum|a||b| per element
(float32; 1e-12 for float64), exactly 0 where that sum is 0.  Deterministic
kernels must repeat bit for bit and give each column the same bits alone or in
a batch.
"""
import numpy as np
import pytest
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import (PRODUCTS, TOL, aligned, assert_arrays_equal, assert_close, build,
                         dense_operand, gpu_out_rows, oracle_arrays, oracle_product,
                         oracle_triples, workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()
    yield
    torch.cuda.synchronize()


def _variants(major, direction):
    return ["deterministic"] if aligned(major, direction) else ["deterministic", "two_phase",
                                                                "atomic", "transposed"]


def _run(A, B, direction, variant):
    if variant == "transposed":
        A.attach_transpose()
    out = vs.spmm(A, B, direction, variant)
    torch.cuda.synchronize()
    return out


# ----------------------------------------------------------------------------- assembly


@pytest.mark.parametrize("layout,major", [("csr", "row"), ("csr", "col"), ("vcs", "row"),
                                          ("vcs", "col")])
@pytest.mark.parametrize("case", ["tiny", "tiny_permuted", "dups_unsorted", "signed_zero"])
def test_assembly_bit_exact(layout, major, case):
    if case == "tiny":
        coo = workload("tiny")
    elif case == "tiny_permuted":
        coo = W.permute(workload("tiny"), seed=3)
    elif case == "dups_unsorted":
        coo = W.random_coo(3000, 700, 40000, seed=2, duplicates=True, empty_rows=0.1, sort=False,
                           values="normal")
    else:
        coo = W.random_coo(500, 300, 20000, seed=4, duplicates=True, sort=False,
                           values="signed_zero")
    A = build(coo, layout, major)
    assert_arrays_equal(A, oracle_arrays(coo, layout, major))
    info = A.info()
    assert info["nnz"] == coo.nnz
    lb, _ = A.nbytes()
    n_major = coo.n_rows if major == "row" else coo.n_cols
    if layout == "vcs":  # stays compressed: no per-nonzero value array
        assert lb == 4 * (n_major + 1) + 4 * coo.nnz + 4 * info["n_runs"] + 4 * (info["n_runs"] + 1)
    A.destroy()


def test_assembly_float64_csr_bit_exact():
    coo = W.random_coo(4000, 900, 60000, seed=6, values="normal", dtype=torch.float64,
                       duplicates=True, sort=False)
    for major in ("row", "col"):
        A = build(coo, "csr", major)
        assert_arrays_equal(A, oracle_arrays(coo, "csr", major))


def test_assembly_rejects_bad_coordinates_and_nan():
    dev = torch.device("cuda")
    r = torch.tensor([0, 5], dtype=torch.int32, device=dev)
    c = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    v = torch.ones(2, device=dev)
    with pytest.raises(vs.VsError) as e:
        vs.build_csr(r, c, v, (5, 3))
    assert e.value.status == 4
    with pytest.raises(vs.VsError) as e:
        vs.build_vcs(r - 0, c, torch.tensor([1.0, float("nan")], device=dev), (6, 3))
    assert e.value.status == 9


def test_transpose_matches_oracle_build_of_layout_order():
    coo = W.random_coo(2500, 800, 30000, seed=8, duplicates=True, sort=False, values="normal")
    A = build(coo, "csr", "row").attach_transpose()
    # the exact transpose lists, per column, the entries in CSR order
    arr = oracle_arrays(coo, "csr", "row")
    ptr = arr["ptr"]
    rows = np.repeat(np.arange(coo.n_rows, dtype=np.int32), np.diff(ptr))
    t = W.Coo(coo.n_rows, coo.n_cols, torch.tensor(rows), torch.tensor(arr["indices"]),
              torch.tensor(arr["values"]))
    assert A.info()["has_transpose"] == 1
    B, Bt = dense_operand(coo, "A@B", 8, torch.float32)
    out_t = vs.spmm(A, B, "A@B", "deterministic")  # aligned: unaffected by the transpose
    # misaligned B@CSR through the transpose equals the aligned gather over that CSC
    Bl, Blt = dense_operand(coo, "B@A", 8, torch.float32)
    got = gpu_out_rows(vs.spmm(A, Bl, "B@A", "transposed"), "B@A")
    C = build(t, "csr", "col")
    want = gpu_out_rows(vs.spmm(C, Bl, "B@A", "deterministic"), "B@A")
    assert np.array_equal(got, want)
    del out_t


# ----------------------------------------------------------------------------- products


WIDTHS = [0, 1, 2, 3, 4, 5, 7, 8, 12, 15, 16, 17, 31, 32, 33, 63, 64, 65, 100]


@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
@pytest.mark.parametrize("w", WIDTHS)
def test_products_tiny_workload(layout, major, direction, w):
    coo = workload("tiny")
    A = build(coo, layout, major)
    tri = oracle_triples(coo, layout, major)
    B, Bt = dense_operand(coo, direction, w, torch.float32)
    want, D = oracle_product(coo, tri, direction, Bt)
    for variant in _variants(major, direction):
        got = gpu_out_rows(_run(A, B, direction, variant), direction)
        assert_close(got, want, D, TOL[torch.float32], f"{layout}/{major} {direction} {variant} w={w}")


@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
def test_products_long_slices_and_empty_rows(layout, major, direction):
    # a few slices far longer than the chunk length, many empty ones, duplicates
    g = torch.Generator().manual_seed(5)
    n_rows, n_cols = 700, 6000
    long_rows = torch.tensor([0, 3, 350, 699])
    r = [long_rows.repeat_interleave(torch.tensor([5000, 2100, 1025, 4097]))]
    c = [torch.cat([torch.randperm(n_cols, generator=g)[:k] for k in (5000, 2100, 1025, 4097)])]
    short = torch.randint(0, n_rows, (9000,), generator=g)
    r.append(short)
    c.append(torch.randint(0, n_cols, (9000,), generator=g))
    rows = torch.cat(r).to(torch.int32)
    cols = torch.cat(c).to(torch.int32)
    vals = torch.empty(rows.numel()).geometric_(0.5, generator=g).float()
    coo = W.permute(W.Coo(n_rows, n_cols, rows, cols, vals), seed=1)
    A = build(coo, layout, major)
    assert_arrays_equal(A, oracle_arrays(coo, layout, major))
    tri = oracle_triples(coo, layout, major)
    for w in (1, 16, 33):
        B, Bt = dense_operand(coo, direction, w, torch.float32)
        want, D = oracle_product(coo, tri, direction, Bt)
        for variant in _variants(major, direction):
            got = gpu_out_rows(_run(A, B, direction, variant), direction)
            assert_close(got, want, D, TOL[torch.float32], f"{layout}/{major} {direction} {variant} w={w}")


@pytest.mark.parametrize("direction", ["A@B", "B@A"])
@pytest.mark.parametrize("major", ["row", "col"])
def test_products_float64_csr(direction, major):
    coo = W.random_coo(3000, 1100, 50000, seed=9, values="normal", dtype=torch.float64,
                       duplicates=True, sort=False)
    A = build(coo, "csr", major)
    tri = oracle_triples(coo, "csr", major)
    for w in (1, 4, 6, 32, 70):
        B, Bt = dense_operand(coo, direction, w, torch.float64)
        want, D = oracle_product(coo, tri, direction, Bt)
        for variant in _variants(major, direction):
            got = gpu_out_rows(_run(A, B, direction, variant), direction)
            assert_close(got, want, D, TOL[torch.float64], f"f64 {major} {direction} {variant} w={w}")


@pytest.mark.parametrize("shape,nnz", [((0, 7), 0), ((9, 0), 0), ((5, 5), 0), ((1, 400), 400),
                                       ((400, 1), 400), ((1, 1), 1)])
@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
def test_degenerate_shapes(shape, nnz, layout, major, direction):
    n_rows, n_cols = shape
    if nnz:
        coo = W.random_coo(n_rows, n_cols, nnz, seed=1)
    else:
        z = torch.empty(0, dtype=torch.int32)
        coo = W.Coo(n_rows, n_cols, z, z.clone(), torch.empty(0))
    A = build(coo, layout, major)
    tri = oracle_triples(coo, layout, major)
    for w in (0, 1, 4, 9):
        B, Bt = dense_operand(coo, direction, w, torch.float32)
        want, D = oracle_product(coo, tri, direction, Bt)
        for variant in _variants(major, direction):
            out = vs.empty_out(A, w, direction)
            out.fill_(float("nan"))  # every element must be written
            if variant == "transposed":
                A.attach_transpose()
            vs.spmm(A, B, direction, variant, out=out)
            torch.cuda.synchronize()
            got = gpu_out_rows(out, direction)
            assert_close(got, want, D, TOL[torch.float32], f"{shape} {layout}/{major} {direction} {variant}")


def test_strided_operands_and_layout_errors():
    coo = workload("tiny")
    A = build(coo, "vcs", "row")
    tri = oracle_triples(coo, "vcs", "row")
    big = W.dense(coo.n_cols, 40, seed=2).cuda()
    B = big[:, 3:19]   # row stride 40, unaligned start
    want, D = oracle_product(coo, tri, "A@B", B.cpu().double().numpy())
    out_big = torch.full((coo.n_rows, 50), float("nan"), device="cuda")
    out = out_big[:, 5:21]
    vs.spmm(A, B, "A@B", out=out)
    torch.cuda.synchronize()
    assert_close(out.cpu().double().numpy(), want, D, 1e-5, "strided")
    assert torch.isnan(out_big[:, :5]).all() and torch.isnan(out_big[:, 21:]).all()
    with pytest.raises(vs.VsError) as e:      # width axis not contiguous
        vs.spmm(A, big.t().contiguous().t()[:, :16], "A@B")
    assert e.value.status == 3
    with pytest.raises(vs.VsError) as e:      # wrong shape
        vs.spmm(A, big[:100, :16], "A@B")
    assert e.value.status == 2
    with pytest.raises(vs.VsError) as e:      # dtype mismatch between B and out
        vs.spmm(A, big[:, :16].double(), "A@B",
                out=torch.empty((coo.n_rows, 16), device="cuda"))
    assert e.value.status == 1
    with pytest.raises(vs.VsError):           # transposed variant without a transpose
        vs.spmm(build(coo, "vcs", "col"), big[:, :16].contiguous(), "A@B", "transposed")


# ----------------------------------------------------------------------------- determinism


@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
def test_repeats_bit_identical_and_column_alone_equals_batch(layout, major, direction):
    coo = workload("tiny")
    A = build(coo, layout, major)
    variants = (["deterministic"] if aligned(major, direction)
                else ["deterministic", "two_phase", "transposed"])
    B, _ = dense_operand(coo, direction, 33, torch.float32)
    for variant in variants:
        ref = _run(A, B, direction, variant).clone()
        for _ in range(20):
            assert torch.equal(_run(A, B, direction, variant), ref)
        for c in (0, 5, 16, 32):
            Bc = (B[:, c:c + 1] if direction == "A@B" else B[c:c + 1, :]).contiguous()
            if direction == "B@A":
                Bc = Bc.t().contiguous().t()
            alone = _run(A, Bc, direction, variant)
            col = ref[:, c:c + 1] if direction == "A@B" else ref[c:c + 1, :]
            assert torch.equal(alone.reshape(-1), col.reshape(-1)), (variant, c)


def _columns(B, direction, c0, c1):
    """Columns [c0, c1) of the dense operand as a new operand of the same layout."""
    if direction == "A@B":
        return B[:, c0:c1].contiguous()
    return B[c0:c1, :].t().contiguous().t()


@pytest.mark.parametrize("layout", ["csr", "vcs"])
@pytest.mark.parametrize("major,direction", [("row", "A@B"), ("col", "B@A")])
def test_shared_slab_and_l1_gathers_agree_bitwise(layout, major, direction):
    """X of 6,000 rows: widths 1 and 4 keep it in a shared-memory slab, width 16
    reads it through L1.  The summation tree is fixed by the matrix, so every
    column has the same bits either way."""
    shape = (3000, 6000) if major == "row" else (6000, 3000)
    coo = W.random_coo(*shape, 600_000, seed=31, values="counts", sort=False)
    A = build(coo, layout, major)
    B, Bt = dense_operand(coo, direction, 16, torch.float32, seed=3)
    batch = _run(A, B, direction, "deterministic")
    want, D = oracle_product(coo, oracle_triples(coo, layout, major), direction, Bt)
    assert_close(gpu_out_rows(batch, direction), want, D, 1e-5, f"{layout}/{major} w=16")
    for c0, c1 in ((0, 1), (7, 8), (15, 16), (4, 8), (12, 16)):
        part = _run(A, _columns(B, direction, c0, c1), direction, "deterministic")
        ref = batch[:, c0:c1] if direction == "A@B" else batch[c0:c1, :]
        assert torch.equal(part, ref), (c0, c1)
    A.destroy()


def test_atomic_and_deterministic_agree_within_tolerance_on_main_workload():
    coo = workload("main")
    for layout, major, direction in [("vcs", "col", "A@B"), ("vcs", "row", "B@A"),
                                     ("csr", "row", "B@A")]:
        A = build(coo, layout, major)
        B, Bt = dense_operand(coo, direction, 16, torch.float32)
        tri = oracle_triples(coo, layout, major)
        want, D = oracle_product(coo, tri, direction, Bt)
        for variant in ("deterministic", "two_phase", "atomic", "transposed"):
            got = gpu_out_rows(_run(A, B, direction, variant), direction)
            assert_close(got, want, D, 1e-5, f"main {layout}/{major} {direction} {variant}")
        A.destroy()


@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
def test_main_workload_full_parity(layout, major, direction):
    """60,000 x 2,000, ~6M nonzeros, width 16: every output element against the oracle."""
    coo = workload("main")
    A = build(coo, layout, major)
    assert_arrays_equal(A, oracle_arrays(coo, layout, major))
    tri = oracle_triples(coo, layout, major)
    B, Bt = dense_operand(coo, direction, 16, torch.float32)
    want, D = oracle_product(coo, tri, direction, Bt)
    for variant in _variants(major, direction):
        got = gpu_out_rows(_run(A, B, direction, variant), direction)
        assert_close(got, want, D, 1e-5, f"main {layout}/{major} {direction} {variant}")
    A.destroy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.float64])
@pytest.mark.parametrize("direction", ["A@B", "B@A"])
def test_regrid_workload(dtype, direction):
    """Backprojection rows of 2-4 entries and their exact transpose; widths 1, 4, 32."""
    coo = workload("regrid", dtype=dtype)
    A = build(coo, "csr", "row")
    info = A.info()
    assert info["group_size"] == 2      # mean 3 entries per row
    A.attach_transpose()
    tri = oracle_triples(coo, "csr", "row")
    for w in (1, 4, 32):
        B, Bt = dense_operand(coo, direction, w, dtype)
        want, D = oracle_product(coo, tri, direction, Bt)
        variants = (["deterministic"] if direction == "A@B"
                    else ["deterministic", "two_phase", "atomic", "transposed"])
        for variant in variants:
            out = _run(A, B, direction, variant)
            got = gpu_out_rows(out, direction)
            assert_close(got, want, D, TOL[dtype], f"regrid {dtype} {direction} {variant} w={w}")
            if variant != "atomic":
                for _ in range(3):
                    assert torch.equal(_run(A, B, direction, variant), out)


@pytest.mark.parametrize("w", [16, 64])
def test_two_phase_partial_tiles_sorted_runs_with_duplicates(w):
    """VCSC@B and B@VCSR whose output spans several shared-memory tiles: the
    two-phase records come from per-run searches and stay in entry order;
    duplicate (row, column) entries land in the same step.  Against the oracle,
    and bit-identical on repeats."""
    coo = W.random_coo(6000, 4000, 200_000, seed=71, values="counts", duplicates=True,
                       sort=False)
    for major, direction in (("col", "A@B"), ("row", "B@A")):
        A = build(coo, "vcs", major)
        tri = oracle_triples(coo, "vcs", major)
        B, Bt = dense_operand(coo, direction, w, torch.float32, seed=w)
        want, D = oracle_product(coo, tri, direction, Bt)
        out = vs.spmm(A, B, direction, "two_phase")
        assert_close(gpu_out_rows(out, direction), want, D, TOL[torch.float32],
                     f"two_phase vcs/{major} {direction} w={w}")
        for _ in range(2):
            assert torch.equal(vs.spmm(A, B, direction, "two_phase"), out)
        A.destroy()
