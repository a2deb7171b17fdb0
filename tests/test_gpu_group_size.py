"""Every group size against the oracle ("Regridder", "Tests": each group size
from 1 to 32 matches the dense product).

vs_force_group_size fixes g for a matrix's gathers (and its transpose's), so
every (G slots, NP partials per lane) instantiation the width and g select is
run: g in {1, 2, 4, 8, 16, 32} at widths 1, 16 and 33 (scalar lanes, 16-byte
vectors, and a ragged second column pass), on a matrix with short slices, empty
slices and slices long enough to be cut into chunks and shares.  Each product
must match the float64 oracle within 1e-5 * sum|a||b|, repeat bit for bit, and
give a column the same bits alone as in the batch.
"""
import pytest
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import (PRODUCTS, TOL, aligned, assert_close, build, dense_operand, gpu_out_rows,
                         oracle_product, oracle_triples)

pytestmark = pytest.mark.gpu

GROUP_SIZES = [1, 2, 4, 8, 16, 32]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


@pytest.fixture(scope="module")
def coo():
    """1,200 x 3,000 with ~30 entries per row (some rows empty), plus three rows
    of 1,100, 2,500 and 3,000 entries (chunked, with shares)."""
    base = W.random_coo(1200, 3000, 36_000, seed=41, values="counts", duplicates=True,
                        empty_rows=0.05, sort=False)
    g = torch.Generator().manual_seed(42)
    rows, cols = [base.rows], [base.cols]
    for r, k in ((7, 1100), (500, 2500), (1199, 3000)):
        rows.append(torch.full((k,), r, dtype=torch.int32))
        cols.append(torch.randperm(3000, generator=g)[:k].to(torch.int32))
    n = sum(x.numel() for x in rows) - base.nnz
    vals = torch.cat([base.vals, torch.empty(n).geometric_(0.5, generator=g).float()])
    return W.permute(W.Coo(1200, 3000, torch.cat(rows), torch.cat(cols), vals), seed=43)


def _column(B, direction, c):
    if direction == "A@B":
        return B[:, c:c + 1].contiguous()
    return B[c:c + 1, :].t().contiguous().t()


@pytest.mark.parametrize("g", GROUP_SIZES)
@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
def test_forced_group_size_matches_oracle(coo, layout, major, direction, g):
    A = build(coo, layout, major)
    A.force_group_size(g)
    assert A.info()["group_size"] == g
    A.attach_transpose()  # misaligned products gather over it, with the same g
    tri = oracle_triples(coo, layout, major)
    variants = ["deterministic"] if aligned(major, direction) else ["deterministic", "atomic"]
    for w in (1, 16, 33):
        B, Bt = dense_operand(coo, direction, w, torch.float32, seed=w)
        want, D = oracle_product(coo, tri, direction, Bt)
        for variant in variants:
            out = vs.spmm(A, B, direction, variant)
            torch.cuda.synchronize()
            assert_close(gpu_out_rows(out, direction), want, D, TOL[torch.float32],
                         f"g={g} {layout}/{major} {direction} {variant} w={w}")
            if variant == "atomic":
                continue
            for _ in range(3):
                assert torch.equal(vs.spmm(A, B, direction, variant), out)
            for c in {0, w // 2, w - 1}:
                alone = vs.spmm(A, _column(B, direction, c), direction, variant)
                col = out[:, c:c + 1] if direction == "A@B" else out[c:c + 1, :]
                assert torch.equal(alone.reshape(-1), col.reshape(-1)), (g, w, c)
    A.destroy()


def test_group_size_rule_restored_and_bad_values_rejected(coo):
    A = build(coo, "csr", "row")
    rule = A.info()["group_size"]
    mean = coo.nnz // coo.n_rows          # 42,600 entries over 1,200 rows: 35
    assert rule == min(32, 1 << (mean.bit_length() - 1))
    A.force_group_size(4)
    assert A.info()["group_size"] == 4
    A.force_group_size(0)
    assert A.info()["group_size"] == rule
    for bad in (3, 64, -1):
        with pytest.raises(vs.VsError) as e:
            A.force_group_size(bad)
        assert e.value.status == 1
    A.destroy()
