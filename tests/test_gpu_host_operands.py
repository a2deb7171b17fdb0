"""vs_spmm_host: the product with B and out in host memory (the end-to-end
path of the benchmark) matches the float64 oracle within the tolerance and
equals the device product bit for bit, for pinned and pageable buffers (a
pinned output of a gather is written in place by the kernel, a pageable one is
staged and copied back), pitched and strided host views, and leaves host memory
outside the logical output untouched."""
import pytest
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import (PRODUCTS, TOL, assert_close, build, dense_operand, gpu_out_rows,
                         oracle_product, oracle_triples)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def _host_out(A, w, direction, dtype, pin, pad):
    """A host output of the product's shape inside a wider (or taller) NaN-filled buffer."""
    n_rows, n_cols = A.shape
    if direction == "A@B":
        big = torch.full((n_rows, w + pad), float("nan"), dtype=dtype, pin_memory=pin)
        return big, big[:, :w]
    big = torch.full((n_cols, w + pad), float("nan"), dtype=dtype, pin_memory=pin).t()
    return big, big[:w, :]


@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
@pytest.mark.parametrize("w,pad,pin", [(16, 0, True), (5, 0, False), (8, 3, True)])
def test_host_operands_match_device_product(layout, major, direction, w, pad, pin):
    coo = W.random_coo(900, 700, 40_000, seed=61, values="counts", sort=False)
    A = build(coo, layout, major)
    A.attach_transpose()
    B, Bt = dense_operand(coo, direction, w, torch.float32, seed=3)
    ref, D = oracle_product(coo, oracle_triples(coo, layout, major), direction, Bt)
    want = vs.spmm(A, B, direction).cpu()
    if direction == "A@B":
        Bh = B.cpu()
        if pin:                      # pinned: read by a copy kernel through its mapping
            Bh = Bh.pin_memory()
    else:                            # the host operand keeps the width-contiguous layout
        Bh = torch.empty(B.shape[1], B.shape[0], dtype=B.dtype, pin_memory=pin)
        Bh.copy_(B.t().cpu())
        Bh = Bh.t()
    big, out = _host_out(A, w, direction, torch.float32, pin, pad)
    vs.spmm_host(A, Bh, direction, "deterministic", out=out)
    assert_close(gpu_out_rows(out, direction), ref, D, TOL[torch.float32],
                 f"host {layout}/{major} {direction} w={w} pin={pin}")
    assert torch.equal(out, want)
    if pad:
        rest = big[:, w:] if direction == "A@B" else big[w:, :]
        assert torch.isnan(rest).all(), "host memory outside the output was written"
    A.destroy()


def test_host_operands_mixed_precision():
    coo = W.random_coo(500, 400, 20_000, seed=62, values="counts", sort=False)
    A = build(coo, "vcs", "row")
    B, Bt = dense_operand(coo, "A@B", 16, torch.float64, seed=4)
    ref, D = oracle_product(coo, oracle_triples(coo, "vcs", "row"), "A@B", Bt)
    want = vs.spmm(A, B, "A@B").cpu()
    got = vs.spmm_host(A, B.cpu().pin_memory(), "A@B", "deterministic")
    assert got.dtype == torch.float64 and torch.equal(got, want)
    assert_close(gpu_out_rows(got, "A@B"), ref, D, TOL[torch.float64], "host mixed")
    A.destroy()


@pytest.mark.parametrize("variant", ["two_phase", "transposed"])
def test_host_operands_misaligned_variants(variant):
    # two_phase stages the output and copies it back; transposed (a gather)
    # writes the pinned output in place: both equal the device product
    coo = W.random_coo(700, 500, 30_000, seed=63, values="counts", sort=False)
    A = build(coo, "vcs", "row")
    A.attach_transpose()
    B, Bt = dense_operand(coo, "B@A", 16, torch.float32, seed=5)
    ref, D = oracle_product(coo, oracle_triples(coo, "vcs", "row"), "B@A", Bt)
    want = vs.spmm(A, B, "B@A", variant).cpu()
    Bh = B.cpu().t().contiguous().t()            # width-contiguous, pageable
    # a pinned, width-contiguous output inside a taller NaN-filled buffer
    big = torch.empty(coo.n_cols, 16 + 2, pin_memory=True).fill_(float("nan")).t()
    out = big[:16, :]
    vs.spmm_host(A, Bh, "B@A", variant, out=out)
    assert_close(gpu_out_rows(out, "B@A"), ref, D, TOL[torch.float32], f"host B@VCSR {variant}")
    assert torch.equal(out, want)
    assert torch.isnan(big[16:, :]).all(), "host memory outside the output was written"
    A.destroy()
