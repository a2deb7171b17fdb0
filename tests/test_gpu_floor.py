"""vs_gather_floor, the measurement kernel of the second roof: it runs for every
product of a step (the misaligned ones over the attached transpose), costs no
more than the product it bounds, and refuses what it cannot measure."""
import pytest
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import _lib as L
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import PRODUCTS, build, dense_operand

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def _ms(fn, reps=5):
    fn()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return sorted(out)[len(out) // 2]


@pytest.mark.parametrize("layout,major,direction", PRODUCTS)
def test_floor_runs_and_bounds_the_product(layout, major, direction):
    coo = W.random_coo(20_000, 3000, 1_000_000, seed=71, values="counts", sort=False)
    A = build(coo, layout, major)
    B, _ = dense_operand(coo, direction, 16, torch.float32)
    misaligned = (direction == "A@B") != (major == "row")
    if misaligned:
        with pytest.raises(L.VsError) as e:
            vs.gather_floor(A, B, direction)
        assert L.STATUS[e.value.status] == "VS_ERR_UNSUPPORTED"
        A.attach_transpose()
    floor = _ms(lambda: vs.gather_floor(A, B, direction))
    product = _ms(lambda: vs.spmm(A, B, direction))
    assert floor <= product * 1.5, (floor, product)
    A.destroy()


def test_floor_rejects_unsupported_widths():
    coo = W.random_coo(300, 200, 5000, seed=72, values="counts", sort=False)
    A = build(coo, "csr", "row")
    B, _ = dense_operand(coo, "A@B", 6, torch.float32)
    with pytest.raises(L.VsError) as e:
        vs.gather_floor(A, B, "A@B")
    assert L.STATUS[e.value.status] == "VS_ERR_UNSUPPORTED"
    A.destroy()
