"""The failure path of the product kernels, exercised without a GPU fault: a
test hook makes the next gather's producer issue nothing, so its consumers'
bounded waits (about a second) run out; the kernel marks the handle and
exits.  The host reads the mark as VS_ERR_TIMEOUT, and the same handle and
context then compute correct products again."""
import ctypes

import pytest
import torch

import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import _lib as L
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import TOL, assert_close, build, dense_operand, gpu_out_rows, oracle_product, \
    oracle_triples

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def _status(A) -> str:
    lib = L.load()
    st = lib.vs_device_status(A.handle, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return L.STATUS[st]


@pytest.mark.parametrize("layout,n_cols", [("csr", 60_000), ("vcs", 700)])
def test_stalled_producer_times_out_and_the_handle_recovers(layout, n_cols):
    # csr with a wide X: the L1 gather; vcs with a narrow one: the shared-memory
    # slab gather with its expanding warps
    coo = W.random_coo(2000, n_cols, 50_000, seed=81, values="counts", sort=False)
    A = build(coo, layout, "row")
    B, Bt = dense_operand(coo, "A@B", 16, torch.float32)
    assert _status(A) == "VS_OK"
    L.load().vs_test_stall_producers(1)
    vs.spmm(A, B, "A@B")
    assert _status(A) == "VS_ERR_TIMEOUT"
    assert _status(A) == "VS_OK"                      # reported once
    want, D = oracle_product(coo, oracle_triples(coo, layout, "row"), "A@B", Bt)
    got = gpu_out_rows(vs.spmm(A, B, "A@B"), "A@B")
    assert_close(got, want, D, TOL[torch.float32], "after the timeout")
    assert _status(A) == "VS_OK"
    A.destroy()


def test_host_entry_reports_the_timeout_and_recovers():
    # vs_spmm_host reads the handle's marks back with its output: a stalled
    # gather comes back as VS_ERR_TIMEOUT from the call itself, once
    coo = W.random_coo(2000, 700, 50_000, seed=82, values="counts", sort=False)
    A = build(coo, "vcs", "row")
    B, Bt = dense_operand(coo, "A@B", 16, torch.float32)
    Bh = B.cpu().pin_memory()
    out = vs.empty_out(A, 16, "A@B", device="cpu", pin_memory=True)
    L.load().vs_test_stall_producers(1)
    with pytest.raises(L.VsError) as e:
        vs.spmm_host(A, Bh, "A@B", "deterministic", out=out)
    assert L.STATUS[e.value.status] == "VS_ERR_TIMEOUT"
    assert _status(A) == "VS_OK"                      # reported once
    vs.spmm_host(A, Bh, "A@B", "deterministic", out=out)
    want, D = oracle_product(coo, oracle_triples(coo, "vcs", "row"), "A@B", Bt)
    assert_close(out.double().numpy(), want, D, TOL[torch.float32], "after the timeout")
    A.destroy()
