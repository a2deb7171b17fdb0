"""Shared helpers of the GPU parity tests: oracle references and comparisons."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import workloads as W

# |gpu - oracle| <= TOL * sum|a||b| for every output element; exact 0 where that sum is 0.
TOL = {torch.float32: 1e-5, torch.float64: 1e-12}

PRODUCTS = [  # (layout, major, direction): the six products and their CSC relatives
    ("vcs", "row", "A@B"),   # VCSR@B   aligned
    ("vcs", "col", "A@B"),   # VCSC@B   misaligned
    ("vcs", "row", "B@A"),   # B@VCSR   misaligned
    ("vcs", "col", "B@A"),   # B@VCSC   aligned
    ("csr", "row", "A@B"),   # CSR@B    aligned
    ("csr", "row", "B@A"),   # B@CSR    misaligned
    ("csr", "col", "A@B"),   # CSC@B    misaligned
    ("csr", "col", "B@A"),   # B@CSC    aligned
]


@functools.lru_cache(maxsize=8)
def workload(name: str, seed: int = 0, dtype=torch.float32) -> W.Coo:
    """A named workload, generated once per test session (CPU tensors)."""
    return W.make(name, seed=seed, dtype=dtype)


def aligned(major: str, direction: str) -> bool:
    return (direction == "A@B") == (major == "row")


def build(coo: W.Coo, layout: str, major: str) -> vs.SparseMatrix:
    dev = torch.device("cuda")
    c = coo.to(dev)
    if layout == "vcs":
        return vs.build_vcs(c.rows, c.cols, c.vals, (coo.n_rows, coo.n_cols), major)
    return vs.build_csr(c.rows, c.cols, c.vals, (coo.n_rows, coo.n_cols), major)


def oracle_arrays(coo: W.Coo, layout: str, major: str) -> dict:
    r, c, v = coo.rows.cpu().numpy(), coo.cols.cpu().numpy(), coo.vals.cpu().numpy()
    maj, mnr = (r, c) if major == "row" else (c, r)
    nm, nn = (coo.n_rows, coo.n_cols) if major == "row" else (coo.n_cols, coo.n_rows)
    if layout == "vcs":
        mp, vals, vp, ind = oracle.vcs_build(nm, nn, maj, mnr, v)
        return {"ptr": mp, "values": vals, "value_ptr": vp, "indices": ind}
    ptr, idx, vals = oracle.csr_build(nm, nn, maj, mnr, v)
    return {"ptr": ptr, "indices": idx, "values": vals}


def oracle_triples(coo: W.Coo, layout: str, major: str):
    a = oracle_arrays(coo, layout, major)
    row = major == "row"
    if layout == "vcs":
        return oracle.vcs_triples(row, a["ptr"], a["values"], a["value_ptr"], a["indices"])
    return oracle.csr_triples(row, a["ptr"], a["indices"], a["values"])


def assert_arrays_equal(A: vs.SparseMatrix, want: dict) -> None:
    got = A.arrays()
    for k, w in want.items():
        g = got[k].cpu().numpy()
        assert g.dtype == w.dtype, (k, g.dtype, w.dtype)
        if g.dtype.kind == "f":
            g, w = g.view(np.uint32 if g.itemsize == 4 else np.uint64), \
                w.view(np.uint32 if w.itemsize == 4 else np.uint64)
        assert g.shape == w.shape, (k, g.shape, w.shape)
        if not np.array_equal(g, w):
            bad = np.nonzero(g != w)[0]
            raise AssertionError(f"{k}: {bad.size} mismatches, first at {bad[:5]}: "
                                 f"got {g[bad[:5]]} want {w[bad[:5]]}")


def dense_operand(coo: W.Coo, direction: str, w: int, dtype, seed=1, kind="normal"):
    """B for the product, on the device in the width-contiguous layout, plus B^T rows (n x w)."""
    n = coo.n_cols if direction == "A@B" else coo.n_rows
    Bt = W.dense(n, w, seed=seed, dtype=dtype, kind=kind)     # row-major n x w
    dev = Bt.to("cuda")
    B = dev if direction == "A@B" else dev.t()                # B@A takes w x n with stride(0)=1
    return B, Bt.to(torch.float64).numpy()


def oracle_product(coo: W.Coo, triples, direction: str, Bt_rows: np.ndarray):
    """Reference (out, D) in the (slice-frame) n_out x w layout."""
    ti, tj, ta = triples
    if direction == "A@B":
        return oracle.spmm_ab(coo.n_rows, coo.n_cols, ti, tj, ta, Bt_rows)
    out, D = oracle.spmm_ba(coo.n_rows, coo.n_cols, ti, tj, ta, Bt_rows.T)
    return out.T, D.T


def gpu_out_rows(out: torch.Tensor, direction: str) -> np.ndarray:
    o = out if direction == "A@B" else out.t()
    return o.detach().cpu().to(torch.float64).numpy()


def assert_close(got: np.ndarray, want: np.ndarray, D: np.ndarray, tol: float, what="") -> float:
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want)
    bound = tol * D
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond {tol}*D; first {i.tolist()}: "
                             f"got {got[bad][:5]} want {want[bad][:5]} D {D[bad][:5]}")
    assert np.all(got[D == 0] == 0), f"{what}: nonzero where the exact result is 0"
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(D > 0, err / np.where(D > 0, D, 1), 0)
    return float(rel.max()) if rel.size else 0.0
