"""Parity at full size: the 1,000,000 x 20,000 count matrix (~200M nonzeros, the
four VCS directions at widths 8 and 32) and the 500,000 x 500,000 power-law CSR
(~50M nonzeros, rows up to 200,000 entries, CSR@B and B@CSR at width 64).

The workloads are generated on the GPU and run through the same library calls
the benchmark makes.  The float64 oracle computes sampled output rows one by
one from the triples of those rows (random rows plus the longest ones, whose
long-slice share tree is the interesting case); the layouts are checked by
invariants that hold at any size and, for sampled slices, bit-exactly against
the oracle's build of those slices' entries.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_dense_products_gb300 as vs
from sparse_dense_products_gb300 import build as vs_build
from sparse_dense_products_gb300 import workloads as W

from gpu_helpers import TOL, assert_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_SAMPLE = 48


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device; none is visible"
    vs_build.build()


def _sample(lengths: torch.Tensor, k: int, seed: int) -> np.ndarray:
    """k distinct slice numbers: the 8 longest slices and random others."""
    n = lengths.numel()
    top = torch.topk(lengths, min(8, n)).indices
    g = torch.Generator(device="cpu").manual_seed(seed)
    rnd = torch.randperm(n, generator=g)[: k - top.numel()].to(lengths.device)
    sel = torch.unique(torch.cat([top, rnd]))
    return np.sort(sel.cpu().numpy().astype(np.int64))


def _triples_of(coo: W.Coo, major: str, sel: np.ndarray):
    """The triples whose major coordinate is in sel, in input order (host arrays)."""
    key = coo.rows if major == "row" else coo.cols
    mask = torch.isin(key, torch.as_tensor(sel, device=key.device, dtype=key.dtype))
    r, c, v = coo.rows[mask], coo.cols[mask], coo.vals[mask]
    return r.cpu().numpy(), c.cpu().numpy(), v.cpu().numpy()


def _check_layout_invariants(A: vs.SparseMatrix, nnz: int, vcs: bool):
    a = A.arrays()
    p = a["ptr"].to(torch.int64)
    assert int(p[0]) == 0 and bool((p[1:] >= p[:-1]).all())
    if vcs:
        vp = a["value_ptr"].to(torch.int64)
        R = a["values"].numel()
        assert int(p[-1]) == R and int(vp[0]) == 0 and int(vp[-1]) == nnz
        assert bool((vp[1:] > vp[:-1]).all()), "empty run"
    else:
        assert int(p[-1]) == nnz
    return a


def _check_sampled_slices(A_arrays: dict, coo: W.Coo, layout: str, major: str, sel: np.ndarray):
    """Slices sel of the GPU layout == the oracle's build of those slices' entries."""
    r, c, v = _triples_of(coo, major, sel)
    maj, mnr = (r, c) if major == "row" else (c, r)
    remap = np.searchsorted(sel, maj)  # sel is sorted: slice sel[k] becomes major k
    n_minor = coo.n_cols if major == "row" else coo.n_rows
    p = A_arrays["ptr"].cpu().numpy().astype(np.int64)
    if layout == "vcs":
        mp, vals, vp, ind = oracle.vcs_build(sel.size, n_minor, remap, mnr, v)
        gv = A_arrays["values"].cpu().numpy()
        gvp = A_arrays["value_ptr"].cpu().numpy().astype(np.int64)
        gi = A_arrays["indices"].cpu().numpy()
        for k, s in enumerate(sel):
            r0, r1 = p[s], p[s + 1]
            assert r1 - r0 == mp[k + 1] - mp[k], f"slice {s}: run count"
            assert np.array_equal(gv[r0:r1].view(np.uint32), vals[mp[k]:mp[k + 1]].view(np.uint32))
            lens_g = np.diff(gvp[r0:r1 + 1])
            lens_o = np.diff(vp[mp[k]:mp[k + 1] + 1])
            assert np.array_equal(lens_g, lens_o), f"slice {s}: run lengths"
            assert np.array_equal(gi[gvp[r0]:gvp[r1]], ind[vp[mp[k]]:vp[mp[k + 1]]]), f"slice {s}"
    else:
        op, oi, ov = oracle.csr_build(sel.size, n_minor, remap, mnr, v)
        gi = A_arrays["indices"].cpu().numpy()
        gv = A_arrays["values"].cpu().numpy()
        for k, s in enumerate(sel):
            e0, e1 = p[s], p[s + 1]
            assert e1 - e0 == op[k + 1] - op[k], f"slice {s}: entry count"
            assert np.array_equal(gi[e0:e1], oi[op[k]:op[k + 1]])
            assert np.array_equal(gv[e0:e1].view(np.uint32), ov[op[k]:op[k + 1]].view(np.uint32))


def _check_product(coo, A, direction, w, variants, sel_rows, sel_cols, seed):
    dev = torch.device("cuda")
    if direction == "A@B":
        X = W.dense(coo.n_cols, w, seed=seed, device=dev)
        B = X
        sel = sel_rows
        ti, tj, ta = _triples_of(coo, "row", sel)
        want, D = oracle.spmm_ab_rows(coo.n_rows, ti, tj, ta, X.double().cpu().numpy(), sel)
    else:
        Xt = W.dense(coo.n_rows, w, seed=seed, device=dev)   # B^T rows
        B = Xt.t()
        sel = sel_cols
        ti, tj, ta = _triples_of(coo, "col", sel)
        want, D = oracle.spmm_ba_cols(coo.n_cols, ti, tj, ta, Xt.double().cpu().numpy(), sel)
    idx = torch.as_tensor(sel, device=dev)
    for variant in variants:
        out = vs.spmm(A, B, direction, variant)
        rows = out.index_select(0, idx) if direction == "A@B" else out.index_select(1, idx).t()
        got = rows.double().cpu().numpy()
        assert_close(got, want, D, TOL[torch.float32], f"{direction} w={w} {variant}")
        if variant != "atomic":
            again = vs.spmm(A, B, direction, variant)
            assert torch.equal(again, out), f"{direction} w={w} {variant}: repeat differs"


def test_large_count_matrix_four_vcs_directions():
    coo = W.make("large", seed=0, device="cuda")
    assert coo.nnz > 150_000_000
    row_len = torch.bincount(coo.rows, minlength=coo.n_rows)
    col_len = torch.bincount(coo.cols, minlength=coo.n_cols)
    sel_rows = _sample(row_len, N_SAMPLE, 1)
    sel_cols = _sample(col_len, N_SAMPLE, 2)
    for major in ("row", "col"):
        A = vs.build_vcs(coo.rows, coo.cols, coo.vals, (coo.n_rows, coo.n_cols), major)
        arr = _check_layout_invariants(A, coo.nnz, vcs=True)
        _check_sampled_slices(arr, coo, "vcs", major, sel_rows if major == "row" else sel_cols)
        del arr
        A.attach_transpose()
        for direction in ("A@B", "B@A"):
            misaligned = (direction == "A@B") != (major == "row")
            variants = ["deterministic", "atomic", "two_phase"] if misaligned else ["deterministic"]
            for w in (8, 32):
                _check_product(coo, A, direction, w, variants, sel_rows, sel_cols, seed=10 + w)
        A.destroy()
        torch.cuda.empty_cache()


def test_skewed_power_law_csr_width_64():
    coo = W.make("skewed", seed=0, device="cuda")
    assert coo.nnz > 30_000_000
    row_len = torch.bincount(coo.rows, minlength=coo.n_rows)
    col_len = torch.bincount(coo.cols, minlength=coo.n_cols)
    assert int(row_len.max()) > 50_000          # the power-law tail is there
    sel_rows = _sample(row_len, N_SAMPLE, 3)
    sel_cols = _sample(col_len, N_SAMPLE, 4)
    A = vs.build_csr(coo.rows, coo.cols, coo.vals, (coo.n_rows, coo.n_cols), "row")
    arr = _check_layout_invariants(A, coo.nnz, vcs=False)
    _check_sampled_slices(arr, coo, "csr", "row", sel_rows)
    del arr
    _check_product(coo, A, "A@B", 64, ["deterministic"], sel_rows, sel_cols, seed=7)
    A.attach_transpose()
    _check_product(coo, A, "B@A", 64, ["deterministic", "atomic", "two_phase"], sel_rows, sel_cols,
                   seed=8)
    A.destroy()
