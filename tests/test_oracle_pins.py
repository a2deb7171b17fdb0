"""Pins of the float64 oracle against facts fixed outside the oracle itself.

Each test checks the oracle against something it cannot agree with by
construction: hand-worked examples (tests/golden/), brute force written here
in Python, closed forms (dense matmul with exact small integers, permutation
matrices), and invariants (the dot-product identity <A B, C> = <B, A^T C>,
multiset preservation, ordering).  The pages print no numeric example for the
products, so the golden files are worked by hand from the layout definitions.
"""
import json
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from sparse_dense_products_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(coo):
    return coo.rows.numpy(), coo.cols.numpy(), coo.vals.numpy()


def _total_order(v: float) -> int:
    """IEEE total-order key of a float32, computed with struct (independent of the oracle)."""
    (b,) = struct.unpack("<I", struct.pack("<f", v))
    return (~b) & 0xFFFFFFFF if b >> 31 else b | 0x80000000


def _dense(n_rows, n_cols, ti, tj, ta):
    A = np.zeros((n_rows, n_cols), np.float64)
    np.add.at(A, (ti, tj), ta)
    return A


# ----------------------------------------------------------------------------- golden


def test_golden_worked_example_layouts():
    g = json.load(open(os.path.join(GOLDEN, "vcs_worked_example.json")))
    r, c = np.array(g["coo_rows"]), np.array(g["coo_cols"])
    v = np.array(g["coo_vals"], np.float32)
    ptr, idx, vals = oracle.csr_build(g["n_rows"], g["n_cols"], r, c, v)
    assert ptr.tolist() == g["csr"]["ptr"] and idx.tolist() == g["csr"]["idx"]
    assert vals.tolist() == g["csr"]["vals"]
    ptr, idx, vals = oracle.csr_build(g["n_cols"], g["n_rows"], c, r, v)
    assert ptr.tolist() == g["csc"]["ptr"] and idx.tolist() == g["csc"]["idx"]
    assert vals.tolist() == g["csc"]["vals"]
    for key, (maj, mnr, nm, nn) in {"vcsr": (r, c, g["n_rows"], g["n_cols"]),
                                    "vcsc": (c, r, g["n_cols"], g["n_rows"])}.items():
        mp, values, vp, ind = oracle.vcs_build(nm, nn, maj, mnr, v)
        assert mp.tolist() == g[key]["major_ptr"], key
        assert values.tolist() == g[key]["values"], key
        assert vp.tolist() == g[key]["value_ptr"], key
        assert ind.tolist() == g[key]["indices"], key


@pytest.mark.parametrize("layout", ["csr", "csc", "vcsr", "vcsc"])
def test_golden_worked_example_products(layout):
    g = json.load(open(os.path.join(GOLDEN, "vcs_worked_example.json")))
    n_rows, n_cols = g["n_rows"], g["n_cols"]
    L = g[layout]
    row_major = layout in ("csr", "vcsr")
    if layout.startswith("v"):
        ti, tj, ta = oracle.vcs_triples(row_major, L["major_ptr"], L["values"], L["value_ptr"],
                                        L["indices"])
    else:
        ti, tj, ta = oracle.csr_triples(row_major, L["ptr"], L["idx"], L["vals"])
    out, _ = oracle.spmm_ab(n_rows, n_cols, ti, tj, ta, np.array(g["B_right"]))
    assert out.tolist() == g["A_times_B"]
    out, _ = oracle.spmm_ba(n_rows, n_cols, ti, tj, ta, np.array(g["B_left"]))
    assert out.tolist() == g["B_times_A"]


def test_golden_signed_zero_runs():
    g = json.load(open(os.path.join(GOLDEN, "vcs_signed_zero.json")))
    mp, values, vp, ind = oracle.vcs_build(g["n_rows"], g["n_cols"], g["coo_rows"], g["coo_cols"],
                                           np.array(g["coo_vals"], np.float32))
    assert mp.tolist() == g["vcsr"]["major_ptr"]
    assert vp.tolist() == g["vcsr"]["value_ptr"]
    assert ind.tolist() == g["vcsr"]["indices"]
    want = np.array(g["vcsr"]["values"], np.float32)
    assert values.view(np.uint32).tolist() == want.view(np.uint32).tolist()


# ----------------------------------------------------------------------------- assembly


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("major_is_row", [True, False])
def test_csr_build_is_stable_counting_sort(seed, major_is_row):
    coo = W.random_coo(37, 23, 300, seed=seed, duplicates=True, empty_rows=0.2, sort=False,
                       values="normal")
    r, c, v = _np(coo)
    maj, mnr = (r, c) if major_is_row else (c, r)
    n_major, n_minor = (37, 23) if major_is_row else (23, 37)
    ptr, idx, vals = oracle.csr_build(n_major, n_minor, maj, mnr, v)
    # brute force: each slice lists its entries in input order
    for m in range(n_major):
        pos = [t for t in range(len(maj)) if maj[t] == m]
        assert ptr[m + 1] - ptr[m] == len(pos)
        assert idx[ptr[m]:ptr[m + 1]].tolist() == [int(mnr[t]) for t in pos]
        assert vals[ptr[m]:ptr[m + 1]].view(np.uint32).tolist() == \
            v[pos].view(np.uint32).tolist()
    assert ptr[0] == 0 and ptr[-1] == len(maj)


def test_csr_keeps_input_order_under_permutation():
    coo = W.make("tiny")
    perm = W.permute(coo, seed=5)
    r, c, v = _np(perm)
    ptr, idx, vals = oracle.csr_build(coo.n_rows, coo.n_cols, r, c, v)
    # the i-th entry of row m is the i-th occurrence of row m in the permuted input
    order = np.argsort(r, kind="stable")
    assert idx.tolist() == c[order].tolist()
    assert vals.view(np.uint32).tolist() == v[order].view(np.uint32).tolist()


def _vcs_bruteforce(n_major, maj, mnr, vals):
    runs = {}
    for t in range(len(maj)):
        runs.setdefault(int(maj[t]), {}).setdefault(_total_order(float(vals[t])), []).append(
            (int(mnr[t]), t))
    major_ptr, values, value_ptr, indices = [0], [], [0], []
    for m in range(n_major):
        for key in sorted(runs.get(m, {})):
            members = sorted(runs[m][key])          # ascending minor, then input position
            values.append(vals[members[0][1]])
            indices.extend(mn for mn, _ in members)
            value_ptr.append(len(indices))
        major_ptr.append(len(values))
    return major_ptr, np.array(values, np.float32), value_ptr, indices


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("values", ["counts", "signed_zero", "normal"])
def test_vcs_build_matches_bruteforce(seed, values):
    coo = W.random_coo(29, 31, 400, seed=seed, duplicates=True, empty_rows=0.15, sort=False,
                       values=values)
    r, c, v = _np(coo)
    for maj, mnr, nm, nn in ((r, c, 29, 31), (c, r, 31, 29)):
        mp, vals, vp, ind = oracle.vcs_build(nm, nn, maj, mnr, v)
        bmp, bvals, bvp, bind = _vcs_bruteforce(nm, maj, mnr, v)
        assert mp.tolist() == bmp
        assert vals.view(np.uint32).tolist() == bvals.view(np.uint32).tolist()
        assert vp.tolist() == bvp
        assert ind.tolist() == bind


def test_vcs_invariants_on_tiny_workload():
    coo = W.make("tiny")
    r, c, v = _np(coo)
    for maj, mnr, nm in ((r, c, coo.n_rows), (c, r, coo.n_cols)):
        mp, vals, vp, ind = oracle.vcs_build(nm, 10 ** 6, maj, mnr, v)
        R = vals.size
        assert mp[0] == 0 and mp[-1] == R and np.all(np.diff(mp) >= 0)
        assert vp[0] == 0 and vp[-1] == coo.nnz and np.all(np.diff(vp) > 0)
        keys = np.array([_total_order(float(x)) for x in vals], np.int64)
        for m in range(nm):
            seg = keys[mp[m]:mp[m + 1]]
            assert np.all(np.diff(seg) > 0), "values must strictly increase inside a slice"
        for rr in range(R):
            assert np.all(np.diff(ind[vp[rr]:vp[rr + 1]]) >= 0)
        # the multiset of (major, minor, value) is preserved
        ti, tj, ta = oracle.vcs_triples(True, mp, vals, vp, ind)
        got = sorted(zip(ti.tolist(), tj.tolist(), ta.tolist()))
        want = sorted(zip(maj.tolist(), mnr.tolist(), v.astype(np.float64).tolist()))
        assert got == want


def test_vcs_is_independent_of_input_order():
    coo = W.make("tiny")
    a = oracle.vcs_build(coo.n_rows, coo.n_cols, *_np(coo))
    b = oracle.vcs_build(coo.n_rows, coo.n_cols, *_np(W.permute(coo, seed=9)))
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32) if x.dtype == np.float32 else x,
                              y.view(np.uint32) if y.dtype == np.float32 else y)


def test_assembly_rejects_bad_input():
    with pytest.raises(oracle.OracleError):
        oracle.csr_build(3, 3, [0, 3], [0, 0], np.ones(2, np.float32))
    with pytest.raises(oracle.OracleError):
        oracle.csr_build(3, 3, [0, 1], [0, -1], np.ones(2, np.float32))
    with pytest.raises(oracle.OracleError):
        oracle.vcs_build(3, 3, [0, 1], [0, 1], np.array([1.0, np.nan], np.float32))


# ----------------------------------------------------------------------------- products


def _all_layout_triples(coo):
    """Triples of the same matrix through all four oracle layouts."""
    r, c, v = _np(coo)
    out = {}
    ptr, idx, vals = oracle.csr_build(coo.n_rows, coo.n_cols, r, c, v)
    out["csr"] = oracle.csr_triples(True, ptr, idx, vals)
    ptr, idx, vals = oracle.csr_build(coo.n_cols, coo.n_rows, c, r, v)
    out["csc"] = oracle.csr_triples(False, ptr, idx, vals)
    if v.dtype == np.float32:
        out["vcsr"] = oracle.vcs_triples(True, *oracle.vcs_build(coo.n_rows, coo.n_cols, r, c, v))
        out["vcsc"] = oracle.vcs_triples(False, *oracle.vcs_build(coo.n_cols, coo.n_rows, c, r, v))
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_products_equal_dense_matmul_exactly(seed):
    # small integers: every partial sum is exact in float64, so equality is exact
    coo = W.random_coo(41, 19, 250, seed=seed, duplicates=True, empty_rows=0.2,
                       values="small_int", sort=False)
    r, c, v = _np(coo)
    A = np.zeros((41, 19), np.int64)
    np.add.at(A, (r, c), v.astype(np.int64))
    Aabs = np.zeros((41, 19), np.int64)      # D sums |a| per stored entry, duplicates apart
    np.add.at(Aabs, (r, c), np.abs(v.astype(np.int64)))
    B = W.dense(19, 7, seed=3, kind="small_int").numpy().astype(np.int64)
    Bl = W.dense(5, 41, seed=4, kind="small_int").numpy().astype(np.int64)
    for name, (ti, tj, ta) in _all_layout_triples(coo).items():
        out, D = oracle.spmm_ab(41, 19, ti, tj, ta, B)
        assert np.array_equal(out, (A @ B).astype(np.float64)), name
        assert np.array_equal(D, (Aabs @ np.abs(B)).astype(np.float64)), name
        out, D = oracle.spmm_ba(41, 19, ti, tj, ta, Bl)
        assert np.array_equal(out, (Bl @ A).astype(np.float64)), name
        assert np.array_equal(D, (np.abs(Bl) @ Aabs).astype(np.float64)), name


def test_dot_product_identity():
    # <A X, C> = <X, A^T C>, with A^T C computed as (C^T A)^T by the B.A product
    coo = W.random_coo(300, 170, 4000, seed=7, values="normal")
    rng = np.random.default_rng(0)
    X = rng.standard_normal((170, 6))
    C = rng.standard_normal((300, 6))
    for name, (ti, tj, ta) in _all_layout_triples(coo).items():
        AX, _ = oracle.spmm_ab(300, 170, ti, tj, ta, X)
        CtA, _ = oracle.spmm_ba(300, 170, ti, tj, ta, C.T)
        lhs, rhs = float(np.sum(AX * C)), float(np.sum(X * CtA.T))
        assert abs(lhs - rhs) <= 1e-12 * (np.sum(np.abs(AX) * np.abs(C)) + 1.0), name


def test_permutation_matrix_permutes_exactly():
    n = 64
    perm = np.random.default_rng(1).permutation(n)
    coo = W.Coo(n, n, torch.arange(n, dtype=torch.int32), torch.tensor(perm, dtype=torch.int32),
                torch.ones(n, dtype=torch.float32))
    B = np.random.default_rng(2).standard_normal((n, 5))
    for name, (ti, tj, ta) in _all_layout_triples(coo).items():
        out, _ = oracle.spmm_ab(n, n, ti, tj, ta, B)
        assert np.array_equal(out, B[perm]), name
        out, _ = oracle.spmm_ba(n, n, ti, tj, ta, B.T)
        inv = np.argsort(perm)
        assert np.array_equal(out, B.T[:, inv]), name


def test_empty_rows_zero_width_and_empty_matrix():
    coo = W.random_coo(50, 30, 200, seed=3, empty_rows=0.5)
    r = coo.rows.numpy()
    empty = np.setdiff1d(np.arange(50), r)
    assert empty.size > 0
    for name, (ti, tj, ta) in _all_layout_triples(coo).items():
        out, _ = oracle.spmm_ab(50, 30, ti, tj, ta, np.ones((30, 3)))
        assert np.all(out[empty] == 0.0), name
        out, D = oracle.spmm_ab(50, 30, ti, tj, ta, np.ones((30, 0)))
        assert out.shape == (50, 0) and D.shape == (50, 0)
        out, _ = oracle.spmm_ba(50, 30, ti, tj, ta, np.ones((0, 50)))
        assert out.shape == (0, 30)
    z = np.zeros(0, np.int32)
    out, _ = oracle.spmm_ab(4, 3, z, z, np.zeros(0), np.ones((3, 2)))
    assert np.array_equal(out, np.zeros((4, 2)))
    ptr, idx, vals = oracle.csr_build(4, 3, z, z, np.zeros(0, np.float32))
    assert ptr.tolist() == [0, 0, 0, 0, 0] and idx.size == 0
    mp, values, vp, ind = oracle.vcs_build(4, 3, z, z, np.zeros(0, np.float32))
    assert mp.tolist() == [0] * 5 and values.size == 0 and vp.tolist() == [0]


def test_duplicates_are_summed():
    coo = W.Coo(2, 3, torch.tensor([0, 0, 0, 1], dtype=torch.int32),
                torch.tensor([1, 1, 2, 0], dtype=torch.int32),
                torch.tensor([2.0, 3.0, 1.0, 4.0]))
    B = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0]])
    for name, (ti, tj, ta) in _all_layout_triples(coo).items():
        out, _ = oracle.spmm_ab(2, 3, ti, tj, ta, B)
        assert out.tolist() == [[150.0, 300.0], [4.0, 8.0]], name


def test_vcs_and_csr_products_agree_on_workload():
    coo = W.make("tiny")
    B = W.dense(coo.n_cols, 8, seed=1).numpy()
    Bl = W.dense(8, coo.n_rows, seed=2).numpy()
    res = {}
    for name, (ti, tj, ta) in _all_layout_triples(coo).items():
        res[name] = (oracle.spmm_ab(coo.n_rows, coo.n_cols, ti, tj, ta, B)[0],
                     oracle.spmm_ba(coo.n_rows, coo.n_cols, ti, tj, ta, Bl)[0])
    A = _dense(coo.n_rows, coo.n_cols, coo.rows.numpy(), coo.cols.numpy(),
               coo.vals.numpy().astype(np.float64))
    for name, (ab, ba) in res.items():
        assert np.allclose(ab, A @ B.astype(np.float64), rtol=1e-12, atol=1e-12), name
        assert np.allclose(ba, Bl.astype(np.float64) @ A, rtol=1e-12, atol=1e-12), name


def test_sampled_products_match_full():
    coo = W.random_coo(120, 90, 2000, seed=11, values="normal", duplicates=True)
    r, c, v = _np(coo)
    B = W.dense(90, 5, seed=1).numpy()
    Bt = W.dense(120, 5, seed=2).numpy()
    full, Dfull = oracle.spmm_ab(120, 90, r, c, v, B)
    sel = np.array([0, 5, 119, 64])
    part, Dpart = oracle.spmm_ab_rows(120, r, c, v, B, sel)
    assert np.array_equal(part, full[sel]) and np.array_equal(Dpart, Dfull[sel])
    full, Dfull = oracle.spmm_ba(120, 90, r, c, v, Bt.T)
    sel = np.array([89, 0, 33])
    part, Dpart = oracle.spmm_ba_cols(90, r, c, v, Bt, sel)
    assert np.array_equal(part, full[:, sel].T) and np.array_equal(Dpart, Dfull[:, sel].T)


# ----------------------------------------------------------------------------- views


def test_golden_view_worked_example():
    """view_triples against the hand-worked view example, every map, with both
    scalings and with the row scaling alone."""
    g = json.load(open(os.path.join(GOLDEN, "view_worked_example.json")))
    ti, tj, ta = np.array(g["ti"]), np.array(g["tj"]), np.array(g["ta"])
    r, c = np.array(g["row_scale"]), np.array(g["col_scale"])
    for name, want in g["views"].items():
        _, _, got = oracle.view_triples(ti, tj, ta, name, r, c)
        np.testing.assert_allclose(got, want, rtol=1e-15, atol=0, err_msg=name)
    for name, want in g["views_row_scale_only"].items():
        _, _, got = oracle.view_triples(ti, tj, ta, name, r, None)
        np.testing.assert_allclose(got, want, rtol=1e-15, atol=0, err_msg=name)
    _, _, a = oracle.view_triples(ti, tj, ta, "sqrt", r, c)
    out, _ = oracle.spmm_ab(g["n_rows"], g["n_cols"], ti, tj, a, np.array(g["B"]))
    assert out.tolist() == g["sqrt_view_times_B"]


def test_view_closed_forms():
    """Identity without scalings returns the values; power-of-two scalings are
    exact; the column scaling of A equals scaling the rows of B (and the row
    scaling of A equals scaling the output rows) in a product."""
    coo = W.make("tiny", seed=3)
    ti, tj, ta = oracle.csr_triples(True, *oracle.csr_build(coo.n_rows, coo.n_cols, *_np(coo)))
    assert np.array_equal(oracle.view_triples(ti, tj, ta)[2], ta)
    rng = np.random.default_rng(5)
    r = 2.0 ** rng.integers(-3, 4, coo.n_rows)
    c = 2.0 ** rng.integers(-3, 4, coo.n_cols)
    _, _, a = oracle.view_triples(ti, tj, ta, "identity", r, c)
    assert np.array_equal(a, ta * r[ti] * c[tj])
    B = rng.integers(-3, 4, (coo.n_cols, 5)).astype(np.float64)
    rs = rng.integers(1, 4, coo.n_rows).astype(np.float64)
    cs = rng.integers(1, 4, coo.n_cols).astype(np.float64)
    _, _, av = oracle.view_triples(ti, tj, ta, "identity", rs, cs)
    got, _ = oracle.spmm_ab(coo.n_rows, coo.n_cols, ti, tj, av, B)
    want = rs[:, None] * (_dense(coo.n_rows, coo.n_cols, ti, tj, ta) @ (cs[:, None] * B))
    assert np.array_equal(got, want)  # small integers: every sum is exact
    # the maps against numpy's own log1p / sqrt on the stored values
    for name, f in (("log1p", np.log1p), ("sqrt", np.sqrt)):
        np.testing.assert_allclose(oracle.view_triples(ti, tj, ta, name)[2], f(ta), rtol=1e-15)


# ----------------------------------------------------------------------------- threaded products


def _frames(coo):
    """(label, ptr, idx, vals, value_ptr, n_major, n_minor, triples) of the four layouts."""
    r, c, v = _np(coo)
    out = []
    for major in ("row", "col"):
        maj, mnr = (r, c) if major == "row" else (c, r)
        nm, nn = (coo.n_rows, coo.n_cols) if major == "row" else (coo.n_cols, coo.n_rows)
        p, i, vv = oracle.csr_build(nm, nn, maj, mnr, v)
        out.append((f"csr/{major}", p, i, vv, None, nm, nn,
                    oracle.csr_triples(major == "row", p, i, vv)))
        mp, vals, vp, ind = oracle.vcs_build(nm, nn, maj, mnr, v)
        out.append((f"vcs/{major}", mp, ind, vals, vp, nm, nn,
                    oracle.vcs_triples(major == "row", mp, vals, vp, ind)))
    return out


def _serial_frame(coo, major_is_row, aligned, tri, X):
    """The serial products of the triples, in the slice frame of a layout."""
    ti, tj, ta = tri
    # slice frame: aligned products with a row major are A @ X; with a column
    # major they are A^T @ X (= (X^T A)^T); misaligned ones the other way round
    if major_is_row == aligned:
        return oracle.spmm_ab(coo.n_rows, coo.n_cols, ti, tj, ta, X)
    out, D = oracle.spmm_ba(coo.n_rows, coo.n_cols, ti, tj, ta, np.ascontiguousarray(X.T))
    return out.T, D.T


@pytest.mark.parametrize("threads", [1, 3, 8])
def test_threaded_products_match_serial(threads):
    """Aligned frames: bit-identical to the serial products (each output row is
    summed in entry order either way).  Misaligned frames: within 1e-12 * D of
    the serial products, and bit-identical on one thread."""
    coo = W.make("tiny", seed=7)
    rng = np.random.default_rng(threads)
    for label, p, i, vals, vp, nm, nn, tri in _frames(coo):
        row = label.endswith("row")
        for aligned in (True, False):
            X = rng.standard_normal((nn if aligned else nm, 6))
            got, gD = oracle.spmm_slices(p, i, vals, X, aligned, nn, vp, threads)
            want, wD = _serial_frame(coo, row, aligned, tri, X)
            if aligned or threads == 1:
                assert np.array_equal(got, want), (label, aligned)
                assert np.array_equal(gD, wD), (label, aligned)
            else:
                assert np.all(np.abs(got - want) <= 1e-12 * wD), (label, aligned)
                assert np.allclose(gD, wD, rtol=1e-12, atol=0), (label, aligned)


def test_threaded_products_equal_dense_matmul_exactly():
    """Small-integer operands: every partial sum is exact, so each frame equals
    numpy's integer matmul of the dense matrix bit for bit, at any thread count."""
    coo = W.random_coo(300, 170, 4000, seed=12, duplicates=True, sort=False)
    A = _dense(coo.n_rows, coo.n_cols, coo.rows.numpy(), coo.cols.numpy(),
               coo.vals.numpy().astype(np.float64))
    rng = np.random.default_rng(1)
    for label, p, i, vals, vp, nm, nn, _ in _frames(coo):
        M = A if label.endswith("row") else A.T          # n_major x n_minor
        for aligned in (True, False):
            X = rng.integers(-4, 5, (nn if aligned else nm, 5)).astype(np.float64)
            want = M @ X if aligned else M.T @ X
            for threads in (1, 4, 7):
                got, _ = oracle.spmm_slices(p, i, vals, X, aligned, nn, vp, threads)
                assert np.array_equal(got, want), (label, aligned, threads)
