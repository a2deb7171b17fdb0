"""The seeded generator: reproducible, well-formed COO with the stated shapes."""
import numpy as np
import torch

from sparse_dense_products_gb300 import workloads as W


def test_same_seed_same_tensors():
    a, b = W.make("tiny", seed=3), W.make("tiny", seed=3)
    assert torch.equal(a.rows, b.rows) and torch.equal(a.cols, b.cols) and torch.equal(a.vals, b.vals)
    c = W.make("tiny", seed=4)
    assert c.nnz != a.nnz or not torch.equal(a.cols, c.cols)


def test_tiny_shape_and_values():
    c = W.make("tiny")
    r, k, v = c.rows.numpy().astype(np.int64), c.cols.numpy().astype(np.int64), c.vals.numpy()
    assert c.n_rows == 2000 and c.n_cols == 500
    assert 15_000 < c.nnz < 25_000
    key = r * c.n_cols + k
    assert np.all(np.diff(key) > 0), "sorted by (row, col), no duplicates"
    assert r.min() >= 0 and r.max() < 2000 and k.min() >= 0 and k.max() < 500
    assert v.min() >= 1.0 and np.all(v == np.floor(v)), "1+Geometric counts"
    assert abs(float(np.mean(v == 1.0)) - 0.6) < 0.02


def test_regrid_rows_have_two_to_four_entries_and_sum_to_one():
    c = W.make("regrid", dtype=torch.float64)
    cnt = torch.bincount(c.rows.long(), minlength=c.n_rows)
    assert int(cnt.min()) == 2 and int(cnt.max()) == 4
    s = torch.zeros(c.n_rows, dtype=torch.float64).index_add_(0, c.rows.long(), c.vals)
    assert torch.allclose(s, torch.ones_like(s), atol=1e-12)


def test_random_coo_options():
    c = W.random_coo(10, 7, 50, seed=1, duplicates=True, sort=False, values="signed_zero")
    assert c.nnz == 50
    v = c.vals.numpy()
    assert np.any(np.signbit(v) & (v == 0)) and np.any(~np.signbit(v) & (v == 0))
    p = W.permute(c, seed=2)
    assert sorted(zip(p.rows.tolist(), p.cols.tolist())) == sorted(zip(c.rows.tolist(), c.cols.tolist()))
