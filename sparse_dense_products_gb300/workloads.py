"""Seeded synthetic inputs: COO triples and dense operands.

This module draws random numbers and lays them out as COO triples
``(row, col, val)`` and dense matrices.  It holds none of the product's
arithmetic and none of the layout construction: both the CUDA path and the
float64 oracle receive exactly the tensors produced here.

Every workload mirrors a shape the pages measure on:

* ``tiny``    -- 2,000 x 500 count matrix, row nnz NegBin(mean 10, r=2), columns
  uniform without replacement, values 1+Geometric(0.6) (support >= 1), dense
  width 8 (vsparse PR #61, "Testing": small CUDA parity cases).
* ``main``    -- 60,000 x 2,000 count matrix, row nnz NegBin(mean 100, r=2)
  clipped to 2,000, Zipf(1.1) column popularity sampled without replacement,
  values 1+Geometric(0.5), dense width 16 (vsparse PR #61, "Benchmarks":
  60k x 2k, 6M nonzeros, width 16).
* ``regrid``  -- 400,000 backprojection rows with {2,3,4} entries over 2,290
  columns whose expected lengths are log-uniform in [10, 3000]; weights U(0,1)
  normalised per row (regridding PR #70, "How it is built" and "Performance").
* ``large``   -- 1,000,000 x 20,000 count matrix, row nnz NegBin(mean 200, r=2),
  Zipf(1.1) columns, values 1+Geometric(0.5): about 200M nonzeros.
* ``skewed``  -- 500,000 x 500,000, row lengths Pareto(alpha=1.5, x_m=34)
  clipped to [1, 200,000] (about 50M nonzeros), columns uniform without
  replacement, values N(0,1).

Readings taken where the recipe is open:

* 1+Geometric(p) has support {1, 2, ...} with P(1) = p.
* NegBin(mean mu, r) is the Gamma(r, mu/r)-Poisson mixture; r = 2 is an
  integer, so the Gamma draw is the scaled sum of two unit exponentials.
* Sampling columns "without replacement, proportional to a weight" is
  successive sampling: draw with replacement from the weights and keep the
  first k distinct columns in draw order.
* COO triples are emitted sorted by (row, col); tests that need another input
  order permute them explicitly with :func:`permute`.

All generation runs through ``torch`` on the requested device with a
``torch.Generator`` seeded from ``seed``; the same (name, seed, device) always
gives the same tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = ["Coo", "CONFIGS", "make", "random_coo", "dense", "permute", "dense_width"]


@dataclass
class Coo:
    """COO triples of an ``n_rows x n_cols`` sparse matrix (int32 indices)."""

    n_rows: int
    n_cols: int
    rows: torch.Tensor
    cols: torch.Tensor
    vals: torch.Tensor

    @property
    def nnz(self) -> int:
        return int(self.rows.numel())

    def to(self, device) -> "Coo":
        return Coo(self.n_rows, self.n_cols, self.rows.to(device), self.cols.to(device),
                   self.vals.to(device))


# name -> (n_rows, n_cols, dense widths)
CONFIGS = {
    "tiny": (2_000, 500, (8,)),
    "main": (60_000, 2_000, (16,)),
    "regrid": (400_000, 2_290, (1, 4, 32)),
    "large": (1_000_000, 20_000, (8, 32)),
    "skewed": (500_000, 500_000, (64,)),
}


def dense_width(name: str) -> int:
    """The first (headline) dense width of a named workload."""
    return CONFIGS[name][2][0]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _negbin(n: int, mean: float, r: int, g: torch.Generator, device) -> torch.Tensor:
    """NegBin(mean, r) counts as a Gamma(r, mean/r)-Poisson mixture (integer r)."""
    e = torch.empty((n, r), dtype=torch.float64, device=device).exponential_(1.0, generator=g)
    lam = e.sum(dim=1) * (mean / r)
    return torch.poisson(lam, generator=g).to(torch.int64)


def _successive_sample(need: torch.Tensor, n_cols: int, cdf: torch.Tensor | None,
                       g: torch.Generator, device, block_entries: int = 1 << 24):
    """Per row r, ``need[r]`` distinct columns drawn without replacement.

    Columns are drawn with replacement (uniformly when ``cdf`` is None, else by
    inverting the cumulative weights ``cdf``) and the first ``need[r]`` distinct
    ones in draw order are kept.  Rows are handled in blocks so that memory
    stays bounded.  Returns (row, col) int64 tensors sorted by (row, col).
    """
    n_rows = need.numel()
    out_r, out_c = [], []
    csum = torch.cumsum(need, 0)
    start = 0
    while start < n_rows:
        # rows [start, stop) hold at most ~block_entries needed entries
        base = int(csum[start - 1]) if start > 0 else 0
        stop = int(torch.searchsorted(csum, torch.tensor(base + block_entries, device=device),
                                      right=True))
        stop = max(stop, start + 1)
        stop = min(stop, n_rows)
        r_need = need[start:stop]
        rows_local = torch.arange(stop - start, device=device)
        keys = torch.empty(0, dtype=torch.int64, device=device)   # row_local * n_cols + col
        pos = torch.empty(0, dtype=torch.int64, device=device)    # global draw position
        have = torch.zeros_like(r_need)
        pending = r_need > 0
        next_pos = 0
        done_r, done_c = [], []
        while bool(pending.any()):
            pr = rows_local[pending]
            deficit = (r_need[pending] - have[pending])
            m = deficit * 2 + 8
            rr = torch.repeat_interleave(pr, m)
            u = torch.rand(rr.numel(), dtype=torch.float64, device=device, generator=g)
            if cdf is None:
                c = torch.clamp((u * n_cols).to(torch.int64), max=n_cols - 1)
            else:
                c = torch.searchsorted(cdf, u * cdf[-1], right=True).clamp_(max=n_cols - 1)
            new_keys = rr * n_cols + c
            new_pos = next_pos + torch.arange(rr.numel(), device=device, dtype=torch.int64)
            next_pos += rr.numel()
            keys = torch.cat([keys, new_keys])
            pos = torch.cat([pos, new_pos])
            # first occurrence of each (row, col) in draw order
            kk, order = torch.sort(keys, stable=True)
            pp = pos[order]
            first = torch.ones_like(kk, dtype=torch.bool)
            first[1:] = kk[1:] != kk[:-1]
            fk, fp = kk[first], pp[first]
            frow = fk // n_cols
            have = torch.bincount(frow, minlength=stop - start)
            fin = (have >= r_need) & pending
            if bool(fin.any()):
                sel = fin[frow]
                fk2, fp2, frow2 = fk[sel], fp[sel], frow[sel]
                # rank of each distinct column within its row by draw position
                o2 = torch.argsort(frow2 * (next_pos + 1) + fp2)
                fk2, frow2 = fk2[o2], frow2[o2]
                row_start = torch.zeros(stop - start + 1, dtype=torch.int64, device=device)
                row_start[1:] = torch.cumsum(torch.bincount(frow2, minlength=stop - start), 0)
                rank = torch.arange(fk2.numel(), device=device) - row_start[frow2]
                keep = rank < r_need[frow2]
                done_r.append(frow2[keep] + start)
                done_c.append(fk2[keep] % n_cols)
            pending = pending & ~fin
            keep_draw = pending[keys // n_cols]
            keys, pos = keys[keep_draw], pos[keep_draw]
        if done_r:
            rr = torch.cat(done_r)
            cc = torch.cat(done_c)
            o = torch.argsort(rr * n_cols + cc)
            out_r.append(rr[o])
            out_c.append(cc[o])
        start = stop
    if not out_r:
        z = torch.empty(0, dtype=torch.int64, device=device)
        return z, z.clone()
    return torch.cat(out_r), torch.cat(out_c)


def _zipf_cdf(n_cols: int, s: float, device) -> torch.Tensor:
    k = torch.arange(1, n_cols + 1, dtype=torch.float64, device=device)
    return torch.cumsum(k.pow(-s), 0)


def make(name: str, seed: int = 0, device="cpu", dtype=torch.float32,
         rows: int | None = None) -> Coo:
    """COO triples of a named workload (see the module docstring).  ``rows``
    draws a smaller (or larger) matrix of the same recipe: the same columns and
    per-row distributions, that many rows."""
    if name not in CONFIGS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}")
    n_rows, n_cols, _ = CONFIGS[name]
    if rows is not None:
        n_rows = int(rows)
    g = _gen(seed, device)
    if name == "tiny":
        need = _negbin(n_rows, 10.0, 2, g, device).clamp_(0, n_cols)
        r, c = _successive_sample(need, n_cols, None, g, device)
        v = torch.empty(r.numel(), dtype=torch.float32, device=device).geometric_(0.6, generator=g)
    elif name in ("main", "large"):
        mean = 100.0 if name == "main" else 200.0
        need = _negbin(n_rows, mean, 2, g, device).clamp_(0, n_cols)
        r, c = _successive_sample(need, n_cols, _zipf_cdf(n_cols, 1.1, device), g, device)
        v = torch.empty(r.numel(), dtype=torch.float32, device=device).geometric_(0.5, generator=g)
    elif name == "regrid":
        need = torch.randint(2, 5, (n_rows,), generator=g, device=device, dtype=torch.int64)
        lo, hi = math.log(10.0), math.log(3000.0)
        lengths = torch.exp(lo + (hi - lo) * torch.rand(n_cols, dtype=torch.float64,
                                                         device=device, generator=g))
        r, c = _successive_sample(need, n_cols, torch.cumsum(lengths, 0), g, device)
        u = torch.rand(r.numel(), dtype=torch.float64, device=device, generator=g)
        rowsum = torch.zeros(n_rows, dtype=torch.float64, device=device).index_add_(0, r, u)
        v = (u / rowsum[r]).to(dtype)
    elif name == "skewed":
        u = torch.rand(n_rows, dtype=torch.float64, device=device, generator=g)
        need = torch.floor(34.0 * u.pow(-1.0 / 1.5)).clamp_(1, 200_000).to(torch.int64)
        r, c = _successive_sample(need, n_cols, None, g, device)
        v = torch.randn(r.numel(), dtype=torch.float32, device=device, generator=g)
    else:  # pragma: no cover
        raise AssertionError(name)
    if name != "regrid":
        v = v.to(dtype)
    return Coo(n_rows, n_cols, r.to(torch.int32), c.to(torch.int32), v)


def random_coo(n_rows: int, n_cols: int, nnz: int, seed: int = 0, device="cpu",
               dtype=torch.float32, values: str = "counts", duplicates: bool = False,
               empty_rows: float = 0.0, sort: bool = True) -> Coo:
    """Small random COO for parity and edge-case tests.

    ``values``: "counts" (1+Geometric(0.5)), "normal" (N(0,1)), "small_int"
    (integers in [-3, 3], exact in float32 sums), or "signed_zero" (a mix of
    +0.0, -0.0 and small integers).  ``duplicates`` allows repeated (row, col)
    pairs; ``empty_rows`` is the fraction of rows forced empty; ``sort``
    orders the triples by (row, col), otherwise they come in draw order.
    """
    g = _gen(seed, device)
    if n_rows == 0 or n_cols == 0 or nnz == 0:
        z = torch.empty(0, dtype=torch.int32, device=device)
        return Coo(n_rows, n_cols, z, z.clone(), torch.empty(0, dtype=dtype, device=device))
    allowed = torch.ones(n_rows, dtype=torch.bool, device=device)
    if empty_rows > 0:
        allowed = torch.rand(n_rows, generator=g, device=device) >= empty_rows
        if not bool(allowed.any()):
            allowed[0] = True
    row_pool = torch.nonzero(allowed).flatten()
    if duplicates:
        r = row_pool[torch.randint(0, row_pool.numel(), (nnz,), generator=g, device=device)]
        c = torch.randint(0, n_cols, (nnz,), generator=g, device=device)
    else:
        cap = row_pool.numel() * n_cols
        nnz = min(nnz, cap)
        flat = torch.randperm(cap, generator=g, device=device)[:nnz]
        r = row_pool[flat // n_cols]
        c = flat % n_cols
    if sort:
        o = torch.argsort(r.to(torch.int64) * n_cols + c, stable=True)
        r, c = r[o], c[o]
    n = r.numel()
    if values == "counts":
        v = torch.empty(n, dtype=torch.float64, device=device).geometric_(0.5, generator=g)
    elif values == "normal":
        v = torch.randn(n, dtype=torch.float64, device=device, generator=g)
    elif values == "small_int":
        v = torch.randint(-3, 4, (n,), generator=g, device=device).to(torch.float64)
    elif values == "signed_zero":
        k = torch.randint(0, 4, (n,), generator=g, device=device)
        v = torch.where(k == 0, torch.tensor(0.0, device=device, dtype=torch.float64),
                        torch.where(k == 1, torch.tensor(-0.0, device=device, dtype=torch.float64),
                                    k.to(torch.float64)))
    else:
        raise ValueError(values)
    return Coo(n_rows, n_cols, r.to(torch.int32), c.to(torch.int32), v.to(dtype))


def permute(coo: Coo, seed: int) -> Coo:
    """The same triples in a seeded random order."""
    g = _gen(seed, coo.rows.device)
    o = torch.randperm(coo.nnz, generator=g, device=coo.rows.device)
    return Coo(coo.n_rows, coo.n_cols, coo.rows[o], coo.cols[o], coo.vals[o])


def dense(rows: int, cols: int, seed: int = 1, device="cpu", dtype=torch.float32,
          kind: str = "normal") -> torch.Tensor:
    """A row-major dense operand: N(0,1) ("normal") or integers in [-4, 4] ("small_int")."""
    g = _gen(seed, device)
    if kind == "normal":
        return torch.randn(rows, cols, generator=g, device=device, dtype=torch.float64).to(dtype)
    if kind == "small_int":
        return torch.randint(-4, 5, (rows, cols), generator=g, device=device).to(dtype)
    raise ValueError(kind)
