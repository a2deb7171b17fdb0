"""The float64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and it
shares no code with the CUDA library.  The arithmetic lives in
``vs_oracle.c`` (plain C, float64, ``-ffp-contract=off``); this module compiles
it with gcc into ``oracle/_build/`` and marshals numpy arrays in and out.

Functions and the passages they follow:

* :func:`csr_build` -- counting-sort assembly ("Regridder", "How it is built").
* :func:`vcs_build` -- value-grouped VCS arrays ("Add CUDA transfer and matmul
  kernels for the normalized views", "The layout stays compressed").
* :func:`csr_triples`, :func:`vcs_triples` -- layout back to (i, j, a) triples.
* :func:`spmm_ab`, :func:`spmm_ba` -- out = A B and out = B A in float64, with
  the per-element error scale D = sum |a| |b|.
* :func:`spmm_ab_rows`, :func:`spmm_ba_cols` -- the same for a sample of output
  rows (resp. columns), for matrices too large for a full product.
* :func:`view_triples` -- the triples of a normalized view
  diag(row_scale) g(A) diag(col_scale) ("Add CUDA transfer and matmul kernels
  for the normalized views", "The layout stays compressed").
* :func:`spmm_slices` -- the products over a stored layout on several host
  threads (same page, "The kernels": whole slices per thread where the output
  is aligned with the slices, per-thread private outputs merged in thread order
  where it is not); the host cores' baseline.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vs_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libvs_oracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {-1: "index out of range", -2: "NaN value", -3: "allocation failed",
          -4: "invalid argument"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compiles vs_oracle.c with gcc (no fused multiply-add) and returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-fopenmp", _SRC, "-o", tmp, "-lm"]
    if subprocess.run(cmd).returncode != 0:
        # no OpenMP runtime: the same source, one thread
        cmd.remove("-fopenmp")
        subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(lib):
    """Declares the C signatures on a loaded oracle library."""
    i64, i32p, vp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.or_csr_build.restype = ctypes.c_int
    lib.or_csr_build.argtypes = [i64, i64, i64, i32p, i32p, vp, i64, i32p, i32p, vp]
    lib.or_vcs_build.restype = ctypes.c_int64
    lib.or_vcs_build.argtypes = [i64, i64, i64, i32p, i32p, vp, i32p, vp, i32p, i32p]
    lib.or_csr_triples.restype = None
    lib.or_csr_triples.argtypes = [i64, ctypes.c_int, i32p, i32p, vp, i32p, i32p, vp]
    lib.or_vcs_triples.restype = None
    lib.or_vcs_triples.argtypes = [i64, ctypes.c_int, i32p, vp, i32p, i32p, i32p, i32p, vp]
    for name in ("or_spmm_ab", "or_spmm_ba"):
        f = getattr(lib, name)
        f.restype = None
        f.argtypes = [i64, i64, i64, i32p, i32p, vp, vp, i64, i64, vp, vp, i64]
    for name in ("or_spmm_ab_rows", "or_spmm_ba_cols"):
        f = getattr(lib, name)
        f.restype = None
        f.argtypes = [i64, i64, i32p, i32p, vp, vp, i64, i64, i64, vp, vp, vp, vp]
    lib.or_view_triples.restype = ctypes.c_int
    lib.or_view_triples.argtypes = [i64, i32p, i32p, vp, ctypes.c_int, vp, vp, vp]
    lib.or_threads_available.restype = ctypes.c_int
    lib.or_threads_available.argtypes = []
    lib.or_spmm_slices.restype = ctypes.c_int
    lib.or_spmm_slices.argtypes = [i64, i64, i32p, i32p, i32p, vp, ctypes.c_int, vp, i64, vp, vp,
                                   ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


class use_library:
    """Test hook: run the oracle functions on another build of vs_oracle.c (a
    copy with a planted mistake, to check that the pins catch it)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        with _lock:
            self.saved = _lib
            _lib = _configure(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _check(code: int):
    if code < 0:
        raise OracleError(ERRORS.get(int(code), f"error {code}"))


def csr_build(n_major: int, n_minor: int, major, minor, vals):
    """Counting-sort CSR (major = rows) or CSC (major = columns) of COO entries.

    Returns (ptr int32[n_major+1], idx int32[nnz], vals[nnz]); values keep their
    dtype and bits.  A slice keeps its entries in input order.
    """
    lib = _load()
    major, minor = _i32(major), _i32(minor)
    vals = np.ascontiguousarray(vals)
    nnz = major.size
    if minor.size != nnz or vals.size != nnz:
        raise OracleError("length mismatch")
    ptr = np.zeros(n_major + 1, dtype=np.int32)
    idx = np.zeros(max(nnz, 1), dtype=np.int32)
    out = np.zeros(max(nnz, 1), dtype=vals.dtype)
    _check(lib.or_csr_build(n_major, n_minor, nnz, _p(major), _p(minor), _p(vals),
                            vals.dtype.itemsize, _p(ptr), _p(idx), _p(out)))
    return ptr, idx[:nnz], out[:nnz]


def vcs_build(n_major: int, n_minor: int, major, minor, vals):
    """VCS arrays (major_ptr, values float32[R], value_ptr int32[R+1], indices)."""
    lib = _load()
    major, minor = _i32(major), _i32(minor)
    vals = np.ascontiguousarray(vals, dtype=np.float32)
    nnz = major.size
    if minor.size != nnz or vals.size != nnz:
        raise OracleError("length mismatch")
    major_ptr = np.zeros(n_major + 1, dtype=np.int32)
    values = np.zeros(max(nnz, 1), dtype=np.float32)
    value_ptr = np.zeros(nnz + 1, dtype=np.int32)
    indices = np.zeros(max(nnz, 1), dtype=np.int32)
    R = lib.or_vcs_build(n_major, n_minor, nnz, _p(major), _p(minor), _p(vals), _p(major_ptr),
                         _p(values), _p(value_ptr), _p(indices))
    _check(R)
    return major_ptr, values[:R].copy(), value_ptr[:R + 1].copy(), indices[:nnz]


def csr_triples(major_is_row: bool, ptr, idx, vals):
    """(i, j, a) triples of a CSR/CSC in layout order (a as float64)."""
    lib = _load()
    ptr, idx = _i32(ptr), _i32(idx)
    vals = np.ascontiguousarray(vals, dtype=np.float64)
    nnz = idx.size
    ti = np.zeros(max(nnz, 1), np.int32)
    tj = np.zeros(max(nnz, 1), np.int32)
    ta = np.zeros(max(nnz, 1), np.float64)
    lib.or_csr_triples(ptr.size - 1, int(bool(major_is_row)), _p(ptr), _p(idx), _p(vals),
                       _p(ti), _p(tj), _p(ta))
    return ti[:nnz], tj[:nnz], ta[:nnz]


def vcs_triples(major_is_row: bool, major_ptr, values, value_ptr, indices):
    """(i, j, a) triples of a VCSR/VCSC in layout order (a as float64)."""
    lib = _load()
    major_ptr, value_ptr, indices = _i32(major_ptr), _i32(value_ptr), _i32(indices)
    values = np.ascontiguousarray(values, dtype=np.float32)
    nnz = indices.size
    ti = np.zeros(max(nnz, 1), np.int32)
    tj = np.zeros(max(nnz, 1), np.int32)
    ta = np.zeros(max(nnz, 1), np.float64)
    lib.or_vcs_triples(major_ptr.size - 1, int(bool(major_is_row)), _p(major_ptr), _p(values),
                       _p(value_ptr), _p(indices), _p(ti), _p(tj), _p(ta))
    return ti[:nnz], tj[:nnz], ta[:nnz]


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.float64)


def spmm_ab(n_rows: int, n_cols: int, ti, tj, ta, B):
    """out = A B (float64) and D = sum |a||b|; B is n_cols x w."""
    lib = _load()
    ti, tj, ta, B = _i32(ti), _i32(tj), _f64(ta), _f64(B)
    if B.ndim != 2 or B.shape[0] != n_cols:
        raise OracleError("B must be n_cols x w")
    w = B.shape[1]
    out = np.zeros((n_rows, w), np.float64)
    D = np.zeros((n_rows, w), np.float64)
    lib.or_spmm_ab(n_rows, n_cols, ti.size, _p(ti), _p(tj), _p(ta), _p(B), w, w, _p(out), _p(D), w)
    return out, D


def spmm_ba(n_rows: int, n_cols: int, ti, tj, ta, B):
    """out = B A (float64) and D = sum |b||a|; B is w x n_rows."""
    lib = _load()
    ti, tj, ta, B = _i32(ti), _i32(tj), _f64(ta), _f64(B)
    if B.ndim != 2 or B.shape[1] != n_rows:
        raise OracleError("B must be w x n_rows")
    w = B.shape[0]
    out = np.zeros((w, n_cols), np.float64)
    D = np.zeros((w, n_cols), np.float64)
    lib.or_spmm_ba(n_rows, n_cols, ti.size, _p(ti), _p(tj), _p(ta), _p(B), n_rows, w, _p(out),
                   _p(D), n_cols)
    return out, D


def spmm_ab_rows(n_rows: int, ti, tj, ta, B, sel):
    """Rows ``sel`` of A B: returns (out, D), each len(sel) x w."""
    lib = _load()
    ti, tj, ta, B = _i32(ti), _i32(tj), _f64(ta), _f64(B)
    sel = np.ascontiguousarray(sel, dtype=np.int64)
    if sel.size and (sel.min() < 0 or sel.max() >= n_rows or np.unique(sel).size != sel.size):
        raise OracleError("sel must be distinct rows in range")
    w = B.shape[1]
    slot = np.zeros(max(n_rows, 1), np.int64)
    out = np.zeros((sel.size, w), np.float64)
    D = np.zeros((sel.size, w), np.float64)
    lib.or_spmm_ab_rows(n_rows, ti.size, _p(ti), _p(tj), _p(ta), _p(B), B.shape[1], w, sel.size,
                        _p(sel), _p(slot), _p(out), _p(D))
    return out, D


def spmm_ba_cols(n_cols: int, ti, tj, ta, Bt, sel):
    """Columns ``sel`` of B A with B given TRANSPOSED (``Bt`` = B^T, n_rows x w).

    Returns (out, D) with row s holding output column sel[s] (len(sel) x w).
    """
    lib = _load()
    ti, tj, ta = _i32(ti), _i32(tj), _f64(ta)
    B = _f64(np.asarray(Bt).T)          # w x n_rows, the layout the C function expects
    sel = np.ascontiguousarray(sel, dtype=np.int64)
    if sel.size and (sel.min() < 0 or sel.max() >= n_cols or np.unique(sel).size != sel.size):
        raise OracleError("sel must be distinct columns in range")
    w = B.shape[0]
    slot = np.zeros(max(n_cols, 1), np.int64)
    out = np.zeros((sel.size, w), np.float64)
    D = np.zeros((sel.size, w), np.float64)
    lib.or_spmm_ba_cols(n_cols, ti.size, _p(ti), _p(tj), _p(ta), _p(B), B.shape[1], w, sel.size,
                        _p(sel), _p(slot), _p(out), _p(D))
    return out, D


MAPS = {"identity": 0, "log1p": 1, "sqrt": 2}


def view_triples(ti, tj, ta, map: str = "identity", row_scale=None, col_scale=None):
    """Triples of the view diag(row_scale) g(A) diag(col_scale): (ti, tj, a') with
    a' = row_scale[i] * g(a) * col_scale[j] in float64 (None: all ones)."""
    lib = _load()
    ti, tj, ta = _i32(ti), _i32(tj), _f64(ta)
    rs = None if row_scale is None else _f64(row_scale)
    cs = None if col_scale is None else _f64(col_scale)
    if rs is not None and ti.size and int(ti.max()) >= rs.size:
        raise OracleError("row_scale shorter than the rows")
    if cs is not None and tj.size and int(tj.max()) >= cs.size:
        raise OracleError("col_scale shorter than the columns")
    out = np.zeros(max(ta.size, 1), np.float64)
    _check(lib.or_view_triples(ta.size, _p(ti), _p(tj), _p(ta), MAPS[map],
                               None if rs is None else _p(rs), None if cs is None else _p(cs),
                               _p(out)))
    return ti, tj, out[:ta.size]


def threads_available() -> int:
    """Threads the threaded oracle products use by default (1 without OpenMP)."""
    return int(_load().or_threads_available())


def spmm_slices(ptr, idx, vals, X, aligned: bool, n_minor: int, value_ptr=None,
                threads: int = 0):
    """The product over a stored layout in the slice frame, on ``threads`` host
    threads (0: all OpenMP offers).

    ``ptr`` (n_major+1) indexes entries (CSR) or runs (VCS, with ``value_ptr``);
    ``vals`` holds one value per entry (CSR) or per run (VCS).
    aligned:   Y[s] = sum a X[t] over the entries (t, a) of slice s; X is n_minor x w.
    misaligned: Y[t] = sum a X[s]; X is n_major x w, Y is n_minor x w.
    Returns (Y, D), D = sum |a||x| per element.
    """
    lib = _load()
    ptr, idx = _i32(ptr), _i32(idx)
    vals = _f64(vals)
    vp_ = None if value_ptr is None else _i32(value_ptr)
    X = _f64(X)
    n_major = ptr.size - 1
    w = X.shape[1]
    if X.shape[0] != (n_minor if aligned else n_major):
        raise OracleError("X has the wrong number of rows for this frame")
    n_out = n_major if aligned else n_minor
    Y = np.zeros((n_out, w), np.float64)
    D = np.zeros((n_out, w), np.float64)
    _check(lib.or_spmm_slices(n_major, n_minor, _p(ptr), None if vp_ is None else _p(vp_),
                              _p(idx), _p(vals), int(bool(aligned)), _p(X), w, _p(Y), _p(D),
                              int(threads)))
    return Y, D
