"""Python binding of libvs: argument marshalling only.

Every step of assembly and of the products runs in the CUDA library through
its C ABI (include/vs.h); PyTorch supplies device memory and streams.  The
names follow the C entry points:

* :func:`build_csr`, :func:`build_vcs` -> :class:`SparseMatrix` (wraps a
  ``vs_handle``)
* :func:`spmm` (``vs_spmm``), :func:`spmm_host` (``vs_spmm_host``)
* :meth:`SparseMatrix.attach_transpose`, :meth:`SparseMatrix.info`,
  :meth:`SparseMatrix.arrays`, :meth:`SparseMatrix.nbytes`,
  :meth:`SparseMatrix.destroy`
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib as L

_DTYPES = {torch.float32: L.F32, torch.float64: L.F64}
_MAJORS = {"row": L.MAJOR_ROW, "col": L.MAJOR_COL}
_DIRS = {"A@B": L.A_B, "B@A": L.B_A}
_VARIANTS = {"deterministic": L.DETERMINISTIC, "atomic": L.ATOMIC, "transposed": L.TRANSPOSED,
             "two_phase": L.TWO_PHASE}


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _require_cuda(*tensors):
    for t in tensors:
        if not t.is_cuda:
            raise ValueError("device tensors expected (use spmm_host for host operands)")


class SparseMatrix:
    """A CSR/CSC or VCSR/VCSC matrix held by libvs on one GPU."""

    def __init__(self, handle: int, shape, device):
        self._h = ctypes.c_void_p(handle)
        self.shape = tuple(int(s) for s in shape)
        self.device = torch.device(device)

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise RuntimeError("matrix has been destroyed")
        return self._h

    def info(self) -> dict:
        inf = L.Info()
        L.check(L.load().vs_info(self.handle, ctypes.byref(inf)))
        return {f: getattr(inf, f) for f, _ in L.Info._fields_ if f != "reserved"}

    @property
    def layout(self) -> str:
        return "vcs" if self.info()["layout"] == L.LAYOUT_VCS else "csr"

    @property
    def major(self) -> str:
        return "row" if self.info()["major"] == L.MAJOR_ROW else "col"

    @property
    def dtype(self) -> torch.dtype:
        return torch.float64 if self.info()["dtype"] == L.F64 else torch.float32

    def arrays(self) -> dict:
        """Copies of the layout arrays as torch tensors on the device."""
        a = L.Arrays()
        L.check(L.load().vs_export(self.handle, ctypes.byref(a)))
        inf = self.info()
        vcs = inf["layout"] == L.LAYOUT_VCS
        n_major, nnz, R = a.n_major, a.nnz, a.n_runs

        def view(ptr, n, dtype):
            # zero-copy view of the handle's memory, then a copy owned by torch
            if n == 0:
                return torch.empty(0, dtype=dtype, device=self.device)
            cai = _DeviceArray(ptr, n, _TYPESTR[dtype])
            return torch.as_tensor(cai, device=self.device).clone()

        pt = torch.int64 if a.pointer_bits == 64 else torch.int32
        res = {"ptr": view(a.ptr, n_major + 1, pt),
               "indices": view(a.indices, nnz, torch.int32)}
        if vcs:
            res["values"] = view(a.values, R, torch.float32)
            res["value_ptr"] = view(a.value_ptr, R + 1, pt)
        else:
            res["values"] = view(a.values, nnz, self.dtype)
        return res

    def nbytes(self) -> tuple[int, int]:
        """(layout bytes, scratch bytes) held on the device."""
        lb, sb = ctypes.c_int64(), ctypes.c_int64()
        L.check(L.load().vs_handle_bytes(self.handle, ctypes.byref(lb), ctypes.byref(sb)))
        return lb.value, sb.value

    def attach_transpose(self) -> "SparseMatrix":
        L.check(L.load().vs_attach_transpose(self.handle, ctypes.c_void_p(_stream_ptr(self.device))))
        return self

    def transpose(self) -> "SparseMatrix":
        """A new matrix holding the exact transpose (shape swapped, other major axis)."""
        h = ctypes.c_void_p()
        L.check(L.load().vs_transpose(self.handle, ctypes.c_void_p(_stream_ptr(self.device)),
                                      ctypes.byref(h)))
        return SparseMatrix(h.value, (self.shape[1], self.shape[0]), self.device)

    def scale_entries(self, factors: torch.Tensor) -> "SparseMatrix":
        """A new CSR matrix sharing this one's indices, values[e] * factors[e]
        (factors in storage order, the order of arrays()["values"])."""
        _require_cuda(factors)
        if factors.dtype != self.dtype or factors.numel() != self.info()["nnz"] or \
                not factors.is_contiguous():
            raise ValueError("factors must be a contiguous tensor of nnz values of the matrix dtype")
        h = ctypes.c_void_p()
        L.check(L.load().vs_scale_entries(self.handle, ctypes.c_void_p(factors.data_ptr()),
                                          ctypes.c_void_p(_stream_ptr(self.device)),
                                          ctypes.byref(h)))
        return SparseMatrix(h.value, self.shape, self.device)

    def force_group_size(self, g: int) -> "SparseMatrix":
        """``vs_force_group_size``: test hook fixing the group size g of this
        matrix's gathers (1, 2, 4, ..., 32; 0 restores the matrix rule)."""
        L.check(L.load().vs_force_group_size(self.handle, int(g)))
        return self

    def destroy(self) -> None:
        if self._h:
            L.check(L.load().vs_destroy(self._h))
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            if self._h:
                L.load().vs_destroy(self._h)
                self._h = ctypes.c_void_p(0)
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()


_TYPESTR = {torch.int32: "<i4", torch.int64: "<i8", torch.float32: "<f4", torch.float64: "<f8"}


class _DeviceArray:
    """A 1-D device array exposed through __cuda_array_interface__ (copied, never written)."""

    def __init__(self, ptr: int, n: int, typestr: str):
        self.__cuda_array_interface__ = {"shape": (int(n),), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def _coo_args(rows: torch.Tensor, cols: torch.Tensor, vals: torch.Tensor):
    _require_cuda(rows, cols, vals)
    if rows.dtype != torch.int32 or cols.dtype != torch.int32:
        raise TypeError("rows and cols must be int32")
    if rows.numel() != cols.numel() or rows.numel() != vals.numel():
        raise ValueError("rows, cols and vals must have the same length")
    return rows.contiguous(), cols.contiguous(), vals.contiguous()


def _options(pointer_bits, segment_entries, two_phase_tile_rows):
    if pointer_bits is None and segment_entries is None and two_phase_tile_rows is None:
        return None
    return L.BuildOptions(int(pointer_bits or 0), int(two_phase_tile_rows or 0),
                          int(segment_entries or 0))


def build_csr(rows: torch.Tensor, cols: torch.Tensor, vals: torch.Tensor, shape,
              major: str = "row", *, pointer_bits: int | None = None,
              segment_entries: int | None = None,
              two_phase_tile_rows: int | None = None) -> SparseMatrix:
    """``vs_build_csr`` (``vs_build_csr_opts`` with options): CSR (major="row")
    or CSC (major="col") from device COO.

    Each slice keeps its entries in COO input order ("Regridder", "How it is built").
    ``pointer_bits`` (32, 64; default automatic), ``segment_entries`` and
    ``two_phase_tile_rows`` are the build options of include/vs.h.
    """
    rows, cols, vals = _coo_args(rows, cols, vals)
    if vals.dtype not in _DTYPES:
        raise TypeError("values must be float32 or float64")
    h = ctypes.c_void_p()
    opts = _options(pointer_bits, segment_entries, two_phase_tile_rows)
    args = (int(shape[0]), int(shape[1]), rows.numel(), rows.data_ptr(), cols.data_ptr(),
            vals.data_ptr(), _DTYPES[vals.dtype], _MAJORS[major])
    stream = ctypes.c_void_p(_stream_ptr(rows.device))
    if opts is None:
        L.check(L.load().vs_build_csr(*args, stream, ctypes.byref(h)))
    else:
        L.check(L.load().vs_build_csr_opts(*args, ctypes.byref(opts), stream, ctypes.byref(h)))
    return SparseMatrix(h.value, shape, rows.device)


def build_vcs(rows: torch.Tensor, cols: torch.Tensor, vals: torch.Tensor, shape,
              major: str = "row", *, pointer_bits: int | None = None,
              segment_entries: int | None = None,
              two_phase_tile_rows: int | None = None) -> SparseMatrix:
    """``vs_build_vcs`` (``vs_build_vcs_opts`` with options): VCSR (major="row")
    or VCSC (major="col") from device COO (float32)."""
    rows, cols, vals = _coo_args(rows, cols, vals)
    if vals.dtype != torch.float32:
        raise TypeError("VCS values are float32")
    h = ctypes.c_void_p()
    opts = _options(pointer_bits, segment_entries, two_phase_tile_rows)
    args = (int(shape[0]), int(shape[1]), rows.numel(), rows.data_ptr(), cols.data_ptr(),
            vals.data_ptr(), _MAJORS[major])
    stream = ctypes.c_void_p(_stream_ptr(rows.device))
    if opts is None:
        L.check(L.load().vs_build_vcs(*args, stream, ctypes.byref(h)))
    else:
        L.check(L.load().vs_build_vcs_opts(*args, ctypes.byref(opts), stream, ctypes.byref(h)))
    return SparseMatrix(h.value, shape, rows.device)


def _dense(t: torch.Tensor) -> L.Dense:
    if t.dim() != 2:
        raise ValueError("dense operands are 2-D")
    dt = _DTYPES.get(t.dtype)
    if dt is None:
        raise TypeError("dense operands must be float32 or float64")
    rows, cols = t.shape
    rs, cs = t.stride()
    return L.Dense(t.data_ptr() if rows and cols else 0, rows, cols, rs, cs, dt)


def empty_out(A: SparseMatrix, w: int, direction: str = "A@B", dtype=None, device=None,
              pin_memory: bool = False) -> torch.Tensor:
    """An output tensor in the width-contiguous layout the product needs."""
    dtype = dtype or A.dtype
    device = device or A.device
    n_rows, n_cols = A.shape
    if direction == "A@B":
        return torch.empty(n_rows, w, dtype=dtype, device=device, pin_memory=pin_memory)
    return torch.empty(n_cols, w, dtype=dtype, device=device, pin_memory=pin_memory).t()


def spmm(A: SparseMatrix, B: torch.Tensor, direction: str = "A@B",
         variant: str = "deterministic", out: torch.Tensor | None = None, *,
         map: str | None = None, row_scale: torch.Tensor | None = None,
         col_scale: torch.Tensor | None = None) -> torch.Tensor:
    """``vs_spmm``: out = A @ B or out = B @ A on the current CUDA stream.

    A@B: B is n_cols x w with stride(1) == 1; B@A: B is w x n_rows with
    stride(0) == 1 (e.g. ``Bt.t()`` for a contiguous n_rows x w ``Bt``).

    With ``map`` ("identity", "log1p", "sqrt"), ``row_scale`` (n_rows) or
    ``col_scale`` (n_cols) the product uses the normalized view
    diag(row_scale) g(A) diag(col_scale) instead of A (``vs_spmm_view``).
    """
    _require_cuda(B)
    w = B.shape[1] if direction == "A@B" else B.shape[0]
    if out is None:
        out = empty_out(A, w, direction, B.dtype, B.device)
    _require_cuda(out)
    bd, od = _dense(B), _dense(out)
    stream = ctypes.c_void_p(_stream_ptr(B.device))
    if map is None and row_scale is None and col_scale is None:
        L.check(L.load().vs_spmm(A.handle, ctypes.byref(bd), ctypes.byref(od), _DIRS[direction],
                                 _VARIANTS[variant], stream))
        return out
    view = L.View(L.MAPS[map or "identity"], None, None)
    for name, t, n in (("row_scale", row_scale, A.shape[0]), ("col_scale", col_scale, A.shape[1])):
        if t is not None:
            _require_cuda(t)
            if t.dtype != B.dtype or t.numel() != n or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous tensor of {n} values of B's dtype")
            setattr(view, name, t.data_ptr())
    L.check(L.load().vs_spmm_view(A.handle, ctypes.byref(bd), ctypes.byref(od), _DIRS[direction],
                                  _VARIANTS[variant], ctypes.byref(view), stream))
    return out


def spmm_host(A: SparseMatrix, B: torch.Tensor, direction: str = "A@B",
              variant: str = "deterministic", out: torch.Tensor | None = None) -> torch.Tensor:
    """``vs_spmm_host``: the product with B and out in (preferably pinned) host memory."""
    if B.is_cuda:
        raise ValueError("spmm_host takes host tensors")
    w = B.shape[1] if direction == "A@B" else B.shape[0]
    if out is None:
        out = empty_out(A, w, direction, B.dtype, "cpu", pin_memory=B.is_pinned())
    bd, od = _dense(B), _dense(out)
    L.check(L.load().vs_spmm_host(A.handle, ctypes.byref(bd), ctypes.byref(od), _DIRS[direction],
                                  _VARIANTS[variant], ctypes.c_void_p(_stream_ptr(A.device))))
    return out


def gather_floor(A: SparseMatrix, B: torch.Tensor, direction: str = "A@B") -> None:
    """``vs_gather_floor``: enqueue the gather-only measurement kernel for the
    product ``spmm(A, B, direction)`` (time it with CUDA events)."""
    _require_cuda(B)
    bd = _dense(B)
    L.check(L.load().vs_gather_floor(A.handle, ctypes.byref(bd), _DIRS[direction],
                                     ctypes.c_void_p(_stream_ptr(B.device))))


def version() -> int:
    return int(L.load().vs_version())


def kernel_launches() -> int:
    """``vs_kernel_launches``: kernels libvs has launched in this process."""
    return int(L.load().vs_kernel_launches())
