"""ctypes declarations of the libvs C ABI (include/vs.h).

The shared library is built in-tree by :mod:`sparse_dense_products_gb300.build`
into ``_build/libvs.so``.  Loading fails loudly when it is missing: there is no
fallback implementation of any product.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

_lock = threading.Lock()
_lib = None

VS_OK = 0
STATUS = {
    0: "VS_OK", 1: "VS_ERR_INVALID", 2: "VS_ERR_SHAPE", 3: "VS_ERR_LAYOUT", 4: "VS_ERR_RANGE",
    5: "VS_ERR_ALLOC", 6: "VS_ERR_CUDA", 7: "VS_ERR_TIMEOUT", 8: "VS_ERR_UNSUPPORTED",
    9: "VS_ERR_NAN",
}
F32, F64 = 0, 1
MAJOR_ROW, MAJOR_COL = 0, 1
A_B, B_A = 0, 1
DETERMINISTIC, ATOMIC, TRANSPOSED, TWO_PHASE = 0, 1, 2, 3
LAYOUT_CSR, LAYOUT_VCS = 0, 1


class Dense(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("row_stride", ctypes.c_int64), ("col_stride", ctypes.c_int64),
                ("dtype", ctypes.c_int)]


class Info(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int32), ("major", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("group_size", ctypes.c_int32), ("n_rows", ctypes.c_int64),
                ("n_cols", ctypes.c_int64), ("nnz", ctypes.c_int64), ("n_runs", ctypes.c_int64),
                ("chunk_len", ctypes.c_int64), ("n_long_slices", ctypes.c_int64),
                ("n_chunks", ctypes.c_int64), ("n_blocks", ctypes.c_int64),
                ("has_transpose", ctypes.c_int32),
                ("pointer_bits", ctypes.c_int32),
                ("n_segments", ctypes.c_int32),
                ("two_phase_tiles", ctypes.c_int32)]


class BuildOptions(ctypes.Structure):
    _fields_ = [("pointer_bits", ctypes.c_int32), ("two_phase_tile_rows", ctypes.c_int32),
                ("segment_entries", ctypes.c_int64)]


class View(ctypes.Structure):
    _fields_ = [("map", ctypes.c_int), ("row_scale", ctypes.c_void_p),
                ("col_scale", ctypes.c_void_p)]


MAPS = {"identity": 0, "log1p": 1, "sqrt": 2}


class Arrays(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("indices", ctypes.c_void_p), ("values", ctypes.c_void_p),
                ("value_ptr", ctypes.c_void_p), ("n_major", ctypes.c_int64), ("nnz", ctypes.c_int64),
                ("n_runs", ctypes.c_int64), ("pointer_bits", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class VsError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {message}")


def load() -> ctypes.CDLL:
    """Loads libvs.so (raises if it has not been built)."""
    global _lib
    lib = _lib
    if lib is not None:  # loaded: no lock on the per-call path
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB):
            raise RuntimeError(f"libvs is not built ({LIB} missing); run "
                               "`python -m sparse_dense_products_gb300.build`")
        lib = ctypes.CDLL(LIB)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        H = ctypes.c_void_p
        lib.vs_build_csr.argtypes = [i64, i64, i64, vp, vp, vp, i32, i32, vp, ctypes.POINTER(H)]
        lib.vs_build_vcs.argtypes = [i64, i64, i64, vp, vp, vp, i32, vp, ctypes.POINTER(H)]
        lib.vs_build_csr_opts.argtypes = [i64, i64, i64, vp, vp, vp, i32, i32,
                                          ctypes.POINTER(BuildOptions), vp, ctypes.POINTER(H)]
        lib.vs_build_vcs_opts.argtypes = [i64, i64, i64, vp, vp, vp, i32,
                                          ctypes.POINTER(BuildOptions), vp, ctypes.POINTER(H)]
        lib.vs_spmm.argtypes = [H, ctypes.POINTER(Dense), ctypes.POINTER(Dense), i32, i32, vp]
        lib.vs_spmm_host.argtypes = [H, ctypes.POINTER(Dense), ctypes.POINTER(Dense), i32, i32, vp]
        lib.vs_spmm_noalloc.argtypes = [H, ctypes.POINTER(Dense), ctypes.POINTER(Dense), i32, vp]
        lib.vs_spmm_view.argtypes = [H, ctypes.POINTER(Dense), ctypes.POINTER(Dense), i32, i32,
                                     ctypes.POINTER(View), vp]
        lib.vs_attach_transpose.argtypes = [H, vp]
        lib.vs_transpose.argtypes = [H, vp, ctypes.POINTER(H)]
        lib.vs_gather_floor.argtypes = [H, ctypes.POINTER(Dense), i32, vp]
        lib.vs_device_status.argtypes = [H, vp]
        lib.vs_test_stall_producers.argtypes = [i32]
        lib.vs_test_stall_producers.restype = None
        lib.vs_scale_entries.argtypes = [H, vp, vp, ctypes.POINTER(H)]
        lib.vs_force_group_size.argtypes = [H, ctypes.c_int32]
        lib.vs_info.argtypes = [H, ctypes.POINTER(Info)]
        lib.vs_export.argtypes = [H, ctypes.POINTER(Arrays)]
        lib.vs_handle_bytes.argtypes = [H, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        lib.vs_destroy.argtypes = [H]
        for f in ("vs_build_csr", "vs_build_vcs", "vs_build_csr_opts", "vs_build_vcs_opts", "vs_spmm", "vs_spmm_host", "vs_spmm_noalloc",
                  "vs_spmm_view",
                  "vs_attach_transpose", "vs_transpose", "vs_scale_entries", "vs_force_group_size", "vs_gather_floor", "vs_device_status",
                  "vs_info", "vs_export", "vs_handle_bytes", "vs_destroy"):
            getattr(lib, f).restype = i32
        lib.vs_status_string.argtypes = [i32]
        lib.vs_status_string.restype = ctypes.c_char_p
        lib.vs_last_error.argtypes = []
        lib.vs_last_error.restype = ctypes.c_char_p
        lib.vs_version.argtypes = []
        lib.vs_version.restype = ctypes.c_int32
        lib.vs_kernel_launches.argtypes = []
        lib.vs_kernel_launches.restype = ctypes.c_int64
        _lib = lib
        return lib


def check(status: int) -> None:
    if status != VS_OK:
        msg = load().vs_last_error().decode(errors="replace")
        raise VsError(status, msg)
