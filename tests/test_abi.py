"""The C ABI library builds for sm_103a, loads without a GPU and exports every
entry point include/vs.h declares."""
import os
import re

import pytest

from sparse_dense_products_gb300 import _lib
from sparse_dense_products_gb300 import build as vs_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "vs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vs_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    vs_build.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "vs_spmm" in names and "vs_build_csr" in names and "vs_build_vcs" in names
    assert "vs_destroy" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/vs.h but not exported"


def test_status_strings_and_version(lib):
    assert lib.vs_version() >= 100
    for code in range(10):
        assert lib.vs_status_string(code)
    assert lib.vs_status_string(99) == b"unknown status"


def test_null_arguments_are_rejected_without_a_gpu(lib):
    import ctypes
    assert lib.vs_spmm(None, None, None, 0, 0, None) == 1
    assert lib.vs_info(None, None) == 1
    assert lib.vs_destroy(None) == 0
    assert b"NULL" in lib.vs_last_error()
    h = ctypes.c_void_p()
    assert lib.vs_build_csr(-1, 3, 0, None, None, None, 0, 0, None, ctypes.byref(h)) == 1
    assert lib.vs_build_csr(3, 3, 0, None, None, None, 7, 0, None, ctypes.byref(h)) == 1
    assert lib.vs_build_vcs(1 << 31, 3, 0, None, None, None, 0, None, ctypes.byref(h)) == 8


def test_library_is_built_for_sm_103a():
    flags = " ".join(vs_build.ARCH)
    assert "compute_103a" in flags and "sm_103a" in flags
    assert os.path.exists(vs_build.LIB)


def test_dense_descriptors_marshal_shape_strides_and_dtype():
    import torch

    from sparse_dense_products_gb300 import api

    t = torch.empty(60, 16, dtype=torch.float64).t()          # 16 x 60, width-contiguous
    d = api._dense(t)
    assert (d.rows, d.cols, d.row_stride, d.col_stride) == (16, 60, 1, 16)
    assert d.ptr == t.data_ptr() and d.dtype == 1             # VS_F64
    e = api._dense(torch.empty(0, 16))
    assert not e.ptr and (e.rows, e.cols) == (0, 16)           # no storage: NULL pointer
    with pytest.raises(ValueError):
        api._dense(torch.empty(4))
    with pytest.raises(TypeError):
        api._dense(torch.empty(4, 4, dtype=torch.float16))
