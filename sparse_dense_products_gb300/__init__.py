"""Sparse x dense products over CSR and value-grouped VCS on one GB300 GPU.

The compute path is the CUDA library libvs (C ABI in include/vs.h, sources in
csrc/); this package is its thin Python binding.  Importing the package does
not load the library; the first call does, and fails loudly when libvs has not
been built (``python -m sparse_dense_products_gb300.build``).
"""
from .api import (SparseMatrix, build_csr, build_vcs, empty_out, gather_floor,  # noqa: F401
                  kernel_launches, spmm, spmm_host, version)
from ._lib import VsError  # noqa: F401

__all__ = ["SparseMatrix", "build_csr", "build_vcs", "empty_out", "gather_floor",
           "kernel_launches", "spmm", "spmm_host", "version", "VsError"]
