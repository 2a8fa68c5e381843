"""ctypes loader for ``libspops_gb300.so`` (argument marshalling only).

The library must have been built (``build.build()``); a missing library is an error, not
a reason to fall back to anything else.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_INT = ctypes.c_int
_SZ = ctypes.c_size_t

# name -> (restype, argtypes), in the order of include/spops_gb300.h
SIGNATURES = {
    "spops_status_string": (ctypes.c_char_p, [_INT]),
    "spops_last_error": (ctypes.c_char_p, []),
    "spops_version": (ctypes.c_char_p, []),
    "spops_kernel_launches": (ctypes.c_uint64, []),
    "spops_release_streams": (_INT, []),
    "spops_sort_rows_workspace_size": (_SZ, [_I32]),
    "spops_sort_rows": (_INT, [_P, _I32, _I32, _P, _INT, _P, _SZ, _P]),
    "spops_sort_rows_static": (_INT, [_P, _I32, _I32, _P, _INT, _P]),
    "spops_sort_rows_static_max_rows": (_I32, []),
    "spops_row_bins": (_INT, [_P, _I32, _I32, _P, _P]),
    "spops_spmm_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _INT, _INT]),
    "spops_plan_size": (_SZ, [_I32, _I32, _I32]),
    "spops_plan_build": (_INT, [_P, _P, _P, _INT, _I32, _I32, _I32, _P, _SZ, _P]),
    "spops_plan_stats": (_INT, [_P, _I32, _I32, _I32, _P, _P]),
    "spops_plan_row_order": (_INT, [_P, _I32, _I32, _I32, _P, _P]),
    "spops_spmm": (_INT, [_P, _P, _P, _P, _INT, _INT, _I32, _I32, _I32, _P, _I32, _P, _INT, _P, _P, _SZ, _P]),
    "spops_sddmm_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _INT, _INT, _INT]),
    "spops_sddmm": (_INT, [_P, _P, _P, _INT, _INT, _I32, _I32, _I32, _I32, _P, _P, _P, _INT, _P, _P, _SZ, _P]),
    "spops_csr_add": (_INT, [_P, _P, _P, _P, _INT, _INT, _I32, _I32, _I32, _P, _P, _P]),
    "spops_check_csr_workspace_size": (_SZ, [_I32]),
    "spops_check_csr": (_INT, [_P, _P, _P, _INT, _I32, _I32, _I32, _P, _SZ, _P]),
    "spops_get_device_error": (_INT, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "spops_selftest_wait_timeout": (_INT, [ctypes.c_int64, _P, _P]),
    "spops_csr_transpose_workspace_size": (_SZ, [_I32]),
    "spops_csr_transpose": (_INT, [_P, _P, _P, _INT, _INT, _I32, _I32, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "spops_csr_permute_values": (_INT, [_P, _P, _INT, _I32, _P, _P]),
    "spops_masked_adam": (_INT, [_P, _P, _P, _P, _INT, ctypes.c_int64, _I32, ctypes.c_double, ctypes.c_double,
                                 ctypes.c_double, ctypes.c_double, _INT, _P]),
    "spops_masked_adam_csr": (_INT, [_P, _P, _P, _P, _INT, _P, _P, _INT, _I32, _I32, _I32, _I32, ctypes.c_double,
                                     ctypes.c_double, ctypes.c_double, ctypes.c_double, _INT, _P]),
}

_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the CUDA library; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"spops_gb300 CUDA library not built ({path} missing); "
                               "run unstructured_sparse_linear_gb300.build.build() first")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
