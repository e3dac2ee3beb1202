"""ctypes declarations for the C ABI in include/spmv.h (argument marshalling
only; no computation happens here)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

LIB_PATH = _build.LIB_PATH

c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_p = ctypes.c_void_p

SPMV_F32, SPMV_F16 = 0, 1
SPMV_FORMAT_CSR, SPMV_FORMAT_DELTA4, SPMV_FORMAT_DELTA2, SPMV_FORMAT_DELTA8 = 0, 1, 2, 3
SPMV_FORMAT_DELTA_AUTO, SPMV_FORMAT_SELL, SPMV_FORMAT_AUTO, SPMV_FORMAT_FEM = 4, 5, 6, 7
SPMV_SELL_C = 32
SPMV_DELTA_FEWEST_BYTES, SPMV_DELTA_SPARSITY_TABLE = 0, 1

STATUS_NAMES = {
    0: "SPMV_OK", 1: "SPMV_ERR_INVALID_ARG", 2: "SPMV_ERR_BAD_ROW_PTR",
    3: "SPMV_ERR_COL_OUT_OF_RANGE", 4: "SPMV_ERR_UNSORTED_OR_DUPLICATE_COLS",
    5: "SPMV_ERR_UNSUPPORTED", 6: "SPMV_ERR_OUT_OF_MEMORY", 7: "SPMV_ERR_CUDA",
    8: "SPMV_ERR_TOO_LARGE", 9: "SPMV_ERR_WRONG_DEVICE",
    10: "SPMV_ERR_DEVICE_STATUS",
}


class spmv_csr(ctypes.Structure):
    _fields_ = [("n_rows", c_i32), ("n_cols", c_i32), ("nnz", c_i64),
                ("row_ptr", c_p), ("col_idx", c_p), ("values", c_p),
                ("value_dtype", ctypes.c_int)]


class spmv_delta(ctypes.Structure):
    _fields_ = [("n_rows", c_i32), ("n_cols", c_i32), ("nnz", c_i64),
                ("n_entries", c_i64), ("n_gap_pads", c_i64),
                ("n_align_pads", c_i64), ("n_explicit_zeros", c_i64),
                ("values", c_p), ("words", c_p), ("row_ptr", c_p),
                ("delta_bits", c_i32), ("reserved", c_i32)]


class spmv_sell(ctypes.Structure):
    _fields_ = [("n_rows", c_i32), ("n_cols", c_i32), ("nnz", c_i64),
                ("C", c_i32), ("sigma", c_i32), ("n_slices", c_i64),
                ("n_slots", c_i64), ("slice_ptr", c_p), ("perm", c_p),
                ("cols", c_p), ("values", c_p), ("value_dtype", ctypes.c_int),
                ("reserved", c_i32)]


class spmv_fem_mesh(ctypes.Structure):
    _fields_ = [("nex", c_i32), ("ney", c_i32), ("nez", c_i32), ("reserved", c_i32),
                ("rho", c_p), ("K0", c_p)]


class spmv_pcg_result(ctypes.Structure):
    _fields_ = [("iterations", c_i32), ("status", c_i32), ("rel_residual", ctypes.c_double)]


class spmv_plan_options(ctypes.Structure):
    _fields_ = [("tile_nnz", c_i32), ("tile_rows", c_i32),
                ("cta_row_min", c_i32), ("split_row_min", c_i32),
                ("split_chunk", c_i32), ("x_smem", c_i32), ("reduce", c_i32),
                ("lanes", c_i32), ("interleave", c_i32), ("sell_sigma", c_i32),
                ("csr_kernel", c_i32), ("delta_kernel", c_i32), ("reserved", c_i32 * 4)]


class spmv_plan_info(ctypes.Structure):
    _fields_ = [("n_rows", c_i32), ("n_cols", c_i32), ("nnz", c_i64),
                ("format", c_i32), ("value_dtype", c_i32),
                ("n_entries", c_i64), ("n_tiles", c_i64),
                ("rows_per_bin", c_i64 * 4), ("tiles_per_bin", c_i64 * 4),
                ("n_split_rows", c_i64), ("x_in_smem", c_i32),
                ("grid", c_i32), ("block", c_i32),
                ("launches_per_run", c_i32), ("matrix_bytes", c_i64),
                ("aux_bytes", c_i64), ("algorithmic_bytes", c_i64),
                ("walk_tiles", c_i64), ("interleaved", c_i64), ("segments", c_i64),
                ("reserved", c_i64 * 5)]


# name -> (restype, argtypes); every function declared in include/spmv.h
SIGNATURES = {
    "spmv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "spmv_abi_version": (c_i32, []),
    "spmv_plan_options_init": (None, [ctypes.POINTER(spmv_plan_options)]),
    "spmv_convert": (ctypes.c_int, [ctypes.POINTER(spmv_csr),
                                    ctypes.POINTER(spmv_delta)]),
    "spmv_convert_bits": (ctypes.c_int, [ctypes.POINTER(spmv_csr), c_i32,
                                         ctypes.POINTER(spmv_delta)]),
    "spmv_delta_select_bits": (ctypes.c_int, [ctypes.POINTER(spmv_csr), ctypes.c_int,
                                              ctypes.POINTER(c_i32), ctypes.POINTER(c_i64)]),
    "spmv_delta_free": (None, [ctypes.POINTER(spmv_delta)]),
    "spmv_convert_sell": (ctypes.c_int, [ctypes.POINTER(spmv_csr), c_i32,
                                         ctypes.POINTER(spmv_sell)]),
    "spmv_sell_free": (None, [ctypes.POINTER(spmv_sell)]),
    "spmv_select_format": (ctypes.c_int, [ctypes.POINTER(spmv_csr), ctypes.POINTER(ctypes.c_int),
                                          ctypes.POINTER(c_i32), ctypes.POINTER(ctypes.c_double)]),
    "spmv_plan_inspect": (ctypes.c_int, [ctypes.POINTER(spmv_csr), ctypes.c_int,
                                         ctypes.POINTER(spmv_plan_options),
                                         ctypes.POINTER(spmv_plan_info)]),
    "spmv_plan_create": (ctypes.c_int, [ctypes.POINTER(spmv_csr), ctypes.c_int,
                                        ctypes.POINTER(c_p)]),
    "spmv_plan_create_ex": (ctypes.c_int, [ctypes.POINTER(spmv_csr),
                                           ctypes.c_int,
                                           ctypes.POINTER(spmv_plan_options),
                                           ctypes.POINTER(c_p)]),
    "spmv_plan_create_delta": (ctypes.c_int, [ctypes.POINTER(spmv_delta),
                                              ctypes.POINTER(spmv_plan_options),
                                              ctypes.POINTER(c_p)]),
    "spmv_plan_create_fem": (ctypes.c_int, [ctypes.POINTER(spmv_fem_mesh),
                                            ctypes.POINTER(c_p)]),
    "spmv_pcg_solve": (ctypes.c_int, [c_p, c_p, c_p, c_p, ctypes.c_double, c_i32, c_i32, c_p,
                                      ctypes.POINTER(spmv_pcg_result)]),
    "spmv_plan_get_info": (ctypes.c_int, [c_p, ctypes.POINTER(spmv_plan_info)]),
    "spmv_run": (ctypes.c_int, [c_p, c_p, c_p, c_p]),
    "spmv_run_host": (ctypes.c_int, [c_p, c_p, c_p, c_p]),
    "spmv_run_host_batch": (ctypes.c_int, [c_p, c_i32, c_p, c_p, c_p]),
    "spmv_csr_run_noalloc": (ctypes.c_int, [c_i32, c_i32, c_i64, c_p, c_p, c_p,
                                            ctypes.c_int, c_p, c_p, c_p]),
    "spmv_plan_check": (ctypes.c_int, [c_p]),
    "spmv_checked_build": (c_i32, []),
    "spmv_noalloc_check": (ctypes.c_int, []),
    "spmv_plan_destroy": (None, [c_p]),
}

_lock = threading.Lock()
_lib = None


def library_exists() -> bool:
    return os.path.exists(LIB_PATH)


def load():
    """Load libspmv_gb300.so. Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is None:
            if not library_exists():
                raise ImportError(
                    f"{LIB_PATH} is missing: build it first with "
                    "`python -c \"import __graft_entry__ as g; g.build()\"` "
                    "or `python -m sparse_matrix_vector_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


_checked = None


def load_checked():
    """The checked build of the library (built in-tree on first use): the
    same C ABI, with every column index and row offset tested on the device
    before use (include/spmv.h, spmv_checked_build). For tests and
    debugging; the package's functions use load()."""
    global _checked
    with _lock:
        if _checked is None:
            path = _build.build_library(checked=True)
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _checked = lib
    return _checked
