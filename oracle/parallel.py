"""All-core CPU baseline: the oracle's CSR loop and its column-delta walk with
rows shared out over OpenMP threads (``spmv_omp.c``).

TEST AND BENCHMARK INFRASTRUCTURE ONLY: the benchmark times it beside the GPU
path as a second CPU baseline; it is not the parity oracle (the single-threaded
``oracle.csr_spmv`` is), and the library under test never imports it.

Each row is summed by one thread in fp64 in stored order, so the results equal
the single-threaded oracle's bit for bit (``tests/test_oracle.py`` checks it).
Passages followed: "CUDA CSR SpMV optimisation" 2.1 (the CSR product) and
"MACKO-SpMV" 2.1 (the column-delta format).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spmv_omp.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_omp.so")
_CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-std=c11",
           "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None
_half_table = None


def build(force: bool = False) -> str:
    """Compile the OpenMP baseline with gcc. Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.omp_baseline_threads.argtypes = []
            lib.omp_baseline_threads.restype = ctypes.c_int
            lib.omp_csr_spmv.argtypes = [i64, p, p, p, p, p]
            lib.omp_csr_spmv.restype = ctypes.c_int
            lib.omp_delta_spmv.argtypes = [i64, p, p, p, ctypes.c_int, p, p, p]
            lib.omp_delta_spmv.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def threads() -> int:
    """OpenMP threads the loops run on (OMP_NUM_THREADS, else every core)."""
    return int(_load().omp_baseline_threads())


class CsrOperands:
    """A CSR matrix widened once to the loop's types (int64 indices, fp64
    values and x), so that a timed call does only the product."""

    def __init__(self, row_ptr, col_idx, values, x):
        self.rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
        self.ci = np.ascontiguousarray(col_idx, dtype=np.int64)
        self.a = np.ascontiguousarray(np.asarray(values).astype(np.float64))
        self.x = np.ascontiguousarray(np.asarray(x).astype(np.float64))
        self.y = np.empty(self.rp.shape[0] - 1, dtype=np.float64)

    def __call__(self) -> np.ndarray:
        _load().omp_csr_spmv(self.y.shape[0], _ptr(self.rp), _ptr(self.ci), _ptr(self.a),
                             _ptr(self.x), _ptr(self.y))
        return self.y


class DeltaOperands:
    """A matrix in the column-delta format (an ``oracle.DeltaMatrix``) and x,
    ready for the parallel row walk."""

    def __init__(self, m, x):
        global _half_table
        if _half_table is None:
            _half_table = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
        self.m = m
        self.rp = np.ascontiguousarray(m.row_ptr, dtype=np.int64)
        self.vals = np.ascontiguousarray(m.values, dtype=np.uint16)
        self.words = np.ascontiguousarray(m.words, dtype=np.uint32)
        self.x = np.ascontiguousarray(np.asarray(x).astype(np.float64))
        self.y = np.empty(m.n_rows, dtype=np.float64)

    def __call__(self) -> np.ndarray:
        rc = _load().omp_delta_spmv(self.m.n_rows, _ptr(self.rp), _ptr(self.vals),
                                    _ptr(self.words), int(self.m.bits), _ptr(_half_table),
                                    _ptr(self.x), _ptr(self.y))
        if rc != 0:
            raise ValueError("delta width must be 2, 4 or 8 bits")
        return self.y
