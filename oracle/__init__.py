"""Oracle for y = A x, the column-delta format (fp64, CPU, plain C), the
sliced ELL layout and the matrix-free stiffness operator (numpy).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the library under test never does, and
this package imports nothing from it.

What it computes, and the passages it follows:

* ``csr_spmv`` -- the scalar CSR kernel of the "CUDA CSR SpMV optimisation"
  page, section 2.1: ``y[i] = sum_{k=row_ptr[i]}^{row_ptr[i+1]-1} a_k x[c_k]``,
  summed in stored order in fp64 (every fp32 or fp16 input converts to fp64
  exactly), together with ``s[i] = sum |a_k x[c_k]|`` which scales the parity
  tolerances.
* ``delta_encode`` / ``delta_decode`` -- the "MACKO-SpMV" page, section 2.1
  (delta coding, zero padding when a gap does not fit in 4 bits, eight nibbles
  per 32-bit word, row alignment). The readings taken where the page is
  silent or garbled are listed at the top of ``spmv_oracle.c``.

* ``oracle.sell`` -- the sliced ELL layout and the choice of format by the
  coefficient of variation of the row lengths ("CUDA CSR SpMV optimisation",
  sections 2.1 and 2.2), in numpy; its readings are listed in its docstring.

* ``oracle.fem`` -- the matrix-free stiffness operator of the "Fused FEM
  matvec" page (gather, element product, scatter-add; one element matrix
  scaled by a density per element), in numpy fp64, and the assembled matrix
  it equals.

Parity pins (tests/test_oracle.py): dense brute force on tiny matrices,
identity and permutation matrices, 5-point Laplacian rows on constant vectors,
a row of ones, scipy's CSR product, the page's worked delta example and
hand-derived padding cases, and the encode/decode round trip.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spmv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
           "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA involved). Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64 = ctypes.c_int64
    p = ctypes.c_void_p
    lib.oracle_csr_spmv.argtypes = [i64, p, p, p, p, p, p]
    lib.oracle_csr_spmv.restype = ctypes.c_int
    lib.oracle_delta_count.argtypes = [i64, p, p, p, p, p]
    lib.oracle_delta_count.restype = ctypes.c_int
    lib.oracle_delta_fill.argtypes = [i64, p, p, p, p, p, p]
    lib.oracle_delta_fill.restype = ctypes.c_int
    lib.oracle_delta_decode.argtypes = [i64, p, p, p, p, p, p]
    lib.oracle_delta_decode.restype = i64
    ci = ctypes.c_int
    lib.oracle_delta_count_bits.argtypes = [i64, p, p, ci, p, p, p]
    lib.oracle_delta_count_bits.restype = ctypes.c_int
    lib.oracle_delta_fill_bits.argtypes = [i64, p, p, p, ci, p, p, p]
    lib.oracle_delta_fill_bits.restype = ctypes.c_int
    lib.oracle_delta_decode_bits.argtypes = [i64, p, p, p, ci, p, p, p]
    lib.oracle_delta_decode_bits.restype = i64
    return lib


def compile_variant(source_text: str, out_dir: str, name: str) -> str:
    """Compile an edited copy of the oracle source (used by the tests that
    plant a mistake in the oracle to show that the pins catch it)."""
    os.makedirs(out_dir, exist_ok=True)
    src = os.path.join(out_dir, name + ".c")
    lib = os.path.join(out_dir, name + ".so")
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", *_CFLAGS, "-o", lib, src], check=True)
    return lib


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


class use_library:
    """Context manager: route every oracle call through another build of the
    oracle source for the duration of the block."""

    def __init__(self, path: str):
        self._path = path
        self._saved = None

    def __enter__(self):
        global _lib
        with _lock:
            self._saved = _lib
            _lib = _bind(self._path)
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._saved
        return False


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


def _f64(a) -> np.ndarray:
    # fp16 -> fp64 and fp32 -> fp64 are exact conversions.
    return np.ascontiguousarray(np.asarray(a).astype(np.float64))


def csr_spmv(row_ptr, col_idx, values, x, with_abs: bool = True):
    """fp64 y = A x (and s = |A||x|) for a CSR matrix; stored-order sums."""
    rp, ci = _i64(row_ptr), _i64(col_idx)
    a, xv = _f64(values), _f64(x)
    n_rows = rp.shape[0] - 1
    y = np.empty(n_rows, dtype=np.float64)
    s = np.empty(n_rows, dtype=np.float64) if with_abs else None
    _load().oracle_csr_spmv(n_rows, _ptr(rp), _ptr(ci), _ptr(a), _ptr(xv),
                            _ptr(y), _ptr(s) if with_abs else None)
    return (y, s) if with_abs else y


class DeltaMatrix:
    """The column-delta format as plain numpy arrays (fields of `bits` bits,
    32 / bits to a word; 4 bits unless asked otherwise)."""

    def __init__(self, n_rows, n_cols, row_ptr, values, words, gap_pads,
                 align_pads, bits=4):
        self.n_rows = n_rows
        self.n_cols = n_cols
        self.row_ptr = row_ptr      # int64[n_rows+1], entry offsets
        self.values = values        # uint16[n_entries], fp16 bit patterns
        self.words = words          # uint32[n_entries*bits/32], packed fields
        self.gap_pads = gap_pads
        self.align_pads = align_pads
        self.bits = bits

    @property
    def n_entries(self) -> int:
        return int(self.row_ptr[-1])

    def deltas(self) -> np.ndarray:
        """Unpacked codes, one per entry (lowest field first)."""
        per = 32 // self.bits
        shifts = (self.bits * np.arange(per, dtype=np.uint32))
        d = (self.words[:, None] >> shifts[None, :]) & np.uint32((1 << self.bits) - 1)
        return d.reshape(-1).astype(np.uint8)


def delta_encode(n_cols, row_ptr, col_idx, values_f16, bits: int = 4) -> DeltaMatrix:
    """Encode a CSR matrix with fp16 values into the column-delta format with
    deltas of `bits` bits (2, 4 or 8)."""
    rp, ci = _i64(row_ptr), _i64(col_idx)
    vb = np.ascontiguousarray(np.asarray(values_f16, dtype=np.float16)
                              .view(np.uint16))
    n_rows = rp.shape[0] - 1
    lib = _load()
    out_rp = np.empty(n_rows + 1, dtype=np.int64)
    gaps = np.zeros(1, dtype=np.int64)
    aligns = np.zeros(1, dtype=np.int64)
    rc = lib.oracle_delta_count_bits(n_rows, _ptr(rp), _ptr(ci), int(bits), _ptr(out_rp),
                                     _ptr(gaps), _ptr(aligns))
    if rc == -2:
        raise ValueError("delta width must be 2, 4 or 8 bits")
    if rc != 0:
        raise ValueError("delta format needs strictly increasing, "
                         "non-negative columns in every row")
    n_entries = int(out_rp[-1])
    out_vals = np.zeros(n_entries, dtype=np.uint16)
    out_words = np.zeros(n_entries * bits // 32, dtype=np.uint32)
    lib.oracle_delta_fill_bits(n_rows, _ptr(rp), _ptr(ci), _ptr(vb), int(bits), _ptr(out_rp),
                               _ptr(out_vals), _ptr(out_words))
    return DeltaMatrix(n_rows, int(n_cols), out_rp, out_vals, out_words,
                       int(gaps[0]), int(aligns[0]), bits=int(bits))


def delta_decode(m: DeltaMatrix):
    """Decode back to CSR (row_ptr int64, col int64, values fp16)."""
    rp = _i64(m.row_ptr)
    vals = np.ascontiguousarray(m.values, dtype=np.uint16)
    words = np.ascontiguousarray(m.words, dtype=np.uint32)
    n = m.n_entries
    out_rp = np.empty(m.n_rows + 1, dtype=np.int64)
    out_col = np.empty(max(n, 1), dtype=np.int64)
    out_vals = np.empty(max(n, 1), dtype=np.uint16)
    kept = _load().oracle_delta_decode_bits(m.n_rows, _ptr(rp), _ptr(vals), _ptr(words),
                                            int(m.bits), _ptr(out_rp), _ptr(out_col),
                                            _ptr(out_vals))
    return out_rp, out_col[:kept].copy(), out_vals[:kept].view(np.float16).copy()


def delta_spmv(m: DeltaMatrix, x, with_abs: bool = True):
    """fp64 y = A x for a matrix held in the delta format (decode, then CSR)."""
    rp, col, vals = delta_decode(m)
    return csr_spmv(rp, col, vals, x, with_abs=with_abs)
