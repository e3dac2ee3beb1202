"""Oracle for the sliced ELLPACK layout and the format choice by the
coefficient of variation of the row lengths (numpy, CPU).

TEST INFRASTRUCTURE ONLY, like the rest of this package.

Sources (web pages, by title and section):

* "CUDA CSR SpMV optimisation" (codechina.net), section 2.1: ELL stores every
  row padded with zeros to a common width, and is sensitive to that padding;
  section 2.2: the choice by the coefficient of variation (CV) of the row
  lengths -- below 0.3 ELL, from 0.3 to 0.7 the hybrid ELL + COO format, above
  0.7 CSR with rows reordered.

Readings where the page is silent (each also listed in the design notes):

* CV = population standard deviation of the row lengths / their mean; a
  matrix whose mean row length is 0 has CV 0.
* The ELL layout is cut into slices of C consecutive rows, each padded only to
  its own widest row (sliced ELL; C = n_rows gives plain ELL). Within a slice
  slot (k, lane) holds the k-th stored entry of the slice's lane-th row, at
  ``slice_ptr[s] + k * C + lane`` (column-major, so the C rows of a slice are
  read together). A padding slot stores value 0 at the row's last column (at
  column 0 for an empty row, and for the lanes of the last slice that hold no
  row), so it adds exactly 0 * x[col] for finite x.
* The middle CV band, given to the hybrid ELL + COO format on the page, is
  served by sorting rows by decreasing length inside windows of sigma rows
  before slicing (``sigma > 1``): like HYB's COO spill, it keeps the padding
  of a slice near its own rows' lengths. ``perm[p]`` is the original row at
  sorted position p (-1 past the last row). sigma = 1 keeps the row order.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import csr_spmv

CV_ELL = 0.3    # below: ELL (sliced, rows in order)
CV_CSR = 0.7    # above: CSR; in between: sorted slices
SIGMA_SORTED = 1024


def row_length_cv(row_ptr) -> float:
    """Coefficient of variation of the row lengths (population std / mean)."""
    lengths = np.diff(np.asarray(row_ptr, dtype=np.int64)).astype(np.float64)
    if lengths.size == 0:
        return 0.0
    mean = lengths.mean()
    if mean == 0.0:
        return 0.0
    return float(np.sqrt(np.mean((lengths - mean) ** 2)) / mean)


def select_format(row_ptr):
    """("sell", 1), ("sell", SIGMA_SORTED) or ("csr", 0) by the CV bands."""
    cv = row_length_cv(row_ptr)
    if cv < CV_ELL:
        return "sell", 1
    if cv <= CV_CSR:
        return "sell", SIGMA_SORTED
    return "csr", 0


@dataclass
class SellMatrix:
    n_rows: int
    n_cols: int
    C: int
    sigma: int
    slice_ptr: np.ndarray   # int64[n_slices + 1], slot offsets
    perm: np.ndarray        # int64[n_slices * C], original row or -1
    cols: np.ndarray        # int32[slots]
    vals: np.ndarray        # values' dtype, [slots]

    @property
    def n_slices(self) -> int:
        return self.slice_ptr.size - 1

    @property
    def n_slots(self) -> int:
        return int(self.slice_ptr[-1])


def sell_order(lengths: np.ndarray, sigma: int) -> np.ndarray:
    """Rows in sorted position order: inside each window of sigma rows, by
    decreasing length, ties by row index."""
    n = lengths.size
    order = np.arange(n, dtype=np.int64)
    if sigma > 1:
        for w0 in range(0, n, sigma):
            w1 = min(n, w0 + sigma)
            # stable sort on -length keeps the row order among equal lengths
            order[w0:w1] = w0 + np.argsort(-lengths[w0:w1], kind="stable")
    return order


def sell_encode(n_cols, row_ptr, col_idx, values, C: int = 32, sigma: int = 1) -> SellMatrix:
    rp = np.asarray(row_ptr, dtype=np.int64)
    ci = np.asarray(col_idx, dtype=np.int32)
    vals = np.asarray(values)
    n = rp.size - 1
    lengths = np.diff(rp)
    order = sell_order(lengths, sigma)
    n_slices = (n + C - 1) // C
    perm = np.full(n_slices * C, -1, dtype=np.int64)
    perm[:n] = order
    # width of each slice: its longest row
    padded_len = np.zeros(n_slices * C, dtype=np.int64)
    padded_len[:n] = lengths[order]
    widths = padded_len.reshape(n_slices, C).max(axis=1) if n_slices else np.zeros(0, np.int64)
    slice_ptr = np.zeros(n_slices + 1, dtype=np.int64)
    slice_ptr[1:] = np.cumsum(widths * C)
    slots = int(slice_ptr[-1])
    cols = np.zeros(slots, dtype=np.int32)
    out_vals = np.zeros(slots, dtype=vals.dtype)
    for s in range(n_slices):
        for lane in range(C):
            i = perm[s * C + lane]
            if i < 0:
                continue
            length = int(lengths[i])
            k = np.arange(widths[s])
            at = slice_ptr[s] + k * C + lane
            real = k < length
            cols[at[real]] = ci[rp[i]:rp[i + 1]]
            out_vals[at[real]] = vals[rp[i]:rp[i + 1]]
            if length > 0:
                cols[at[~real]] = ci[rp[i + 1] - 1]
    return SellMatrix(n, int(n_cols), C, sigma, slice_ptr, perm, cols, out_vals)


def sell_spmv(m: SellMatrix, x, with_abs: bool = True):
    """fp64 y = A x read from the sliced layout: for each row, its slots in k
    order (padding included), gathered back to CSR and summed by csr_spmv."""
    row_ptr = np.zeros(m.n_rows + 1, dtype=np.int64)
    cols, vals = [], []
    per_row = [None] * m.n_rows
    for s in range(m.n_slices):
        w = (m.slice_ptr[s + 1] - m.slice_ptr[s]) // m.C
        for lane in range(m.C):
            i = m.perm[s * m.C + lane]
            if i < 0:
                continue
            at = m.slice_ptr[s] + np.arange(w) * m.C + lane
            per_row[i] = at
    for i in range(m.n_rows):
        at = per_row[i] if per_row[i] is not None else np.zeros(0, np.int64)
        cols.append(m.cols[at])
        vals.append(m.vals[at])
        row_ptr[i + 1] = row_ptr[i] + at.size
    c = np.concatenate(cols) if cols else np.zeros(0, np.int32)
    v = np.concatenate(vals) if vals else np.zeros(0, m.vals.dtype)
    return csr_spmv(row_ptr, c, v, x, with_abs=with_abs)


def sell_slot_count(row_ptr, C: int = 32, sigma: int = 1) -> tuple:
    """(slots, slices) of the sliced layout, from the row lengths alone."""
    lengths = np.diff(np.asarray(row_ptr, dtype=np.int64))
    n = lengths.size
    n_slices = (n + C - 1) // C
    padded = np.zeros(n_slices * C, dtype=np.int64)
    padded[:n] = lengths[sell_order(lengths, sigma)]
    widths = padded.reshape(n_slices, C).max(axis=1) if n_slices else padded[:0]
    return int(widths.sum()) * C, n_slices
