"""CPU tests of the C ABI: the library loads, exports every function that
include/spmv.h declares, its structs match the C layout, host-side
validation and the DELTA converter (2-, 4- and 8-bit deltas) behave, and the planner's bins are
consistent. Nothing here launches a kernel."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import workloads
from sparse_matrix_vector_gb300 import _lib
import sparse_matrix_vector_gb300 as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spmv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(spmv_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_function_is_exported(spmv_lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(spmv_lib, n), n
    assert set(names) == set(_lib.SIGNATURES)


def test_abi_version_and_status_strings(spmv_lib):
    assert S.spmv_abi_version() == 6
    for code in range(11):
        s = S.spmv_status_string(code)
        assert s and s != "unknown status"
    assert S.spmv_status_string(99) == "unknown status"


STRUCTS = {
    "spmv_csr": _lib.spmv_csr, "spmv_delta": _lib.spmv_delta,
    "spmv_sell": _lib.spmv_sell, "spmv_fem_mesh": _lib.spmv_fem_mesh,
    "spmv_pcg_result": _lib.spmv_pcg_result,
    "spmv_plan_options": _lib.spmv_plan_options,
    "spmv_plan_info": _lib.spmv_plan_info,
}


def test_struct_layout_matches_c(tmp_path):
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "spmv.h"',
             'int main(void) {']
    for cname, ct in STRUCTS.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in ct._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe),
                    str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True,
                         text=True).stdout.split("\n")
    got = {}
    for line in out:
        if line:
            s, f, v = line.split()
            got[(s, f)] = int(v)
    for cname, ct in STRUCTS.items():
        assert got[(cname, "size")] == ctypes.sizeof(ct), cname
        for f, _ in ct._fields_:
            assert got[(cname, f)] == getattr(ct, f).offset, (cname, f)


def _csr(rp, ci, vals, n_cols):
    return S.api._host_csr(np.asarray(rp), np.asarray(ci), np.asarray(vals), n_cols)


@pytest.mark.parametrize("rp,ci,n_cols,err", [
    ([1, 2], [0, 0], 4, 2),            # row_ptr[0] != 0
    ([0, 2, 1], [0, 1], 4, 2),         # decreasing
    ([0, 1], [0, 1], 4, 2),            # last != nnz
    ([0, 2], [0, 4], 4, 3),            # column == n_cols
    ([0, 2], [-1, 1], 4, 3),           # negative column
])
def test_validation_errors(spmv_lib, rp, ci, n_cols, err):
    vals = np.ones(len(ci), np.float32)
    h = _csr(rp, ci, vals, n_cols)
    h.struct.nnz = len(ci)
    info = _lib.spmv_plan_info()
    st = spmv_lib.spmv_plan_inspect(ctypes.byref(h.struct), 0, None,
                                    ctypes.byref(info))
    assert st == err
    out = ctypes.c_void_p()
    # validation comes before any device call, so this needs no GPU
    st = spmv_lib.spmv_plan_create(ctypes.byref(h.struct), 0, ctypes.byref(out))
    assert st == err and not out.value


def test_delta_needs_sorted_fp16(spmv_lib):
    with pytest.raises(S.SpmvError) as e:
        S.spmv_convert([0, 3], [1, 5, 3], np.ones(3, np.float16), 10)
    assert e.value.status == 4
    with pytest.raises(S.SpmvError) as e:
        S.spmv_convert([0, 2], [1, 1], np.ones(2, np.float16), 10)
    assert e.value.status == 4
    with pytest.raises(S.SpmvError) as e:
        S.spmv_convert([0, 2], [1, 2], np.ones(2, np.float32), 10)
    assert e.value.status == 5
    # CSR accepts unsorted and repeated columns
    S.spmv_plan_inspect([0, 3], [5, 1, 5], np.ones(3, np.float32), 10)


def test_null_and_bad_args(spmv_lib):
    info = _lib.spmv_plan_info()
    assert spmv_lib.spmv_plan_inspect(None, 0, None, ctypes.byref(info)) == 1
    h = _csr([0, 1], [0], np.ones(1, np.float32), 1)
    assert spmv_lib.spmv_plan_inspect(ctypes.byref(h.struct), 7, None,
                                      ctypes.byref(info)) == 1
    h.struct.value_dtype = 5
    assert spmv_lib.spmv_plan_inspect(ctypes.byref(h.struct), 0, None,
                                      ctypes.byref(info)) == 1
    assert spmv_lib.spmv_run(None, None, None, None) == 1
    assert spmv_lib.spmv_run_host(None, None, None, None) == 1
    assert spmv_lib.spmv_run_host_batch(None, 1, None, None, None) == 1
    assert spmv_lib.spmv_plan_check(None) == 1
    spmv_lib.spmv_plan_destroy(None)
    d = _lib.spmv_delta()
    spmv_lib.spmv_delta_free(ctypes.byref(d))
    assert spmv_lib.spmv_convert(None, ctypes.byref(d)) == 1
    h = _csr([0, 1], [0], np.ones(1, np.float16), 4)
    for bad in (0, 1, 3, 16, -4):
        assert spmv_lib.spmv_convert_bits(ctypes.byref(h.struct), bad, ctypes.byref(d)) == 1
    # a DELTA matrix whose width is not 2, 4 or 8 is refused before any
    # device call
    d = _lib.spmv_delta(n_rows=0, n_cols=4, row_ptr=ctypes.addressof(c_zero), delta_bits=3)
    out = ctypes.c_void_p()
    assert spmv_lib.spmv_plan_create_delta(ctypes.byref(d), None, ctypes.byref(out)) == 1
    assert not out.value


c_zero = ctypes.c_int64(0)


def _converter_matches_oracle(m, n_cols=None, bits=4):
    n_cols = m.n_cols if n_cols is None else n_cols
    got = S.spmv_convert(m.row_ptr, m.col_idx, m.values, n_cols, bits=bits)
    ref = oracle.delta_encode(n_cols, m.row_ptr, m.col_idx, m.values, bits=bits)
    assert got.bits == bits
    assert np.array_equal(got.row_ptr, ref.row_ptr)
    assert np.array_equal(got.values, ref.values)
    assert np.array_equal(got.words, ref.words)
    assert got.n_gap_pads == ref.gap_pads and got.n_align_pads == ref.align_pads
    assert got.nnz == m.nnz
    return got


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("sparsity", [0.3, 0.5, 0.7, 0.9, 0.99])
def test_converter_bit_exact_llm_small(spmv_lib, sparsity, bits):
    _converter_matches_oracle(workloads.llm(sparsity, n=700), bits=bits)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_converter_bit_exact_edge_rows(spmv_lib, bits):
    lengths = np.array([0, 1, 8, 7, 9, 0, 0, 16, 33, 1, 2000])
    m = workloads.from_lengths("edges", lengths, 5000, seed=9, dtype=np.float16)
    _converter_matches_oracle(m, bits=bits)
    # first column 0, exact multiples of 3, 15 and 255, a gap spanning the
    # whole row
    rp = np.array([0, 6, 8, 9], np.int32)
    ci = np.array([0, 3, 15, 30, 255, 510, 0, 4999, 2999], np.int32)
    vals = np.arange(1, 10).astype(np.float16)
    m = workloads.CSRInput("hand", 3, 5000, rp, ci, vals, np.zeros(5000, np.float16))
    _converter_matches_oracle(m, bits=bits)
    # explicit +0.0 values are stored as such and counted
    vals0 = vals.copy()
    vals0[2] = 0
    got = S.spmv_convert(rp, ci, vals0, 5000, bits=bits)
    assert got.n_explicit_zeros == 1


@pytest.mark.slow
def test_converter_bit_exact_llm_full(spmv_lib):
    _converter_matches_oracle(workloads.llm(0.9))


def effective(opts, cap=2048):
    """The planner's limits after defaults (0 fields) and clamps, for a
    stage of `cap` nonzeros (2048): tile_nnz <= cap - 16, single-row tiles
    by default above half of that, rows that are not split fit one stage,
    chunks of 64..cap nonzeros."""
    tile_nnz = min(opts.tile_nnz or cap - 16, cap - 16)
    cta = min(opts.cta_row_min or (cap - 16) // 2, tile_nnz)
    srm = min(max(opts.split_row_min or cap, cta), cap)
    chunk = min(max(opts.split_chunk, 64), cap) if opts.split_chunk else cap
    return tile_nnz, cta, srm, chunk, opts.tile_rows or 512


def expected_bins(lengths, opts):
    """Bins and tiles the planner must produce, from the row lengths alone."""
    tile_nnz, cta, srm, chunk, tile_rows = effective(opts)
    split = lengths > srm
    single = (lengths > cta) & ~split
    bins = [int(np.sum((lengths <= 8) & ~split)),
            int(np.sum((lengths > 8) & (lengths <= 256) & ~split)),
            int(np.sum((lengths > 256) & ~split)), int(split.sum())]
    chunks = int(np.sum((lengths[split] + chunk - 1) // chunk))
    return bins, int(single.sum()), chunks, tile_nnz, cta, tile_rows


@pytest.mark.parametrize("kw", [{}, {"cta_row_min": 32},
                                {"cta_row_min": 200, "split_row_min": 300,
                                 "split_chunk": 128},
                                {"tile_nnz": 300, "tile_rows": 64}])
def test_planner_bins(spmv_lib, kw):
    m = workloads.powerlaw(n=40000, nnz=223000, max_len=2500)
    opts = S.spmv_plan_options(csr_kernel=1, **kw)
    info = S.spmv_plan_inspect(m.row_ptr, m.col_idx, m.values, m.n_cols,
                               options=opts)
    L = m.row_lengths()
    bins, n_single, n_chunks, tile_nnz, cta, tile_rows = expected_bins(L, opts)
    assert info["rows_per_bin"] == bins
    assert sum(info["rows_per_bin"]) == m.n_rows
    assert info["tiles_per_bin"][2] == n_single
    assert info["tiles_per_bin"][3] == n_chunks
    assert info["n_split_rows"] == bins[3]
    short = L[L <= cta]
    min_tiles = max(int(np.ceil(short.sum() / tile_nnz)),
                    int(np.ceil(short.size / tile_rows)))
    assert info["tiles_per_bin"][0] >= min_tiles
    assert info["n_tiles"] == sum(info["tiles_per_bin"])
    assert info["algorithmic_bytes"] == (8 * m.nnz + 4 * (m.n_rows + 1)
                                         + 4 * m.n_cols + 4 * m.n_rows)


def test_planner_bins_of_the_workload_shapes(spmv_lib):
    lap = workloads.laplacian(300, 200)
    info = S.spmv_plan_inspect(lap.row_ptr, lap.col_idx, lap.values, lap.n_cols)
    assert info["rows_per_bin"] == [lap.n_rows, 0, 0, 0]   # sub-warp
    assert info["walk_tiles"] == 0                           # regular rows: lanes mode
    pl = workloads.powerlaw(n=300000, nnz=1_670_000, max_len=2500)
    info = S.spmv_plan_inspect(pl.row_ptr, pl.col_idx, pl.values, pl.n_cols,
                               options=S.spmv_plan_options(csr_kernel=1))
    assert info["walk_tiles"] > 0                            # irregular rows: walk mode
    for reduce, walk in ((1, 0), (2, info["tiles_per_bin"][0])):
        forced = S.spmv_plan_inspect(pl.row_ptr, pl.col_idx, pl.values, pl.n_cols,
                                     options=S.spmv_plan_options(reduce=reduce, lanes=4,
                                                                 csr_kernel=1))
        assert forced["walk_tiles"] == walk
    # by default the irregular rows (CV > 2) take mixed warp segments: runs of
    # whole rows packed 256 nonzeros to a segment, longer rows sliced by 256
    info = S.spmv_plan_inspect(pl.row_ptr, pl.col_idx, pl.values, pl.n_cols)
    assert info["segments"] == 1
    L = pl.row_lengths()
    long_rows = L[L > 256]
    assert info["tiles_per_bin"][2] + info["tiles_per_bin"][3] == (-(-long_rows // 256)).sum()
    assert info["rows_per_bin"][1] + info["rows_per_bin"][2] + info["rows_per_bin"][3] >= \
        long_rows.size
    fem = workloads.fem(6, 5, 4)
    info = S.spmv_plan_inspect(fem.row_ptr, fem.col_idx, fem.values, fem.n_cols)
    assert info["rows_per_bin"] == [0, fem.n_rows, 0, 0]   # warp
    llm = workloads.llm(0.3, n=2048)
    tiles = S.spmv_plan_options(csr_kernel=1)
    info = S.spmv_plan_inspect(llm.row_ptr, llm.col_idx, llm.values, llm.n_cols, options=tiles)
    assert info["rows_per_bin"] == [0, 0, llm.n_rows, 0]   # CTA
    assert info["x_in_smem"] == 0 and info["segments"] == 0  # x via L1 by default
    forced = S.spmv_plan_inspect(llm.row_ptr, llm.col_idx, llm.values, llm.n_cols,
                                 options=S.spmv_plan_options(x_smem=1, csr_kernel=1))
    assert forced["x_in_smem"] == 1
    big = workloads.llm(0.3, n=6144)   # ~4300 nonzeros per row > one stage (2048)
    info = S.spmv_plan_inspect(big.row_ptr, big.col_idx, big.values, big.n_cols, options=tiles)
    assert info["rows_per_bin"] == [0, 0, 0, big.n_rows]   # split
    # rows averaging >= 256 nonzeros take warp segments of <= 512 by default
    info = S.spmv_plan_inspect(llm.row_ptr, llm.col_idx, llm.values, llm.n_cols)
    lengths = llm.row_lengths()
    segs = -(-lengths // 512)
    assert info["segments"] == 1 and info["n_tiles"] == segs.sum()
    assert info["rows_per_bin"][3] == (segs > 1).sum()
    assert info["x_in_smem"] == 1                            # 4 KB of fp16 x
    assert info["algorithmic_bytes"] == (6 * llm.nnz + 4 * (llm.n_rows + 1)
                                         + 2 * llm.n_cols + 4 * llm.n_rows)
    info = S.spmv_plan_inspect(llm.row_ptr, llm.col_idx, llm.values, llm.n_cols,
                               format="delta4")
    enc = oracle.delta_encode(llm.n_cols, llm.row_ptr, llm.col_idx, llm.values)
    assert info["n_entries"] == enc.n_entries
    assert info["matrix_bytes"] == 2 * enc.n_entries + enc.n_entries // 2 + 4 * (llm.n_rows + 1)
    for bits in (2, 8):
        info = S.spmv_plan_inspect(llm.row_ptr, llm.col_idx, llm.values, llm.n_cols,
                                   format=f"delta{bits}")
        enc = oracle.delta_encode(llm.n_cols, llm.row_ptr, llm.col_idx, llm.values,
                                  bits=bits)
        assert info["format"] == {2: 2, 8: 3}[bits]
        assert info["n_entries"] == enc.n_entries
        assert info["matrix_bytes"] == (2 * enc.n_entries + enc.n_entries * bits // 8
                                        + 4 * (llm.n_rows + 1))


def test_gather_order_choice(spmv_lib):
    """Element-interleaved products where rows are long and 8 nonzeros of a
    row span over 40 bytes of x; chunks of 8 otherwise; options force."""
    lap = workloads.laplacian(60, 50)
    info = S.spmv_plan_inspect(lap.row_ptr, lap.col_idx, lap.values, lap.n_cols)
    assert info["interleaved"] == 0                      # rows of 5
    sparse = workloads.llm(0.9, n=2048)
    info = S.spmv_plan_inspect(sparse.row_ptr, sparse.col_idx, sparse.values, sparse.n_cols)
    assert info["interleaved"] == 1                      # ~80 fp16 columns per 8
    dense = workloads.llm(0.3, n=2048)
    info = S.spmv_plan_inspect(dense.row_ptr, dense.col_idx, dense.values, dense.n_cols)
    assert info["interleaved"] == 0                      # ~11 columns per 8
    for force, want in ((1, 0), (2, 1)):
        info = S.spmv_plan_inspect(sparse.row_ptr, sparse.col_idx, sparse.values,
                                   sparse.n_cols,
                                   options=S.spmv_plan_options(interleave=force))
        assert info["interleaved"] == want
        info = S.spmv_plan_inspect(lap.row_ptr, lap.col_idx, lap.values, lap.n_cols,
                                   options=S.spmv_plan_options(interleave=force))
        assert info["interleaved"] == want


def test_empty_and_degenerate_inspect(spmv_lib):
    info = S.spmv_plan_inspect(np.zeros(1, np.int32), np.zeros(0, np.int32),
                               np.zeros(0, np.float32), 0)
    assert info["n_tiles"] == 0 and info["launches_per_run"] == 0
    info = S.spmv_plan_inspect(np.zeros(5001, np.int32), np.zeros(0, np.int32),
                               np.zeros(0, np.float32), 3)
    assert sum(info["rows_per_bin"]) == 5000 and info["n_tiles"] >= 5


@pytest.mark.parametrize("sparsity", [0.1, 0.3, 0.5, 0.7, 0.9, 0.97])
def test_delta_width_selection(spmv_lib, sparsity):
    """The entry counts behind the choice equal the oracle encoder's at each
    width; the fewest-bytes choice is the width that stores the fewest bytes
    (ties to the wider field); the sparsity table follows the printed rows."""
    m = workloads.llm(sparsity, n=600, seed=12)
    bits, entries = S.spmv_delta_select_bits(m.row_ptr, m.col_idx, m.values, m.n_cols)
    stored = {}
    for b in (2, 4, 8):
        enc = oracle.delta_encode(m.n_cols, m.row_ptr, m.col_idx, m.values, bits=b)
        assert entries[b] == enc.n_entries
        stored[b] = enc.n_entries * 2 + enc.n_entries * b // 8
    best = min(stored.values())
    assert bits == max(b for b in stored if stored[b] == best)
    table, _ = S.spmv_delta_select_bits(m.row_ptr, m.col_idx, m.values, m.n_cols,
                                        policy="sparsity_table")
    s = 1.0 - m.nnz / (m.n_rows * m.n_cols)
    assert table == (8 if s < 0.3 else 4 if s <= 0.7 else 2)
    info = S.spmv_plan_inspect(m.row_ptr, m.col_idx, m.values, m.n_cols, format="delta")
    assert info["format"] == {4: 1, 2: 2, 8: 3}[bits]
    assert info["n_entries"] == entries[bits]


def test_delta_width_selection_errors(spmv_lib):
    with pytest.raises(S.SpmvError) as e:
        S.spmv_delta_select_bits([0, 2], [1, 2], np.ones(2, np.float32), 4)
    assert e.value.status == 5
    with pytest.raises(S.SpmvError) as e:
        S.spmv_delta_select_bits([0, 2], [2, 1], np.ones(2, np.float16), 4)
    assert e.value.status == 4
    with pytest.raises(S.SpmvError) as e:
        S.spmv_delta_select_bits([0, 2], [1, 2], np.ones(2, np.float16), 4, policy=7)
    assert e.value.status == 1
    # an empty matrix: every width stores nothing; ties go to 8 bits
    bits, entries = S.spmv_delta_select_bits([0, 0], [], np.zeros(0, np.float16), 4)
    assert bits == 8 and entries == {2: 0, 4: 0, 8: 0}


def _sell_matches_oracle(m, sigma):
    from oracle import sell
    got = S.spmv_convert_sell(m.row_ptr, m.col_idx, m.values, m.n_cols, sigma=sigma)
    ref = sell.sell_encode(m.n_cols, m.row_ptr, m.col_idx, m.values, C=32, sigma=sigma)
    assert got.C == 32 and got.sigma == sigma and got.nnz == m.nnz
    assert np.array_equal(got.slice_ptr, ref.slice_ptr)
    assert np.array_equal(got.perm.astype(np.int64), ref.perm)
    assert np.array_equal(got.cols, ref.cols)
    assert got.values.dtype == ref.vals.dtype
    assert np.array_equal(got.values.view(np.uint8), ref.vals.view(np.uint8))
    return got


@pytest.mark.parametrize("sigma", [1, 7, 1024])
@pytest.mark.parametrize("name", ["tiny", "laplacian", "powerlaw", "fem", "llm", "edges"])
def test_sell_converter_bit_exact(spmv_lib, name, sigma):
    if name == "tiny":
        m = workloads.tiny()
    elif name == "laplacian":
        m = workloads.laplacian(70, 41)
    elif name == "powerlaw":
        m = workloads.powerlaw(n=3000, nnz=16700, max_len=400, seed=4)
    elif name == "fem":
        m = workloads.fem(5, 4, 3)
    elif name == "llm":
        m = workloads.llm(0.8, n=300, seed=2)
    else:
        lengths = np.array([0, 1, 8, 7, 9, 0, 0, 16, 33, 1, 200, 0, 3])
        m = workloads.from_lengths("edges", lengths, 500, seed=9)
    _sell_matches_oracle(m, sigma)


def test_sell_converter_unsorted_and_errors(spmv_lib):
    # CSR order is kept inside a row, repeats included
    rp = np.array([0, 3, 3, 5], np.int32)
    ci = np.array([5, 1, 5, 0, 2], np.int32)
    vals = np.arange(1, 6).astype(np.float32)
    m = workloads.CSRInput("unsorted", 3, 6, rp, ci, vals, np.zeros(6, np.float32), {})
    got = _sell_matches_oracle(m, 1)
    assert got.cols[:3 * 32:32].tolist() == [5, 1, 5]
    with pytest.raises(S.SpmvError) as e:
        S.spmv_convert_sell(rp, ci, vals, 6, sigma=0)
    assert e.value.status == 1
    with pytest.raises(S.SpmvError) as e:
        S.spmv_convert_sell(rp, ci, vals, 5, sigma=1)
    assert e.value.status == 3
    empty = S.spmv_convert_sell(np.zeros(1, np.int32), np.zeros(0, np.int32),
                                np.zeros(0, np.float32), 4)
    assert empty.slice_ptr.tolist() == [0] and empty.cols.size == 0


@pytest.mark.parametrize("name", ["tiny", "laplacian", "powerlaw", "fem", "llm", "ragged"])
def test_format_choice_matches_oracle(spmv_lib, name):
    from oracle import sell
    m = {"tiny": lambda: workloads.tiny(),
         "laplacian": lambda: workloads.laplacian(70, 41),
         "powerlaw": lambda: workloads.powerlaw(n=3000, nnz=16700, max_len=400, seed=4),
         "fem": lambda: workloads.fem(5, 4, 3),
         "llm": lambda: workloads.llm(0.8, n=300, seed=2),
         "ragged": lambda: workloads.from_lengths("ragged", np.tile([3, 6, 9, 12], 50), 40,
                                                  seed=3)}[name]()
    fmt, sigma, cv = S.spmv_select_format(m.row_ptr, m.col_idx, m.values, m.n_cols)
    assert abs(cv - sell.row_length_cv(m.row_ptr)) <= 1e-12 * max(cv, 1.0)
    assert (fmt, sigma) == sell.select_format(m.row_ptr)
    info = S.spmv_plan_inspect(m.row_ptr, m.col_idx, m.values, m.n_cols, format="auto")
    off_band = m.nnz > 128 * m.n_rows or m.nnz < 16 * m.n_rows
    assert info["format"] == S.api.FORMATS["csr" if off_band else fmt]
    if fmt == "sell" and not off_band:
        ref = sell.sell_encode(m.n_cols, m.row_ptr, m.col_idx, m.values, C=32, sigma=sigma)
        assert info["n_entries"] == ref.n_slots and info["n_tiles"] == ref.n_slices
        vs = m.values.dtype.itemsize
        assert info["matrix_bytes"] == (ref.n_slots * (4 + vs) + (ref.n_slices + 1) * 4
                                        + (ref.n_slices * 32 * 4 if sigma > 1 else 0))
    # a SELL forced with explicit sigma keeps it
    info = S.spmv_plan_inspect(m.row_ptr, m.col_idx, m.values, m.n_cols, format="sell",
                               options=S.spmv_plan_options(sell_sigma=64))
    ref = sell.sell_encode(m.n_cols, m.row_ptr, m.col_idx, m.values, C=32, sigma=64)
    assert info["format"] == 5 and info["n_entries"] == ref.n_slots


def test_auto_format_sends_long_rows_to_csr(spmv_lib):
    """The CV band alone would give these uniform rows of ~1000 nonzeros to
    SELL; AUTO keeps rows longer than 128 on average in CSR."""
    m = workloads.llm(0.5, n=2048)
    fmt, _, cv = S.spmv_select_format(m.row_ptr, m.col_idx, m.values, m.n_cols)
    assert fmt == "sell" and cv < 0.3
    info = S.spmv_plan_inspect(m.row_ptr, m.col_idx, m.values, m.n_cols, format="auto")
    assert info["format"] == 0


def test_auto_format_sends_short_rows_to_csr(spmv_lib):
    """The 5-point Laplacian's rows have CV < 0.3, the ELL band, but average
    5 nonzeros: AUTO keeps rows shorter than 16 on average in CSR, and still
    gives the stiffness matrix's ~78-long rows to SELL."""
    m = workloads.laplacian(70, 41)
    fmt, _, cv = S.spmv_select_format(m.row_ptr, m.col_idx, m.values, m.n_cols)
    assert fmt == "sell" and cv < 0.3
    info = S.spmv_plan_inspect(m.row_ptr, m.col_idx, m.values, m.n_cols, format="auto")
    assert info["format"] == 0
    f = workloads.fem(5, 4, 3)
    info = S.spmv_plan_inspect(f.row_ptr, f.col_idx, f.values, f.n_cols, format="auto")
    assert info["format"] == 5


def test_fem_plan_argument_errors(spmv_lib):
    """Bad meshes are refused on the host, before any device call."""
    k0 = np.eye(24, dtype=np.float32)
    out = ctypes.c_void_p()
    for dims in ((0, 1, 1), (1, -1, 1), (2, 2, 0)):
        rho = np.ones(max(1, dims[0] * dims[1] * dims[2]), np.float32)
        mesh = _lib.spmv_fem_mesh(nex=dims[0], ney=dims[1], nez=dims[2],
                                  rho=rho.ctypes.data, K0=k0.ctypes.data)
        assert spmv_lib.spmv_plan_create_fem(ctypes.byref(mesh), ctypes.byref(out)) == 1
    rho = np.ones(8, np.float32)
    bad_k = k0.copy()
    bad_k[3, 4] = np.inf
    bad_r = rho.copy()
    bad_r[5] = np.nan
    for r, k in ((bad_r, k0), (rho, bad_k)):
        mesh = _lib.spmv_fem_mesh(nex=2, ney=2, nez=2, rho=r.ctypes.data, K0=k.ctypes.data)
        assert spmv_lib.spmv_plan_create_fem(ctypes.byref(mesh), ctypes.byref(out)) == 1
    mesh = _lib.spmv_fem_mesh(nex=2, ney=2, nez=2, rho=None, K0=k0.ctypes.data)
    assert spmv_lib.spmv_plan_create_fem(ctypes.byref(mesh), ctypes.byref(out)) == 1
    mesh = _lib.spmv_fem_mesh(nex=2000, ney=2000, nez=2000, rho=rho.ctypes.data,
                              K0=k0.ctypes.data)
    assert spmv_lib.spmv_plan_create_fem(ctypes.byref(mesh), ctypes.byref(out)) == 8
    assert not out.value


def test_pcg_argument_errors(spmv_lib):
    """A NULL plan or result pointer is refused without touching a device."""
    res = _lib.spmv_pcg_result()
    assert spmv_lib.spmv_pcg_solve(None, None, None, None, 1e-6, 10, 0, None,
                                   ctypes.byref(res)) == 1
    assert spmv_lib.spmv_pcg_solve(None, None, None, None, 1e-6, 10, 0, None, None) == 1


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_delta_planner_unit_counts(spmv_lib, bits):
    """Every row becomes ceil(words / segment words) segments (none for an
    empty row); segments hold at most 64 words at 2 bits and 128 otherwise;
    only rows of more than one segment can be shared by several warps."""
    lengths = np.array([0, 1, 7, 300, 2000, 5000, 12000, 0, 4096, 4097, 8193])
    m = workloads.from_lengths("units", lengths, 20000, seed=5, dtype=np.float16)
    info = S.spmv_plan_inspect(m.row_ptr, m.col_idx, m.values, m.n_cols, format=f"delta{bits}")
    enc = oracle.delta_encode(m.n_cols, m.row_ptr, m.col_idx, m.values, bits=bits)
    words = np.diff(enc.row_ptr) * bits // 32
    seg_words = 64 if bits == 2 else 128
    segs = -(-words // seg_words)
    assert info["n_tiles"] == segs.sum()
    assert info["tiles_per_bin"][2] == (segs == 1).sum()
    assert info["tiles_per_bin"][3] == segs[segs > 1].sum()
    assert info["rows_per_bin"][3] == (segs > 1).sum()
    assert 0 <= info["n_split_rows"] <= (segs > 1).sum()
    assert info["block"] % 32 == 0
    assert info["n_entries"] == enc.n_entries
