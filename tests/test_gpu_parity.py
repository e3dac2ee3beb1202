"""GPU parity: the library's kernels (through the C ABI) against the fp64
oracle, element by element, on the seeded workloads and on edge cases.

Tolerances (per row i, s_i = sum_j |a_ij x_j| from the oracle):
  fp32 CSR:                   |y - y_ref| <= 1e-5 * s_i + 1e-30
  fp16 values (CSR, DELTA):   |y - y_ref| <= 2e-3 * s_i
"""
import functools

import numpy as np
import scipy.sparse as sp
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
S = pytest.importorskip("sparse_matrix_vector_gb300")

pytestmark = pytest.mark.gpu

TOL32 = 1e-5
TOL16 = 2e-3
DELTAS = ["delta2", "delta4", "delta8"]
FORMAT_CODE = {"csr": 0, "delta4": 1, "delta2": 2, "delta8": 3, "sell": 5}


@functools.lru_cache(maxsize=None)
def full(name):
    return workloads.make(name)


_REF = {}


def reference(m):
    """Oracle result for a workload object (cached by identity)."""
    hit = _REF.get(id(m))
    if hit is None or hit[0] is not m:
        hit = (m, oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, m.x))
        _REF[id(m)] = hit
    return hit[1]


def run_gpu(m, fmt="csr", options=None, x=None, stream=None, repeat=1):
    dev = torch.device("cuda", 0)
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols,
                              format=fmt, options=options)
    xt = torch.from_numpy(np.ascontiguousarray(m.x if x is None else x)).to(dev)
    outs = []
    for _ in range(repeat):
        y = torch.full((m.n_rows,), float("nan"), dtype=torch.float32, device=dev)
        S.spmv_run(plan, xt, y, stream=stream)
        outs.append(y)
    torch.cuda.synchronize()
    S.spmv_plan_check(plan)
    info = plan.info
    S.spmv_plan_destroy(plan)
    ys = [o.cpu().numpy() for o in outs]
    return (ys if repeat > 1 else ys[0]), info


def assert_parity(m, y, tol, y_ref=None, s=None):
    if y_ref is None:
        y_ref, s = reference(m)
    y = y.astype(np.float64)
    assert y.shape == y_ref.shape
    assert np.all(np.isfinite(y)), "non-finite outputs (unwritten rows?)"
    err = np.abs(y - y_ref)
    bound = tol * s + 1e-30
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, (f"{m.name}: {bad.size} rows out of tolerance, first "
                           f"{bad[:5]}, max |dy|/s = {np.max(err / np.maximum(s, 1e-300)):.3e}")


def tol_for(m):
    return TOL32 if m.values.dtype == np.float32 else TOL16


# ------------------------------------------------------------ the workloads

SMALL = {
    "tiny": lambda: workloads.tiny(),
    "laplacian_small": lambda: workloads.laplacian(300, 211),
    "powerlaw_small": lambda: workloads.powerlaw(n=50000, nnz=278500, max_len=4334),
    "fem_small": lambda: workloads.fem(12, 9, 7),
    "llm30_small": lambda: workloads.llm(0.3, n=1536),
    "llm90_small": lambda: workloads.llm(0.9, n=2000),
}


@functools.lru_cache(maxsize=None)
def small(name):
    return SMALL[name]()


@pytest.mark.parametrize("name", list(SMALL))
def test_small_csr(name):
    m = small(name)
    y, _ = run_gpu(m)
    assert_parity(m, y, tol_for(m))


@pytest.mark.parametrize("fmt", DELTAS)
@pytest.mark.parametrize("name", ["llm30_small", "llm90_small"])
def test_small_delta(name, fmt):
    m = small(name)
    y, info = run_gpu(m, fmt)
    assert info["format"] == FORMAT_CODE[fmt]
    assert_parity(m, y, TOL16)


@pytest.mark.parametrize("name", ["tiny", "laplacian", "powerlaw", "fem",
                                  "llm30", "llm50", "llm70", "llm90"])
def test_full_size_csr(name):
    m = full(name)
    y, info = run_gpu(m)
    assert_parity(m, y, tol_for(m))


@pytest.mark.parametrize("fmt", DELTAS)
@pytest.mark.parametrize("name", ["llm30", "llm50", "llm70", "llm90"])
def test_full_size_delta(name, fmt):
    m = full(name)
    y, info = run_gpu(m, fmt)
    assert info["n_entries"] >= m.nnz
    assert_parity(m, y, TOL16)


@pytest.mark.parametrize("kernel", [1, 2, 3])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_csr_every_kernel(name, kernel):
    """Each CSR kernel forced on every small shape: CTA tiles (1), warp
    segments (2, rows cut into slices of at most 512 nonzeros) and mixed warp
    segments (3, runs of short rows packed, longer rows in slices of 256)."""
    m = small(name)
    y, info = run_gpu(m, options=S.spmv_plan_options(csr_kernel=kernel))
    assert info["segments"] == (1 if kernel >= 2 else 0)
    assert_parity(m, y, tol_for(m))


@pytest.mark.parametrize("kernel", [1, 2, 3])
@pytest.mark.parametrize("name", ["laplacian", "llm30", "llm90", "fem", "powerlaw"])
def test_full_size_csr_every_kernel(name, kernel):
    m = full(name)
    y, info = run_gpu(m, options=S.spmv_plan_options(csr_kernel=kernel))
    assert_parity(m, y, tol_for(m))


@pytest.mark.parametrize("x_smem", [0, 1])
def test_csr_mixed_segments_edge_rows(x_smem):
    """Packed runs: 300 empty rows in a row (more than one run), rows of 16
    (summed by one lane) and 17 to 256 (summed by the warp) nonzeros, a run
    ending exactly at 256 nonzeros, rows of 257+ (sliced) between runs, an
    empty last row; fp32 and fp16, repeated runs bit-identical."""
    lengths = np.concatenate([[0] * 300, [32] * 8, [16, 17], [1] * 7, [31, 1], [256, 600, 0, 5],
                              np.tile([1, 2, 0, 16, 32, 257, 3, 100, 200], 20), [1000, 4], [0]])
    opts = S.spmv_plan_options(csr_kernel=3, x_smem=x_smem)
    for dtype, tol in ((np.float32, TOL32), (np.float16, TOL16)):
        m = workloads.from_lengths("packed_edges", lengths, 3000, seed=4, dtype=dtype)
        ys, info = run_gpu(m, options=opts, repeat=3)
        assert info["segments"] == 1
        assert info["x_in_smem"] == x_smem
        for y in ys:
            assert_parity(m, y, tol)
        assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])


@pytest.mark.parametrize("x_smem", [0, 1])
def test_csr_segments_edge_rows(x_smem):
    """Warp segments on rows of 0, 1, 511, 512, 513, 1024 and 30,001
    nonzeros, runs of empty rows, rows shared by several warps; repeated runs
    are bit-identical (split counters re-arm), fp32 and fp16."""
    longest, n_cols = (30001, 40000) if x_smem == 0 else (7001, 8000)  # fp16 x fits smem
    lengths = np.array([0, 1, 511, 512, 513, 0, 0, 1024, longest, 7, 0] * 9 + [2047, 0])
    opts = S.spmv_plan_options(csr_kernel=2, x_smem=x_smem)
    for dtype, tol in ((np.float32, TOL32), (np.float16, TOL16)):
        m = workloads.from_lengths("seg_edges", lengths, n_cols, seed=9, dtype=dtype)
        ys, info = run_gpu(m, options=opts, repeat=3)
        assert info["segments"] == 1 and info["n_split_rows"] > 0
        if dtype == np.float16:
            assert info["x_in_smem"] == x_smem
        for y in ys:
            assert_parity(m, y, tol)
        assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])


# ------------------------------------------------------------ forced paths

@pytest.mark.parametrize("kw", [
    {}, {"cta_row_min": 16}, {"cta_row_min": 1},
    {"cta_row_min": 100, "split_row_min": 200, "split_chunk": 64},
    {"cta_row_min": 900, "split_row_min": 1000, "split_chunk": 1000},
    {"tile_nnz": 97, "tile_rows": 13}, {"tile_nnz": 8}, {"tile_rows": 1},
    {"x_smem": 0}, {"x_smem": 1},
    {"reduce": 1, "lanes": 1}, {"reduce": 1, "lanes": 4}, {"reduce": 1, "lanes": 32},
    {"reduce": 1, "lanes": 64}, {"reduce": 1, "lanes": 256},
    {"reduce": 1, "lanes": 128, "tile_rows": 3},
    {"interleave": 2}, {"interleave": 2, "reduce": 1, "lanes": 4},
    {"interleave": 2, "cta_row_min": 100, "split_row_min": 200, "split_chunk": 64},
    {"interleave": 1},
    {"reduce": 2}, {"reduce": 2, "tile_nnz": 97},
])
def test_forced_planner_paths(kw):
    m = workloads.powerlaw(n=30000, nnz=167000, max_len=3000, seed=11)
    opts = S.spmv_plan_options(csr_kernel=1, **kw)   # the CTA-tile planner's knobs
    y, info = run_gpu(m, options=opts)
    assert_parity(m, y, TOL32)


@pytest.mark.parametrize("kw", [{"x_smem": 0}, {"x_smem": 1},
                                {"cta_row_min": 100, "split_row_min": 150,
                                 "split_chunk": 64},
                                {"cta_row_min": 2000, "reduce": 1, "lanes": 128},
                                {"interleave": 2}, {"interleave": 1}])
def test_forced_paths_fp16_csr(kw):
    m = workloads.llm(0.8, n=1000, seed=3)
    y, _ = run_gpu(m, options=S.spmv_plan_options(csr_kernel=1, **kw))
    assert_parity(m, y, TOL16)


@pytest.mark.parametrize("fmt", DELTAS)
@pytest.mark.parametrize("x_smem", [0, 1])
def test_delta_x_paths(x_smem, fmt):
    m = workloads.llm(0.6, n=3000, seed=8)
    y, info = run_gpu(m, fmt, options=S.spmv_plan_options(x_smem=x_smem))
    assert info["x_in_smem"] == x_smem
    assert_parity(m, y, TOL16)


@pytest.mark.parametrize("fmt", DELTAS)
def test_delta_mixed_rows_deterministic(fmt):
    lengths = np.tile([0, 1, 0, 3, 9, 0, 257, 0, 5000, 2, 20000, 0, 700, 64, 65], 30)
    m = workloads.from_lengths("mixed16", lengths, 30000, seed=17, dtype=np.float16)
    ys, info = run_gpu(m, fmt, repeat=3)
    assert info["n_split_rows"] > 0
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])
    assert_parity(m, ys[0], TOL16)


@pytest.mark.parametrize("dtype,kernel", [(np.float16, 2), (np.float32, 2), (np.float16, 3),
                                          (np.float32, 3)])
def test_segment_plans_split_rows_rearm(dtype, kernel):
    """CSR warp segments (long-row and mixed plans) with rows shared by two
    warps (one exchange per piece) and by many (counted): every run of the
    same plan gives the same bits, so the exchange cells and the counts are
    left empty for the next run."""
    lengths = np.tile([0, 3, 300, 450, 700, 1500, 5000, 20000, 64, 65, 257], 20)
    m = workloads.from_lengths("split16" if dtype == np.float16 else "split32", lengths, 30000,
                               seed=23, dtype=dtype)
    ys, info = run_gpu(m, options=S.spmv_plan_options(csr_kernel=kernel), repeat=4)
    assert info["n_split_rows"] > 0
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])
    assert_parity(m, ys[0], TOL16 if dtype == np.float16 else TOL32)


# ------------------------------------------------------------ edge cases

def make(name, rp, ci, vals, n_cols, x):
    return workloads.CSRInput(name, len(rp) - 1, n_cols, np.asarray(rp, np.int32),
                              np.asarray(ci, np.int32), np.asarray(vals),
                              np.asarray(x), {})


def test_empty_matrix():
    m = make("empty", [0], [], np.zeros(0, np.float32), 5, np.ones(5, np.float32))
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, 5)
    x = torch.ones(5, device="cuda")
    y = torch.empty(0, device="cuda")
    S.spmv_run(plan, x, y)
    torch.cuda.synchronize()
    assert plan.info["launches_per_run"] == 0


def test_rows_without_nonzeros():
    n = 5000
    m = make("zero_nnz", np.zeros(n + 1), [], np.zeros(0, np.float32), 7,
             np.ones(7, np.float32))
    y, _ = run_gpu(m)
    assert np.all(y == 0)


def test_one_by_one_and_single_row():
    m = make("1x1", [0, 1], [0], np.array([3.0], np.float32), 1,
             np.array([2.0], np.float32))
    y, _ = run_gpu(m)
    assert y[0] == 6.0
    n = 250_000
    rng = np.random.default_rng(4)
    m = make("one_long_row", [0, n], np.arange(n), rng.uniform(-1, 1, n).astype(np.float32),
             n, rng.uniform(-1, 1, n).astype(np.float32))
    y, info = run_gpu(m)
    assert info["rows_per_bin"][3] == 1
    assert_parity(m, y, TOL32)


@pytest.mark.parametrize("fmt", ["csr"] + DELTAS)
def test_interleaved_empty_and_long_rows(fmt):
    lengths = np.tile([0, 1, 0, 3, 9, 0, 257, 0, 5000, 2, 20000, 0], 40)
    dt = np.float32 if fmt == "csr" else np.float16
    m = workloads.from_lengths("mixed", lengths, 30000, seed=13, dtype=dt)
    ys, info = run_gpu(m, fmt, repeat=3)
    assert info["n_split_rows"] > 0          # rows cut across CTAs
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])      # partial sums added in a fixed order
    assert_parity(m, ys[0], tol_for(m))


def test_rectangular():
    m = workloads.from_lengths("wide", np.full(10, 3000), 100_000, seed=1)
    y, _ = run_gpu(m)
    assert_parity(m, y, TOL32)
    m = workloads.from_lengths("tall", np.random.default_rng(2).integers(0, 4, 100_000),
                               3, seed=2)
    y, _ = run_gpu(m)
    assert_parity(m, y, TOL32)


def test_unsorted_duplicates_and_explicit_zeros():
    rng = np.random.default_rng(6)
    n_rows, n_cols = 3000, 500
    lengths = rng.integers(0, 40, n_rows)
    rp = np.concatenate([[0], np.cumsum(lengths)])
    ci = rng.integers(0, n_cols, rp[-1])           # unsorted, with repeats
    vals = rng.uniform(-1, 1, rp[-1]).astype(np.float32)
    vals[::7] = 0.0
    m = make("unsorted", rp, ci, vals, n_cols, rng.uniform(-1, 1, n_cols).astype(np.float32))
    y, _ = run_gpu(m)
    assert_parity(m, y, TOL32)


def test_unaligned_row_starts_every_length():
    # row lengths 0..40 repeated: every start offset modulo 4 and 8 appears
    lengths = np.tile(np.arange(41), 30)
    m = workloads.from_lengths("ragged", lengths, 4096, seed=21)
    for kw in ({}, {"tile_nnz": 40}, {"tile_rows": 3}, {"cta_row_min": 8},
               {"reduce": 2}, {"reduce": 1, "lanes": 2}, {"csr_kernel": 2}, {"csr_kernel": 3}):
        y, _ = run_gpu(m, options=S.spmv_plan_options(**kw))
        assert_parity(m, y, TOL32)


def test_x_unaligned_pointer_staging():
    # x starts 4 bytes past a 16-byte boundary: scalar staging path
    m = workloads.tiny()
    dev = torch.device("cuda", 0)
    big = torch.zeros(m.n_cols + 4, dtype=torch.float32, device=dev)
    big[1:1 + m.n_cols] = torch.from_numpy(m.x).to(dev)
    x = big[1:1 + m.n_cols]
    assert x.data_ptr() % 16 == 4
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols,
                              options=S.spmv_plan_options(x_smem=1))
    y = torch.empty(m.n_rows, dtype=torch.float32, device=dev)
    S.spmv_run(plan, x, y)
    torch.cuda.synchronize()
    assert_parity(m, y.cpu().numpy(), TOL32)


@pytest.mark.parametrize("fmt", DELTAS)
def test_delta_gap_patterns(fmt):
    # first column 0; gaps of exactly D, D + 1, 2D and 2D + 1 for each field
    # width (D = 3, 15, 255); a gap across the row
    rows = [[0, 15, 30, 31, 47], [16], [31, 32, 33, 34, 35, 36, 37, 38],
            [0, 3, 7, 13, 20], [3], [4], [0, 255, 511, 1021, 1533], [256], [255],
            [0], [4095], list(range(0, 4096, 17)), list(range(2000, 2050)),
            list(range(0, 4096, 2)), list(range(0, 4096, 4)), list(range(1, 4096, 3))]
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])])
    ci = np.concatenate([np.array(r) for r in rows])
    rng = np.random.default_rng(5)
    vals = rng.normal(0, 0.5, ci.size).astype(np.float16)
    vals[vals == 0] = np.float16(0.25)
    m = make("gaps", rp, ci, vals, 4096, rng.normal(0, 1, 4096).astype(np.float16))
    for kw in ({}, {"x_smem": 0}):
        y, _ = run_gpu(m, fmt, options=S.spmv_plan_options(**kw))
        assert_parity(m, y, TOL16)


@pytest.mark.parametrize("fmt", ["delta4", "delta2"])
@pytest.mark.parametrize("kernel", [1, 2])
def test_delta_decodes(kernel, fmt):
    """2- and 4-bit deltas through both decodes (a lane per word; several
    lanes per word -- 4 for 4-bit, 8 for 2-bit deltas -- with the planner's
    per-word offsets): rows of every length class,
    gaps that need padding, partial segments, rows shared by warps, x in
    shared memory and through L1; repeat runs give the same bits."""
    cases = [workloads.llm(0.3, n=1536, seed=6), workloads.llm(0.6, n=3000, seed=8),
             workloads.llm(0.9, n=2000, seed=2)]
    lengths = np.tile([0, 1, 0, 3, 9, 0, 257, 0, 5000, 2, 20000, 0, 700, 64, 65], 30)
    cases.append(workloads.from_lengths("mixed16", lengths, 30000, seed=17, dtype=np.float16))
    rows = [[0, 15, 30, 31, 47], [16], list(range(0, 4096, 17)), list(range(0, 4096, 2)),
            list(range(1, 4096, 3)), [4095]]
    rp = np.concatenate([[0], np.cumsum([len(r) for r in rows])])
    ci = np.concatenate([np.array(r) for r in rows])
    rng = np.random.default_rng(3)
    vals = rng.normal(0, 0.5, ci.size).astype(np.float16)
    vals[vals == 0] = np.float16(0.25)
    cases.append(make("gaps", rp, ci, vals, 4096, rng.normal(0, 1, 4096).astype(np.float16)))
    for m in cases:
        for xs in (0, 1):
            opts = S.spmv_plan_options(delta_kernel=kernel, x_smem=xs)
            ys, info = run_gpu(m, fmt, options=opts, repeat=2)
            if m.n_cols * 2 <= 32768:   # a larger x does not fit beside the rings
                assert info["x_in_smem"] == xs
            assert np.array_equal(ys[0], ys[1])
            assert_parity(m, ys[0], TOL16)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_plan_from_converted_delta(bits):
    m = workloads.llm(0.75, n=900, seed=4)
    d = S.spmv_convert(m.row_ptr, m.col_idx, m.values, m.n_cols, bits=bits)
    plan = S.spmv_plan_create_delta(d)
    assert plan.info["format"] == FORMAT_CODE[f"delta{bits}"]
    dev = torch.device("cuda", 0)
    y = torch.empty(m.n_rows, dtype=torch.float32, device=dev)
    S.spmv_run(plan, torch.from_numpy(m.x).to(dev), y)
    torch.cuda.synchronize()
    y2, _ = run_gpu(m, f"delta{bits}")
    assert np.array_equal(y.cpu().numpy(), y2)
    assert_parity(m, y2, TOL16)


def test_delta_plan_rejects_bad_columns():
    m = workloads.llm(0.75, n=64, seed=4)
    d = S.spmv_convert(m.row_ptr, m.col_idx, m.values, m.n_cols)
    d.n_cols = int(m.col_idx.max())          # last column now out of range
    with pytest.raises(S.SpmvError) as e:
        S.spmv_plan_create_delta(d)
    assert e.value.status == 3


# ------------------------------------------------------------ runtime behaviour

def test_repeated_runs_identical_and_split_counters_rearm():
    m = workloads.powerlaw(n=20000, nnz=111000, max_len=3000, seed=2)
    ys, info = run_gpu(m, options=S.spmv_plan_options(cta_row_min=200, split_row_min=300,
                                                      split_chunk=100, csr_kernel=1),
                       repeat=4)
    assert info["rows_per_bin"][3] > 0
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])
    assert_parity(m, ys[0], TOL32)


def test_side_stream_and_graph_capture():
    m = small("powerlaw_small")
    dev = torch.device("cuda", 0)
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols)
    x = torch.from_numpy(m.x).to(dev)
    y = torch.zeros(m.n_rows, dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        S.spmv_run(plan, x, y)
    s.synchronize()
    y_stream = y.cpu().numpy().copy()
    g = torch.cuda.CUDAGraph()
    y.zero_()
    with torch.cuda.graph(g):
        S.spmv_run(plan, x, y)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), y_stream)
    assert_parity(m, y_stream, TOL32)
    S.spmv_plan_destroy(plan)


@pytest.mark.parametrize("fmt,name", [("csr", "laplacian_small"), ("delta4", "llm90_small"),
                                      ("delta2", "llm30_small"), ("delta8", "llm90_small")])
def test_run_host_end_to_end(fmt, name):
    m = small(name)
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols, format=fmt)
    xh = torch.from_numpy(m.x).pin_memory().numpy()
    yh = torch.empty(m.n_rows, dtype=torch.float32).pin_memory().numpy()
    S.spmv_run_host(plan, xh, yh)
    assert_parity(m, yh, tol_for(m))
    S.spmv_plan_destroy(plan)


@pytest.mark.parametrize("fmt,name,count", [("csr", "laplacian_small", 5),
                                            ("csr", "powerlaw_small", 2),
                                            ("delta4", "llm90_small", 3),
                                            ("sell", "fem_small", 1), ("csr", "tiny", 0)])
def test_run_host_batch_end_to_end(fmt, name, count):
    """Vectors through the pipelined host-buffer entry point: each y equals
    the oracle's and spmv_run's for its own x (slots reused, two calls in a
    row), and a call over no vectors does nothing."""
    m = small(name)
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols, format=fmt)
    rng = np.random.default_rng(31)
    xs = [m.x] + [rng.uniform(-1, 1, m.n_cols).astype(m.x.dtype) for _ in range(max(count, 1) - 1)]
    xh = torch.from_numpy(np.stack(xs[:count]) if count else
                          np.zeros((0, m.n_cols), m.x.dtype)).pin_memory().numpy()
    dev = torch.device("cuda", 0)
    for _ in range(2):
        yh = torch.full((count, m.n_rows), float("nan"), dtype=torch.float32).pin_memory().numpy()
        S.spmv_run_host_batch(plan, xh, yh)
        for i in range(count):
            y_ref, sm = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, xh[i])
            assert np.all(np.abs(yh[i] - y_ref) <= tol_for(m) * sm + 1e-30)
            yd = torch.empty(m.n_rows, dtype=torch.float32, device=dev)
            S.spmv_run(plan, torch.from_numpy(np.ascontiguousarray(xh[i])).to(dev), yd)
            assert np.array_equal(yd.cpu().numpy(), yh[i])
    with pytest.raises(ValueError):
        S.spmv_run_host_batch(plan, xh.reshape(-1), yh)
    S.spmv_plan_destroy(plan)


def test_argument_errors():
    m = small("tiny")
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols)
    dev = torch.device("cuda", 0)
    x = torch.from_numpy(m.x).to(dev)
    with pytest.raises(TypeError):
        S.spmv_run(plan, x.half(), torch.empty(m.n_rows, device=dev))
    with pytest.raises(ValueError):
        S.spmv_run(plan, x[:-1], torch.empty(m.n_rows, device=dev))
    buf = torch.empty(m.n_rows + m.n_cols, device=dev)
    with pytest.raises(S.SpmvError) as e:         # x and y overlap
        S.spmv_run(plan, buf.data_ptr(), buf.data_ptr() + 8)
    assert e.value.status == 1
    S.spmv_plan_destroy(plan)
    with pytest.raises(ValueError):
        S.spmv_run(plan, x, torch.empty(m.n_rows, device=dev))


@pytest.mark.parametrize("name", ["laplacian_small", "powerlaw_small", "fem_small"])
def test_chained_runs_respect_dependencies(name):
    """y1 = A x, y2 = A y1, y3 = A y2 launched back to back on one stream
    (kernels may start before their predecessor ends and must order their
    reads of x after it): every link matches the oracle applied to the GPU's
    own input. Output buffers start as NaN so an early read would show."""
    m = small(name)
    assert m.n_rows == m.n_cols
    dev = torch.device("cuda", 0)
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols)
    x0 = torch.from_numpy(m.x).to(dev)
    for _ in range(5):
        ys = [torch.full((m.n_rows,), float("nan"), dtype=torch.float32, device=dev)
              for _ in range(3)]
        torch.cuda.synchronize()
        S.spmv_run(plan, x0, ys[0])
        S.spmv_run(plan, ys[0], ys[1])
        S.spmv_run(plan, ys[1], ys[2])
        torch.cuda.synchronize()
        inputs = [m.x] + [y.cpu().numpy() for y in ys[:2]]
        for xin, y in zip(inputs, ys):
            y_ref, s = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, xin)
            assert_parity(m, y.cpu().numpy(), TOL32, y_ref, s)
    S.spmv_plan_destroy(plan)


def test_chained_delta4_after_torch_kernels():
    """DELTA4 runs whose x is produced by a torch kernel right before them."""
    m = small("llm90_small")
    dev = torch.device("cuda", 0)
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols, format="delta4")
    x = torch.from_numpy(m.x).to(dev)
    y1 = torch.full((m.n_rows,), float("nan"), device=dev)
    y2 = torch.full((m.n_rows,), float("nan"), device=dev)
    S.spmv_run(plan, x, y1)
    x2 = (y1 * 0.01).half()          # torch kernels between the two runs
    S.spmv_run(plan, x2, y2)
    torch.cuda.synchronize()
    y_ref, s = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, m.x)
    assert_parity(m, y1.cpu().numpy(), TOL16, y_ref, s)
    y_ref2, s2 = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, x2.cpu().numpy())
    assert_parity(m, y2.cpu().numpy(), TOL16, y_ref2, s2)
    S.spmv_plan_destroy(plan)


@pytest.mark.parametrize("name", ["llm30_small", "llm90_small"])
def test_delta_auto_width(name):
    """format="delta": the width with the fewest stored bytes, reported by
    the plan's format code."""
    m = small(name)
    bits, _ = S.spmv_delta_select_bits(m.row_ptr, m.col_idx, m.values, m.n_cols)
    y, info = run_gpu(m, "delta")
    assert info["format"] == FORMAT_CODE[f"delta{bits}"]
    assert_parity(m, y, TOL16)


# ------------------------------------------------------------ sliced ELL

@pytest.mark.parametrize("sigma", [1, 1024])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_sell(name, sigma):
    m = small(name)
    y, info = run_gpu(m, "sell", options=S.spmv_plan_options(sell_sigma=sigma))
    assert info["format"] == FORMAT_CODE["sell"]
    assert_parity(m, y, tol_for(m))


@pytest.mark.parametrize("name", ["tiny", "laplacian", "fem", "powerlaw", "llm50", "llm90"])
def test_full_size_sell(name):
    m = full(name)
    y, info = run_gpu(m, "sell")
    assert info["n_entries"] >= m.nnz
    assert_parity(m, y, tol_for(m))


@pytest.mark.parametrize("name,band,want", [("laplacian_small", "sell", "csr"),
                                            ("fem_small", "sell", "sell"),
                                            ("powerlaw_small", "csr", "csr")])
def test_auto_format(name, band, want):
    m = small(name)
    fmt, _, _ = S.spmv_select_format(m.row_ptr, m.col_idx, m.values, m.n_cols)
    assert fmt == band
    y, info = run_gpu(m, "auto")
    assert info["format"] == FORMAT_CODE[want]
    assert_parity(m, y, tol_for(m))


def test_sell_edge_cases():
    # rows without nonzeros, a ragged last slice, one long row among empties
    lengths = np.tile([0, 1, 0, 3, 40, 0, 2], 11)          # 77 rows
    m = workloads.from_lengths("ragged_sell", lengths, 300, seed=3)
    for sigma in (1, 5, 1024):
        y, _ = run_gpu(m, "sell", options=S.spmv_plan_options(sell_sigma=sigma))
        assert_parity(m, y, TOL32)
    n = 5000
    z = make("zero_nnz", np.zeros(n + 1), [], np.zeros(0, np.float32), 7, np.ones(7, np.float32))
    y, _ = run_gpu(z, "sell")
    assert np.all(y == 0)
    one = make("1x1", [0, 1], [0], np.array([3.0], np.float32), 1, np.array([2.0], np.float32))
    y, _ = run_gpu(one, "sell")
    assert y[0] == 6.0
    rng = np.random.default_rng(4)
    n = 100_000
    row = make("one_long_row", [0, n], np.arange(n), rng.uniform(-1, 1, n).astype(np.float32),
               n, rng.uniform(-1, 1, n).astype(np.float32))
    y, _ = run_gpu(row, "sell")
    assert_parity(row, y, TOL32)
    empty = make("empty", [0], [], np.zeros(0, np.float32), 5, np.ones(5, np.float32))
    plan = S.spmv_plan_create(empty.row_ptr, empty.col_idx, empty.values, 5, format="sell")
    S.spmv_run(plan, torch.ones(5, device="cuda"), torch.empty(0, device="cuda"))
    torch.cuda.synchronize()
    assert plan.info["launches_per_run"] == 0


def test_sell_unsorted_duplicates_and_rectangular():
    rng = np.random.default_rng(6)
    n_rows, n_cols = 3000, 500
    lengths = rng.integers(0, 40, n_rows)
    rp = np.concatenate([[0], np.cumsum(lengths)])
    ci = rng.integers(0, n_cols, rp[-1])
    vals = rng.uniform(-1, 1, rp[-1]).astype(np.float32)
    m = make("unsorted", rp, ci, vals, n_cols, rng.uniform(-1, 1, n_cols).astype(np.float32))
    y, _ = run_gpu(m, "sell")
    assert_parity(m, y, TOL32)
    wide = workloads.from_lengths("wide", np.full(40, 3000), 100_000, seed=1)
    y, _ = run_gpu(wide, "sell")
    assert_parity(wide, y, TOL32)


@pytest.mark.parametrize("sigma", [1, 1024])
def test_sell_chained_runs_and_graph(sigma):
    """y1 = A x, y2 = A y1, y3 = A y2 back to back on one stream (the kernel
    may start before its predecessor ends), then the same under a CUDA
    graph; every link matches the oracle on the GPU's own input."""
    m = small("laplacian_small")
    dev = torch.device("cuda", 0)
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols, format="sell",
                              options=S.spmv_plan_options(sell_sigma=sigma))
    x0 = torch.from_numpy(m.x).to(dev)
    ys = [torch.full((m.n_rows,), float("nan"), dtype=torch.float32, device=dev)
          for _ in range(3)]
    S.spmv_run(plan, x0, ys[0])
    S.spmv_run(plan, ys[0], ys[1])
    S.spmv_run(plan, ys[1], ys[2])
    torch.cuda.synchronize()
    inputs = [m.x] + [y.cpu().numpy() for y in ys[:2]]
    for xin, y in zip(inputs, ys):
        y_ref, s = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, xin)
        assert_parity(m, y.cpu().numpy(), TOL32, y_ref, s)
    g = torch.cuda.CUDAGraph()
    y = torch.zeros(m.n_rows, dtype=torch.float32, device=dev)
    with torch.cuda.graph(g):
        S.spmv_run(plan, x0, y)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), ys[0].cpu().numpy())
    S.spmv_plan_destroy(plan)


# ------------------------------------------------------------ matrix-free FEM

def run_fem(m, x=None, repeat=1):
    dev = torch.device("cuda", 0)
    plan = S.spmv_plan_create_fem(m.nex, m.ney, m.nez, m.rho, m.K0)
    xt = torch.from_numpy(np.ascontiguousarray(m.x if x is None else x)).to(dev)
    outs = []
    for _ in range(repeat):
        y = torch.full((m.n_dofs,), float("nan"), dtype=torch.float32, device=dev)
        S.spmv_run(plan, xt, y)
        outs.append(y)
    torch.cuda.synchronize()
    S.spmv_plan_check(plan)
    info = plan.info
    S.spmv_plan_destroy(plan)
    ys = [o.cpu().numpy() for o in outs]
    return (ys if repeat > 1 else ys[0]), info


def assert_fem_parity(m, y, x=None):
    from oracle import fem
    y_ref, s = fem.fem_matvec(m.nex, m.ney, m.nez, m.rho, m.K0, m.x if x is None else x)
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y))
    err = np.abs(y - y_ref)
    bad = np.nonzero(err > TOL32 * s + 1e-30)[0]
    assert bad.size == 0, (f"{m.name}: {bad.size} dofs out of tolerance, first {bad[:5]}, "
                           f"max |dy|/s = {np.max(err / np.maximum(s, 1e-300)):.3e}")


@pytest.mark.parametrize("dims", [(1, 1, 1), (2, 1, 1), (1, 1, 3), (4, 3, 2), (13, 7, 5),
                                  (33, 2, 9)])
def test_fem_small(dims):
    m = workloads.fem_simp(*dims, seed=sum(dims))
    y, info = run_fem(m)
    assert info["format"] == 7 and info["n_rows"] == m.n_dofs
    assert info["nnz"] == workloads.fem_nnz(*dims)
    assert_fem_parity(m, y)


def test_fem_full_size_deterministic():
    m = workloads.fem_simp()
    ys, info = run_fem(m, repeat=3)
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])
    assert_fem_parity(m, ys[0])


def test_fem_general_K0_and_single_entries():
    """A non-symmetric K0 (the operator applies K0 as given, rows by
    columns), and K0 with one nonzero entry against the hand rule."""
    m = workloads.fem_simp(3, 2, 2, seed=4)
    k0 = np.random.default_rng(8).normal(size=(24, 24)).astype(np.float32)
    m2 = workloads.FemMesh("fem_nonsym", 3, 2, 2, m.rho, k0, m.x)
    y, _ = run_fem(m2)
    assert_fem_parity(m2, y)
    from oracle import fem
    edof = fem.element_dofs(1, 1, 1)[0]
    x = (np.arange(24, dtype=np.float32) + 1) * 0.25
    for a, b in ((0, 0), (2, 17), (23, 5)):
        k1 = np.zeros((24, 24), np.float32)
        k1[a, b] = 1.0
        one = workloads.FemMesh("one_entry", 1, 1, 1, np.array([2.0], np.float32), k1, x)
        y, _ = run_fem(one)
        want = np.zeros(24, np.float32)
        want[edof[a]] = 2.0 * x[edof[b]]
        assert np.array_equal(y, want)


def test_fem_matches_assembled_csr_on_gpu():
    """The same K x through the matrix-free operator and through the
    assembled matrix (fp32 CSR from the oracle's assembly) agree within both
    kernels' tolerances."""
    from oracle import fem
    m = workloads.fem_simp(20, 10, 6, seed=2)
    rp, ci, v = fem.fem_assemble(m.nex, m.ney, m.nez, m.rho, m.K0)
    csr = workloads.CSRInput("fem_assembled", m.n_dofs, m.n_dofs, rp.astype(np.int32),
                             ci.astype(np.int32), v.astype(np.float32), m.x, {})
    y_mf, _ = run_fem(m)
    y_csr, _ = run_gpu(csr, "csr")
    y_ref, s = fem.fem_matvec(m.nex, m.ney, m.nez, m.rho, m.K0, m.x)
    assert np.all(np.abs(y_mf.astype(np.float64) - y_csr) <= 3e-5 * s + 1e-30)


def test_fem_chained_runs_and_graph():
    m = workloads.fem_simp(10, 8, 6, seed=3)
    dev = torch.device("cuda", 0)
    plan = S.spmv_plan_create_fem(m.nex, m.ney, m.nez, m.rho, m.K0)
    x0 = torch.from_numpy(m.x).to(dev)
    ys = [torch.full((m.n_dofs,), float("nan"), dtype=torch.float32, device=dev)
          for _ in range(3)]
    S.spmv_run(plan, x0, ys[0])
    S.spmv_run(plan, ys[0], ys[1])
    S.spmv_run(plan, ys[1], ys[2])
    torch.cuda.synchronize()
    inputs = [m.x] + [y.cpu().numpy() for y in ys[:2]]
    for xin, y in zip(inputs, ys):
        assert_fem_parity(m, y.cpu().numpy(), x=xin)
    g = torch.cuda.CUDAGraph()
    y = torch.zeros(m.n_dofs, dtype=torch.float32, device=dev)
    with torch.cuda.graph(g):
        S.spmv_run(plan, x0, y)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), ys[0].cpu().numpy())
    xh = torch.from_numpy(m.x).pin_memory().numpy()
    yh = torch.empty(m.n_dofs, dtype=torch.float32).pin_memory().numpy()
    S.spmv_run_host(plan, xh, yh)
    assert np.array_equal(yh, ys[0].cpu().numpy())
    S.spmv_plan_destroy(plan)


# ------------------------------------------------------------ Jacobi-PCG

def _pcg_gpu(plan, b, tol, max_iter, diag=None, check_every=16):
    dev = torch.device("cuda", 0)
    bt = torch.from_numpy(np.ascontiguousarray(b, dtype=np.float32)).to(dev)
    xt = torch.zeros(b.size, dtype=torch.float32, device=dev)
    dt = None if diag is None else torch.from_numpy(np.ascontiguousarray(diag, np.float32)).to(dev)
    res = S.spmv_pcg_solve(plan, bt, xt, rel_tol=tol, max_iter=max_iter,
                           check_every=check_every, diag=dt)
    return xt.cpu().numpy(), res


def _check_pcg(matvec, diag, b, x_gpu, res, tol, max_iter):
    from oracle import pcg
    x_ref, it_ref, st_ref, hist = pcg.jacobi_pcg(matvec, diag, b, np.zeros(b.size), tol, max_iter)
    assert st_ref == 1 and res["status"] == "converged"
    # fp32 vectors against the fp64 recurrence: the step count may differ a
    # little near the threshold
    assert abs(res["iterations"] - it_ref) <= max(3, it_ref // 20), (res, it_ref)
    bn = np.linalg.norm(b)
    true_res = np.linalg.norm(b - matvec(x_gpu.astype(np.float64))) / bn
    assert true_res <= 5 * tol, true_res
    assert np.linalg.norm(x_gpu - x_ref) <= 1e-3 * np.linalg.norm(x_ref)


@pytest.mark.parametrize("fmt", ["csr", "sell"])
def test_pcg_laplacian(fmt):
    m = workloads.laplacian(120, 90)
    A = sp.csr_matrix((m.values.astype(np.float64), m.col_idx, m.row_ptr),
                      shape=(m.n_rows, m.n_cols))
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols, format=fmt)
    b = m.x.astype(np.float64)
    x, res = _pcg_gpu(plan, b, 1e-5, 2000)
    _check_pcg(lambda v: A @ v, A.diagonal(), b, x, res, 1e-5, 2000)
    # same bits on a second solve, and with the diagonal passed explicitly
    x2, res2 = _pcg_gpu(plan, b, 1e-5, 2000, diag=A.diagonal(), check_every=7)
    assert np.array_equal(x, x2) and res == res2
    S.spmv_plan_destroy(plan)


def test_pcg_fem_matrix_free_and_assembled():
    from oracle import fem
    m = workloads.fem_simp(12, 8, 6, seed=7)
    plan = S.spmv_plan_create_fem(m.nex, m.ney, m.nez, m.rho, m.K0)
    rp, ci, v = fem.fem_assemble(m.nex, m.ney, m.nez, m.rho, m.K0)
    A = sp.csr_matrix((v, ci, rp), shape=(m.n_dofs, m.n_dofs))
    b = m.x.astype(np.float64)
    x, res = _pcg_gpu(plan, b, 1e-6, 3000)
    _check_pcg(lambda u: fem.fem_matvec(m.nex, m.ney, m.nez, m.rho, m.K0, u, with_abs=False),
               A.diagonal(), b, x, res, 1e-6, 3000)
    x2, res2 = _pcg_gpu(plan, b, 1e-6, 3000, diag=A.diagonal())
    assert np.array_equal(x, x2)
    S.spmv_plan_destroy(plan)
    # the same system through the assembled fp32 matrix
    csr = S.spmv_plan_create(rp.astype(np.int32), ci.astype(np.int32), v.astype(np.float32),
                             m.n_dofs, format="sell")
    x3, res3 = _pcg_gpu(csr, b, 1e-6, 3000)
    _check_pcg(lambda u: A @ u, A.diagonal(), b, x3, res3, 1e-6, 3000)
    S.spmv_plan_destroy(csr)


def test_pcg_limits_and_breakdown():
    m = workloads.laplacian(60, 40)
    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols)
    x, res = _pcg_gpu(plan, m.x.astype(np.float64), 1e-12, 5)
    assert res["status"] == "iteration limit" and res["iterations"] == 5
    S.spmv_plan_destroy(plan)
    # indefinite: diag(1, -1, 1, -1, ...) gives p . A p = 0 on the first step
    n = 64
    rp = np.arange(n + 1, dtype=np.int32)
    ci = np.arange(n, dtype=np.int32)
    vals = np.where(np.arange(n) % 2 == 0, 1.0, -1.0).astype(np.float32)
    plan = S.spmv_plan_create(rp, ci, vals, n)
    x, res = _pcg_gpu(plan, np.ones(n), 1e-6, 10)
    assert res["status"] == "breakdown"
    S.spmv_plan_destroy(plan)
    # fp16 plans are refused
    llm = workloads.llm(0.9, n=256)
    plan = S.spmv_plan_create(llm.row_ptr, llm.col_idx, llm.values, llm.n_cols)
    with pytest.raises(S.SpmvError):
        _pcg_gpu(plan, np.ones(256), 1e-6, 10)
    S.spmv_plan_destroy(plan)
