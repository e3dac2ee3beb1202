"""The allocation-free entry point spmv_csr_run_noalloc, called through the C
ABI, against the fp64 oracle's y and against the plan-based entry point
(spmv_plan_create + spmv_run); two of the cases also go through the public
Python wrapper.

spmv_csr_run_noalloc exists for callers that may not allocate device memory
(for example a latency-critical loop after its set-up phase, a component
inside a memory pool that owns all device memory, or a plug-in handed device
buffers but no allocator); its scratch lives in a fixed device array inside
the library. Each case calls it twice in a row: the second call must see the
first call's leftovers in that shared array and still be right.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
S = pytest.importorskip("sparse_matrix_vector_gb300")

pytestmark = pytest.mark.gpu

TOL = {np.dtype(np.float32): 1e-5, np.dtype(np.float16): 2e-3}
# cases that also run through sparse_matrix_vector_gb300.spmv_csr_run_noalloc
WRAPPER_CASES = ("llm70", "fem")


def cases():
    rng = np.random.default_rng(17)
    # one very long row (crosses many 2048-nonzero slices), empty rows at the
    # start, middle and end, a row ending exactly on a slice boundary, and a
    # nonzero count that is not a multiple of 4
    lengths = np.concatenate([[0, 0, 3], [300_001], [0] * 5, [2048 - 4],
                              rng.integers(0, 9, 5000), [4096], [0] * 7])
    yield workloads.from_lengths("long_rows", lengths, 400_000, seed=3)
    yield workloads.powerlaw(n=60000, nnz=334000, max_len=4334, seed=7)
    yield workloads.fem(10, 8, 6)
    yield workloads.llm(0.7, n=1500, seed=2)
    yield workloads.from_lengths("no_nonzeros", np.zeros(300, np.int64), 10, seed=1)


def call_noalloc(lib, m, d_rp, d_ci, d_v, d_x, d_y, stream):
    code = S.SPMV_F32 if m.values.dtype == np.float32 else S.SPMV_F16
    st = lib.spmv_csr_run_noalloc(m.n_rows, m.n_cols, m.nnz, d_rp.data_ptr(),
                                  d_ci.data_ptr(), d_v.data_ptr(), code,
                                  d_x.data_ptr(), d_y.data_ptr(),
                                  ctypes.c_void_p(stream.cuda_stream))
    assert st == 0, S.spmv_status_string(st)


@pytest.mark.parametrize("m", list(cases()), ids=lambda m: m.name)
def test_noalloc_matches_plan_entry_point(spmv_lib, m):
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    d_rp = torch.from_numpy(m.row_ptr).to(dev)
    d_ci = torch.from_numpy(m.col_idx).to(dev)
    d_v = torch.from_numpy(m.values).to(dev)
    d_x = torch.from_numpy(m.x).to(dev)

    plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols)
    y_plan = torch.empty(m.n_rows, dtype=torch.float32, device=dev)
    S.spmv_run(plan, d_x, y_plan)
    torch.cuda.synchronize()
    y_plan = y_plan.cpu().numpy().astype(np.float64)
    S.spmv_plan_destroy(plan)

    y_ref, s = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, m.x)
    bound = TOL[m.values.dtype] * s + 1e-30
    outs = []
    for _ in range(2):                      # two calls in a row
        y = torch.full((m.n_rows,), float("nan"), dtype=torch.float32, device=dev)
        call_noalloc(spmv_lib, m, d_rp, d_ci, d_v, d_x, y, stream)
        torch.cuda.synchronize()
        outs.append(y.cpu().numpy().astype(np.float64))
    if m.name in WRAPPER_CASES:             # the public wrapper, twice more
        for _ in range(2):
            y = torch.full((m.n_rows,), float("nan"), dtype=torch.float32, device=dev)
            S.spmv_csr_run_noalloc(m.n_rows, m.n_cols, d_rp, d_ci, d_v, d_x, y)
            torch.cuda.synchronize()
            outs.append(y.cpu().numpy().astype(np.float64))
    for y in outs:
        assert np.all(np.isfinite(y))
        assert np.all(np.abs(y - y_ref) <= bound), \
            f"max |dy|/s = {np.max(np.abs(y - y_ref) / np.maximum(s, 1e-300)):.3e} (oracle)"
        assert np.all(np.abs(y - y_plan) <= bound), \
            f"max |dy|/s = {np.max(np.abs(y - y_plan) / np.maximum(s, 1e-300)):.3e} (plan)"
    for y in outs[1:]:
        assert np.array_equal(outs[0], y)


def test_noalloc_rejects_bad_arguments(spmv_lib):
    dev = torch.device("cuda", 0)
    big = (1 << 27) + 1                      # one past the scratch limit
    y = torch.empty(4, dtype=torch.float32, device=dev)
    rp = torch.zeros(5, dtype=torch.int32, device=dev)
    st = spmv_lib.spmv_csr_run_noalloc(4, 4, big, rp.data_ptr(), rp.data_ptr(),
                                       rp.data_ptr(), S.SPMV_F32, rp.data_ptr(),
                                       y.data_ptr(), None)
    assert st == 8                           # SPMV_ERR_TOO_LARGE
    st = spmv_lib.spmv_csr_run_noalloc(4, 4, 4, rp.data_ptr(), rp.data_ptr() + 4,
                                       rp.data_ptr(), S.SPMV_F32, rp.data_ptr(),
                                       y.data_ptr(), None)
    assert st == 1                           # misaligned col_idx
    st = spmv_lib.spmv_csr_run_noalloc(-1, 4, 0, None, None, None, S.SPMV_F32,
                                       None, None, None)
    assert st == 1
    # y in host memory: refused on the host, before any launch
    y_host = np.zeros(4, np.float32)
    st = spmv_lib.spmv_csr_run_noalloc(4, 4, 0, rp.data_ptr(), None, None, S.SPMV_F32,
                                       None, y_host.ctypes.data, None)
    assert st == 1
