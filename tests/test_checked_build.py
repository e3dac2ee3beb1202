"""The checked build of the library (SPMV_CHECKED=1, include/spmv.h:
spmv_checked_build): its CSR kernels and the allocation-free entry point test
every column index and row offset before use, replace one that is out of
range by a safe one and report it through a status word, with no trap.

On the CPU: the build reports itself, and the two check rules (a column
outside [0, n) becomes column 0; an offset outside [lo, hi] is clamped) are
compiled from the library's own header into a host program and exercised.
On the GPU the checked build runs only valid inputs (the five workloads'
small cases through CTA tiles, warp segments, mixed segments and the
allocation-free entry point): the status words stay clear and y matches the
fp64 oracle at the usual tolerances.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads

S = pytest.importorskip("sparse_matrix_vector_gb300")
from sparse_matrix_vector_gb300 import _lib, api  # noqa: E402
from sparse_matrix_vector_gb300.build import INCLUDE, nvcc_path  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_matrix_vector_gb300", "csrc")

CHECK_RULES = r"""
#include <cstdio>
#include "spmv_internal.h"
int main() {
  using namespace spmv;
  int fails = 0;
  bool bad = false;
  fails += checked_col(5, 10, &bad) != 5 || bad;
  fails += checked_col(0, 10, &bad) != 0 || bad;
  fails += checked_col(9, 10, &bad) != 9 || bad;
  bad = false; fails += checked_col(10, 10, &bad) != 0 || !bad;
  bad = false; fails += checked_col(-1, 10, &bad) != 0 || !bad;
  bad = false; fails += checked_col(0, 0, &bad) != 0 || !bad;
  bad = false; fails += checked_offset(7, 3, 9, &bad) != 7 || bad;
  fails += checked_offset(3, 3, 9, &bad) != 3 || bad;
  fails += checked_offset(9, 3, 9, &bad) != 9 || bad;
  bad = false; fails += checked_offset(2, 3, 9, &bad) != 3 || !bad;
  bad = false; fails += checked_offset(10, 3, 9, &bad) != 9 || !bad;
  std::printf("fails=%d\n", fails);
  return fails == 0 ? 0 : 1;
}
"""


def test_check_rules_on_the_host(tmp_path):
    src = tmp_path / "rules.cu"
    src.write_text(CHECK_RULES)
    exe = tmp_path / "rules"
    subprocess.run([nvcc_path(), "-std=c++17", "-I", INCLUDE, "-I", CSRC, "-o", str(exe),
                    str(src)], check=True, capture_output=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr


def test_builds_report_themselves(spmv_lib):
    assert spmv_lib.spmv_checked_build() == 0
    assert spmv_lib.spmv_noalloc_check() == 0      # ordinary builds: OK at once
    checked = _lib.load_checked()
    assert checked.spmv_checked_build() == 1


def _small_cases():
    yield workloads.tiny()
    yield workloads.laplacian(300, 211)
    yield workloads.powerlaw(n=50000, nnz=278500, max_len=4334)
    yield workloads.fem(12, 9, 7)
    yield workloads.llm(0.7, n=1536)


@pytest.mark.gpu
@pytest.mark.parametrize("m", list(_small_cases()), ids=lambda m: m.name)
def test_checked_build_on_valid_inputs(m):
    torch = pytest.importorskip("torch")
    lib = _lib.load_checked()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    y_ref, s = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, m.x)
    tol = 1e-5 if m.values.dtype == np.float32 else 2e-3
    bound = tol * s + 1e-30
    x = torch.from_numpy(m.x).to(dev)
    h = api._host_csr(m.row_ptr, m.col_idx, m.values, m.n_cols)
    for kernel in (1, 2, 3):                   # CTA tiles, warp segments, mixed segments
        opts = S.spmv_plan_options(csr_kernel=kernel)
        plan = ctypes.c_void_p()
        assert lib.spmv_plan_create_ex(ctypes.byref(h.struct), 0, ctypes.byref(opts),
                                       ctypes.byref(plan)) == 0
        y = torch.full((m.n_rows,), float("nan"), dtype=torch.float32, device=dev)
        assert lib.spmv_run(plan, x.data_ptr(), y.data_ptr(),
                            ctypes.c_void_p(stream.cuda_stream)) == 0
        assert lib.spmv_plan_check(plan) == 0   # no index was out of range
        lib.spmv_plan_destroy(plan)
        yv = y.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(yv - y_ref) <= bound), f"kernel {kernel}"
    # the allocation-free entry point
    d_rp = torch.from_numpy(m.row_ptr).to(dev)
    d_ci = torch.from_numpy(m.col_idx).to(dev)
    d_v = torch.from_numpy(m.values).to(dev)
    y = torch.full((m.n_rows,), float("nan"), dtype=torch.float32, device=dev)
    code = S.SPMV_F32 if m.values.dtype == np.float32 else S.SPMV_F16
    assert lib.spmv_csr_run_noalloc(m.n_rows, m.n_cols, m.nnz, d_rp.data_ptr(), d_ci.data_ptr(),
                                    d_v.data_ptr(), code, x.data_ptr(), y.data_ptr(),
                                    ctypes.c_void_p(stream.cuda_stream)) == 0
    assert lib.spmv_noalloc_check() == 0
    yv = y.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(yv - y_ref) <= bound)


@pytest.mark.gpu
def test_checked_build_reports_bad_columns_through_the_status_word():
    """The checked build on a caller-owned CSR matrix with two column
    indices out of range (one past n_cols, one negative): its own bounds
    checks substitute column 0 before any access, so nothing faults; the
    status word reports the error once (the check clears it); the rows
    without a bad column are right. Only the checked build is given this
    input: the ordinary build trusts the caller's device arrays."""
    torch = pytest.importorskip("torch")
    lib = _lib.load_checked()
    assert lib.spmv_checked_build() == 1
    m = workloads.powerlaw(n=5000, nnz=27800, max_len=400, seed=9)
    ci = m.col_idx.copy()
    bad_at = [int(m.row_ptr[10]), int(m.row_ptr[2000])]
    ci[bad_at[0]] = m.n_cols + 7
    ci[bad_at[1]] = -3
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    d_rp = torch.from_numpy(m.row_ptr).to(dev)
    d_ci = torch.from_numpy(ci).to(dev)
    d_v = torch.from_numpy(m.values).to(dev)
    x = torch.from_numpy(m.x).to(dev)
    y = torch.full((m.n_rows,), float("nan"), dtype=torch.float32, device=dev)
    assert lib.spmv_noalloc_check() == 0                 # nothing pending
    assert lib.spmv_csr_run_noalloc(m.n_rows, m.n_cols, m.nnz, d_rp.data_ptr(),
                                    d_ci.data_ptr(), d_v.data_ptr(), S.SPMV_F32,
                                    x.data_ptr(), y.data_ptr(),
                                    ctypes.c_void_p(stream.cuda_stream)) == 0
    assert lib.spmv_noalloc_check() == 10                # SPMV_ERR_DEVICE_STATUS
    assert lib.spmv_noalloc_check() == 0                 # cleared by the check
    yv = y.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(yv))
    y_ref, s = oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, m.x)
    rows = np.searchsorted(m.row_ptr, bad_at, side="right") - 1
    good = np.ones(m.n_rows, bool)
    good[rows] = False
    assert np.all(np.abs(yv - y_ref)[good] <= 1e-5 * s[good] + 1e-30)
