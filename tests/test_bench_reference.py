"""CPU tests of bench.py's reference arm (the oracle, timed on the host): it
prints one JSON line with the contract's keys for the default workload, the
matrix-free operator and the CG workloads, and its byte counts follow the
format definitions."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402

KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e"}


def run_reference(workload, steps=1, warmup=0):
    out = io.StringIO()
    with redirect_stdout(out):
        rc = bench.main(["--impl", "reference", "--workload", workload,
                         "--steps", str(steps), "--warmup", str(warmup)])
    assert rc == 0
    lines = [ln for ln in out.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["tiny", "fem_matfree", "fem_pcg_matfree"])
def test_reference_line_has_the_contract_keys(workload):
    d = run_reference(workload)
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_oracle_call_bytes_follow_the_formats():
    m = workloads.tiny()
    rows, nbytes, nnz, _ = bench.oracle_call(m, "csr", 1.0)
    assert nbytes == 8 * 5000 + 4 * 1001 + 4 * 1000 + 4 * 1000
    rows, nbytes, nnz, _ = bench.oracle_call(m, "sell", 1.0)
    # 1000 rows of exactly 5: 32 slices (the last with 8 rows), each 5 wide
    assert nbytes == 32 * 32 * 5 * 8 + 33 * 4 + 4 * 1000 + 4 * 1000
    f = bench.load_workload("fem_simp", "fem")
    assert (f.n_rows, f.nnz) == (686_433, workloads.fem_nnz(120, 60, 30))
    rows, nbytes, nnz, _ = bench.oracle_call(f, "fem", 1.0)
    assert nbytes == 216_000 * 4 + 24 * 24 * 4 + 2 * 686_433 * 4
    small = workloads.fem_simp(4, 3, 2)
    small.n_rows = small.n_cols = small.n_dofs
    small.nnz = workloads.fem_nnz(4, 3, 2)
    rows, nbytes, nnz, call = bench.oracle_call(small, "pcg_fem", 1.0)
    assert nbytes == 3 * (bench.fem_bytes(small) + bench.PCG_VECTOR_BYTES * small.n_dofs)
    x, it, status, hist = call()
    assert it == 3 and status == 2 and hist[-1] < hist[0]
