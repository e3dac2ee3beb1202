#!/usr/bin/env python3
"""Benchmark of y = A x on GB300 through the C ABI (include/spmv.h).

One step = one spmv_run (the whole path: the CSR tile kernel, the sliced-ELL
kernel or the DELTA decode kernel) over one resident copy of the workload.
Copies rotate so that the footprint
of the timed loop is several times the L2 size: every step streams its matrix
from HBM. Steps are captured into CUDA graphs and replayed; the timed region
is bracketed by a barrier and torch.cuda.synchronize() and measured with CUDA
events on the launching stream.

Metric (effective bandwidth): bytes = values + indices + row pointers (as
stored by the format, padding included) + x read once + y written, divided by
the time per step; GFLOP/s = 2 * nnz / time.

  python bench.py                       # default workload: 5-point Laplacian
  python bench.py --workload llm50_delta4
  python bench.py --workload all        # one JSON line per workload
  python bench.py --impl reference      # the fp64 CPU oracle on the same config
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = ("SpMV effective GB/s (fraction of GB300 HBM peak) and GFLOP/s "
          "per matrix")
FALLBACK_HBM_GBS = 6800.0

# workload name -> (generator key, format, description)
WORKLOADS = {
    "tiny": ("tiny", "csr", "tiny_1000x1000_5perrow_f32_csr"),
    "laplacian": ("laplacian", "csr", "laplacian_5pt_1000x999_f32_csr"),
    "powerlaw": ("powerlaw", "csr", "powerlaw_zipf2_916428_5105039nnz_f32_csr"),
    "fem": ("fem", "csr", "fem_hex_120x60x30_3dof_f32_csr"),
    "laplacian_sell": ("laplacian", "sell", "laplacian_5pt_1000x999_f32_sell32"),
    "fem_sell": ("fem", "sell", "fem_hex_120x60x30_3dof_f32_sell32"),
    "fem_matfree": ("fem_simp", "fem", "fem_hex_120x60x30_3dof_f32_matrix_free"),
    "fem_pcg_sell": ("fem", "pcg_sell", "fem_hex_120x60x30_3dof_f32_jacobi_pcg_sell32"),
    "fem_pcg_matfree": ("fem_simp", "pcg_fem", "fem_hex_120x60x30_3dof_f32_jacobi_pcg_matrix_free"),
}
# bytes of vector traffic per conjugate-gradient iteration and unknown, next
# to the matrix product's: step length reads p, q (8); the update reads x,
# p, r, q, diag and writes x, r, z (32); the direction reads z, p and writes
# p (12)
PCG_VECTOR_BYTES = 52
# iterations per pass of the solve's device-side loop (the library's default)
PCG_BODY = 2
PCG_TOL = 1e-6
# fp32 fma peak for the matrix-free operator's ALU roofline: 152 SMs x 128
# fp32 lanes x 2 flops at the 2070 MHz maximum SM clock
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12
# flops of the matrix-free operator per element: K0 (24 x 24) times 24
# values, then 24 products with the density
FEM_FLOPS_PER_ELEMENT = 2 * 24 * 24 + 24
for _s in (30, 50, 70, 90):
    WORKLOADS[f"llm{_s}_csr"] = (f"llm{_s}", "csr",
                                 f"llm_12288x12288_sparsity{_s}_f16_csr")
    for _b in (2, 4, 8):
        WORKLOADS[f"llm{_s}_delta{_b}"] = (f"llm{_s}", f"delta{_b}",
                                           f"llm_12288x12288_sparsity{_s}_f16_delta{_b}")
# long rows are the wrong shape for a lane per row; one such line is kept
# as the measured counter-example (the AUTO format never picks it)
WORKLOADS["llm50_sell"] = ("llm50", "sell", "llm_12288x12288_sparsity50_f16_sell32")
DEFAULT_WORKLOAD = "laplacian"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_file(fmt: str, segments: bool = False) -> str:
    """The source file of the kernel a format's plan runs."""
    if fmt.startswith("delta"):
        return "spmv_delta.cu"
    if fmt == "sell":
        return "spmv_sell.cu"
    if fmt == "fem":
        return "spmv_fem.cu"
    return "spmv_csr_seg.cu" if segments else "spmv_csr.cu"


def kernel_source_sha(fmt: str, segments: bool = False) -> str:
    """sha256[:16] of the device sources of a plan's kernel (the shared
    device header and internal header, then the kernel's file)."""
    csrc = os.path.join(ROOT, "sparse_matrix_vector_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("spmv_device.cuh", "spmv_internal.h", kernel_file(fmt, segments)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, fmt: str, segments: bool = False):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None
    if not rec or rec.get("kernel_sha") != kernel_source_sha(fmt, segments):
        return None
    return int(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (read only)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception as e:  # nvidia-smi missing: report no clocks
            log("clock sampling unavailable:", e)
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(ms: float, device, pg) -> float:
    """The slowest rank's timed-region length (ms); every rank gets it."""
    if pg is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX, group=pg)
    torch.distributed.barrier(group=pg)
    return float(t.item())


def job_throughput(nbytes: int, world: int, ms: float, steps: int):
    """Seconds per step, whole-job GB/s (every rank ran `steps` runs of
    `nbytes` in `ms`) and one launch's GB/s."""
    sec_per_step = ms / 1e3 / steps
    return sec_per_step, world * nbytes / sec_per_step / 1e9, nbytes / sec_per_step / 1e9


# A timed region is K back-to-back steps. Regions repeat until about
# REGION_SECONDS of device time has been timed (at least MIN_REGIONS), and the
# line reports their median (min and max beside it).
REGION_SECONDS = 0.6
MIN_REGIONS = 5
MAX_REGIONS = 5000
# clock cycles of torch's bounded spin kernel queued ahead of every region:
# the host submits the region's graph replays while it runs, so the region's
# first event is followed at once by the first SpMV kernel rather than by the
# replay's submission
LEAD_CYCLES = 300_000


def timed_regions(run_region, stream, dev, pg, local, steps, est_step_s, regions=0):
    """Time `steps` steps (one call of run_region, which enqueues them on
    `stream`) several times over. Each
    region is bracketed by a barrier and torch.cuda.synchronize() on both
    sides and timed with CUDA events on the launching stream. Returns the
    per-region statistics in ms (max over ranks of each) and the clock record
    sampled across all regions."""
    import torch
    n = regions or int(min(MAX_REGIONS, max(MIN_REGIONS, math.ceil(
        REGION_SECONDS / max(steps * est_step_s, 1e-7)))))
    clocks = ClockSampler(local)
    clocks.start()
    times = []
    for _ in range(n):
        if pg is not None:
            torch.distributed.barrier(group=pg)
        torch.cuda.synchronize(dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(LEAD_CYCLES)
            ev0.record(stream)
            run_region()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(ev0.elapsed_time(ev1))
    clk = clocks.stop()
    stats = [statistics.median(times), min(times), max(times), times[0]]
    stats = [max_over_ranks(t, dev, pg) for t in stats]
    return {"regions": n, "median_ms": stats[0], "min_ms": stats[1],
            "max_ms": stats[2], "first_ms": stats[3]}, clk


def region_report(regions, steps):
    """config.timing's statistics, per step."""
    return {"regions": regions["regions"], "steps_per_region": steps,
            "median_ms_per_step": regions["median_ms"] / steps,
            "min_ms_per_step": regions["min_ms"] / steps,
            "max_ms_per_step": regions["max_ms"] / steps,
            "first_region_ms_per_step": regions["first_ms"] / steps}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_workload(key, fmt):
    import workloads
    if fmt == "fem":
        m = workloads.fem_simp()
        # the attributes the benchmark reads from a matrix workload
        m.n_rows = m.n_cols = m.n_dofs
        m.nnz = workloads.fem_nnz(m.nex, m.ney, m.nez)
        m.values = m.rho
        return m
    return workloads.make(key)


def fem_bytes(m):
    return m.n_elem * 4 + 24 * 24 * 4 + 2 * m.n_dofs * 4


def oracle_call(m, fmt, frac):
    """The oracle as it stands on the first ceil(frac * n_rows) rows of the
    workload: returns (rows, algorithmic bytes, nonzeros, zero-arg call)."""
    import oracle
    if fmt.startswith("pcg"):   # a few Jacobi-PCG iterations on the whole system
        from oracle import pcg, fem
        k = 3
        if fmt == "pcg_fem":
            matvec = (lambda u: fem.fem_matvec(m.nex, m.ney, m.nez, m.rho, m.K0, u,
                                               with_abs=False))
            diag = fem.fem_diagonal(m.nex, m.ney, m.nez, m.rho, m.K0)
            per_iter = fem_bytes(m)
        else:
            rows = np.repeat(np.arange(m.n_rows), np.diff(m.row_ptr))
            diag = np.zeros(m.n_rows)
            on = m.col_idx == rows
            np.add.at(diag, rows[on], m.values[on].astype(np.float64))
            matvec = (lambda u: oracle.csr_spmv(m.row_ptr, m.col_idx, m.values, u,
                                                with_abs=False))
            per_iter = algorithmic_bytes_csr(m)
        nbytes = k * (per_iter + PCG_VECTOR_BYTES * m.n_rows)
        b = m.x.astype(np.float64)
        return m.n_rows, nbytes, m.nnz, (lambda: pcg.jacobi_pcg(
            matvec, diag, b, np.zeros(m.n_rows), 0.0, k))
    if fmt == "fem":   # one call on the whole mesh (well under a second)
        from oracle import fem
        return m.n_rows, fem_bytes(m), m.nnz, (lambda: fem.fem_matvec(
            m.nex, m.ney, m.nez, m.rho, m.K0, m.x, with_abs=False))
    rows = max(1, min(m.n_rows, int(math.ceil(m.n_rows * frac))))
    rp = m.row_ptr[:rows + 1]
    ci, vals = m.col_idx[:rp[-1]], m.values[:rp[-1]]
    if fmt.startswith("delta"):
        bits = int(fmt[5:])
        enc = oracle.delta_encode(m.n_cols, rp, ci, vals, bits=bits)
        nbytes = (enc.n_entries * 2 + enc.n_entries * bits // 8 + (rows + 1) * 4
                  + m.n_cols * 2 + rows * 4)
        return rows, nbytes, int(rp[-1]), (lambda: oracle.delta_spmv(enc, m.x))
    if fmt == "sell":
        # y = A x is the CSR definition; the bytes are those the sliced
        # layout of these rows stores (rows in order)
        from oracle import sell
        slots, slices = sell.sell_slot_count(rp, 32, 1)
        nbytes = (slots * (vals.dtype.itemsize + 4) + (slices + 1) * 4
                  + m.n_cols * m.x.dtype.itemsize + rows * 4)
        return rows, nbytes, int(rp[-1]), (lambda: oracle.csr_spmv(rp, ci, vals, m.x))
    nbytes = (int(rp[-1]) * (vals.dtype.itemsize + 4) + (rows + 1) * 4
              + m.n_cols * m.x.dtype.itemsize + rows * 4)
    return rows, nbytes, int(rp[-1]), (lambda: oracle.csr_spmv(rp, ci, vals, m.x))


def oracle_baseline(m, fmt, budget_s: float):
    """cpu_baseline: time the oracle (fp64, one CPU thread) as it stands on a
    bounded sample: whole-matrix calls repeated for about budget_s (at least
    two), or one call on a leading block of rows if a whole call is too slow.
    Returns (GB/s, sample description)."""
    rows, nbytes, nnz, call = oracle_call(m, fmt, 1.0)
    t0 = time.perf_counter()
    call()
    t_full = time.perf_counter() - t0
    if t_full * 2 > budget_s:
        rows, nbytes, nnz, call = oracle_call(m, fmt, budget_s / 2 / t_full)
        t0 = time.perf_counter()
        call()
        dt = time.perf_counter() - t0
        return nbytes / dt / 1e9, f"rows 0..{rows - 1} of {m.n_rows}, 1 call"
    reps = max(2, int(budget_s / max(t_full, 1e-6)))
    t0 = time.perf_counter()
    for _ in range(reps):
        call()
    dt = (time.perf_counter() - t0) / reps
    return nbytes / dt / 1e9, f"whole matrix, {reps} calls"


def parallel_baseline(m, fmt, budget_s: float):
    """The all-core CPU baseline: the oracle's loop with its rows shared out
    over OpenMP threads (oracle/parallel.py), on the whole matrix, repeated
    for about budget_s. Same byte model as the GPU line. None for the
    matrix-free operator and the solver, or when it could not be built."""
    if fmt == "fem" or fmt.startswith("pcg"):
        return None
    try:
        import oracle
        from oracle import parallel
        n_threads = parallel.threads()
    except Exception as e:  # noqa: BLE001
        return {"unavailable": f"OpenMP baseline not built: {e}"}
    if fmt.startswith("delta"):
        bits = int(fmt[5:])
        enc = oracle.delta_encode(m.n_cols, m.row_ptr, m.col_idx, m.values, bits=bits)
        call = parallel.DeltaOperands(enc, m.x)
        nbytes = (enc.n_entries * 2 + enc.n_entries * bits // 8 + (m.n_rows + 1) * 4
                  + m.n_cols * 2 + m.n_rows * 4)
    else:
        call = parallel.CsrOperands(m.row_ptr, m.col_idx, m.values, m.x)
        if fmt == "sell":
            from oracle import sell
            slots, slices = sell.sell_slot_count(m.row_ptr, 32, 1)
            nbytes = (slots * (m.values.dtype.itemsize + 4) + (slices + 1) * 4
                      + m.n_cols * m.x.dtype.itemsize + m.n_rows * 4)
        else:
            nbytes = algorithmic_bytes_csr(m)
    call()
    t0 = time.perf_counter()
    call()
    t1 = time.perf_counter() - t0
    reps = max(3, int(budget_s / max(t1, 1e-6)))
    t0 = time.perf_counter()
    for _ in range(reps):
        call()
    dt = (time.perf_counter() - t0) / reps
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": n_threads,
            "nproc": os.cpu_count(), "kind": "oracle loop, rows over OpenMP threads",
            "sample": f"whole matrix, {reps} calls"}


def algorithmic_bytes_csr(m):
    vs = m.values.dtype.itemsize
    return (m.nnz * (vs + 4) + (m.n_rows + 1) * 4 + m.n_cols * m.x.dtype.itemsize
            + m.n_rows * 4)


def run_reference(args, world, rank):
    """--impl reference: the fp64 CPU oracle, as it stands, on this config.
    Each step is one oracle call on a bounded sample of the workload (the
    whole matrix when the K + W calls fit about two minutes, else a leading
    block of rows), so that the run ends within a few minutes."""
    if rank != 0:
        return 0
    key, fmt, desc = WORKLOADS[args.workload]
    m = load_workload(key, "fem" if fmt == "pcg_fem" else fmt)
    steps, warmup = args.steps or 5, max(0, args.warmup)

    rows, nbytes, nnz, call = oracle_call(m, fmt, 1.0)
    t0 = time.perf_counter()
    call()
    t_full = time.perf_counter() - t0
    budget = 120.0
    if t_full * (steps + warmup) > budget:
        frac = budget / (t_full * (steps + warmup))
        rows, nbytes, nnz, call = oracle_call(m, fmt, frac)
    sample = (f"rows 0..{rows - 1} of {m.n_rows} ({nnz} nonzeros) per step"
              if rows < m.n_rows else "whole matrix per step")
    for _ in range(warmup):
        call()
    t0 = time.perf_counter()
    for _ in range(steps):
        call()
    dt = (time.perf_counter() - t0) / steps
    value = nbytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": 1, "steps": steps, "warmup": warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc, "n_rows": m.n_rows, "nnz": m.nnz,
                       "format": fmt},
            "gflops": (m.n_elem * FEM_FLOPS_PER_ELEMENT if fmt == "fem" else 2 * nnz) / dt / 1e9,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def bench_pcg(args, name, world, rank, local, pg):
    """A step is one Jacobi-PCG iteration (one y = A x and its vector
    kernels), timed over whole solves to ||r|| <= 1e-6 ||b|| from x = 0
    (every solve takes the same iterations: checked); the time includes each
    solve's set-up (q = A x0, the initial residual, the graph launch and the
    host's final wait) and, when the iteration count is odd, the skipped
    second half of the last pass of the device-side loop. Bytes per step are
    the product's algorithmic bytes plus PCG_VECTOR_BYTES per unknown."""
    import torch
    import sparse_matrix_vector_gb300 as S

    key, fmt, desc = WORKLOADS[name]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    m = load_workload(key, "fem" if fmt == "pcg_fem" else "csr")
    if fmt == "pcg_fem":
        plan = S.spmv_plan_create_fem(m.nex, m.ney, m.nez, m.rho, m.K0)
    else:
        plan = S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols, format="sell")
    n = m.n_rows
    nbytes = int(plan.info["algorithmic_bytes"]) + PCG_VECTOR_BYTES * n
    b = torch.from_numpy(m.x).to(dev)
    x = torch.zeros(n, dtype=torch.float32, device=dev)
    # "device": the solve's device-side loop (one graph launch a solve);
    # "host": the legacy default stream, on which the library runs host-driven
    # batches of direct launches (for per-kernel profiling; not the headline)
    stream = (torch.cuda.Stream(device=dev) if args.pcg_loop == "device"
              else torch.cuda.default_stream(dev))
    warmup = max(3, args.warmup)
    first = {}

    def solve():
        x.zero_()
        res = S.spmv_pcg_solve(plan, b, x, rel_tol=PCG_TOL, max_iter=20000, stream=stream)
        if res["status"] != "converged" or res["iterations"] != first.setdefault(
                "it", res["iterations"]):
            raise RuntimeError(f"solve did not repeat: {res}, first {first}")
        return res

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            sol = solve()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        solve()
    torch.cuda.synchronize(dev)
    sol_ms = (time.perf_counter() - t0) * 1e3
    iters = first["it"]
    solves = max(3, (args.steps or 2000) // max(iters, 1))
    torch.cuda.synchronize(dev)
    steps = solves * iters

    def solves_region():
        for _ in range(solves):
            solve()

    regions, clk = timed_regions(solves_region, stream, dev, pg, local, steps,
                                 sol_ms / 1e3 / iters, args.regions)
    ms = regions["median_ms"]
    sec_per_step, value, per_launch = job_throughput(nbytes, world, ms, steps)
    t_sol = ms / solves / 1e3
    # end to end: b copied in from pinned host memory, x copied back
    bh = torch.from_numpy(m.x).pin_memory()
    xh = torch.empty(n, dtype=torch.float32).pin_memory()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        b.copy_(bh, non_blocking=True)
        x.zero_()
        res = S.spmv_pcg_solve(plan, b, x, rel_tol=PCG_TOL, max_iter=20000, stream=stream)
        xh.copy_(x, non_blocking=True)
    stream.synchronize()
    e2e_sec = time.perf_counter() - t0
    S.spmv_plan_destroy(plan)
    if rank != 0:
        return None
    traffic = recorded_traffic(name, "fem" if fmt == "pcg_fem" else "sell")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warmup * iters, "ms_per_step": ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": desc, "format": fmt, "n_rows": n, "nnz": m.nnz,
                   "algorithmic_bytes": nbytes,
                   "step": ("one Jacobi-PCG iteration (y = A p with p . q fused in, "
                            "then the update and direction kernels)"),
                   "iterations_per_solve": iters, "rel_tol": PCG_TOL,
                   "pcg_loop": ("device-side loop, one graph launch a solve"
                                if args.pcg_loop == "device" else
                                "host-driven batches on the legacy default stream"),
                   "l2": "matrix >= 3x L2" if nbytes > 3 * 129e6 else
                         "working set fits L2 (matrix-free operator)",
                   "timing": ("CUDA events around each region of whole solves; "
                              "value and ms_per_step from the median region"),
                   "regions": region_report(regions, steps),
                   "parallelism": f"replicas{world}"},
        "solve": {"iterations": sol["iterations"], "status": sol["status"],
                  "ms": t_sol * 1e3, "rel_residual": sol["rel_residual"]},
        "roofline": {"bound": "hbm", "achieved": per_launch, "peak": load_peak()[0],
                     "unit": "GB/s", "frac": per_launch / load_peak()[0],
                     "peak_source": load_peak()[1], "traffic": traffic},
        "e2e": {"value": world * nbytes * res["iterations"] / e2e_sec / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": 4 * n,
                "note": "one whole solve to 1e-6 per step, b in and x out",
                "ms_per_solve": e2e_sec * 1e3},
        # per solve: q = A x0 and the initial residual, then passes of the
        # device-side loop, PCG_BODY iterations of 3 kernels each
        "gpu_launches": solves * (2 + 3 * PCG_BODY * -(-iters // PCG_BODY)),
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        cpu_gbs, sample = oracle_baseline(m, fmt, args.cpu_budget)
        line["cpu_baseline"] = {"value": cpu_gbs, "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": sample}
    return line


def bench_one(args, name, world, rank, local, pg):
    import torch
    import sparse_matrix_vector_gb300 as S

    key, fmt, desc = WORKLOADS[name]
    if fmt.startswith("pcg"):
        return bench_pcg(args, name, world, rank, local, pg)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    t0 = time.perf_counter()
    m = load_workload(key, fmt)
    log(f"[{name}] generated in {time.perf_counter() - t0:.1f}s "
        f"rows={m.n_rows} nnz={m.nnz}")
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)

    def make_plan():
        if fmt == "fem":
            return S.spmv_plan_create_fem(m.nex, m.ney, m.nez, m.rho, m.K0)
        return S.spmv_plan_create(m.row_ptr, m.col_idx, m.values, m.n_cols, format=fmt)

    first = make_plan()
    info = first.info
    nbytes = int(info["algorithmic_bytes"])
    # rotate copies until the loop's footprint is >= 3x L2 (at most 64 copies:
    # below ~6 MB per copy the workload is latency-bound and stays L2-resident)
    copies = min(64, max(1, math.ceil(3 * l2 / nbytes)))
    plans = [first] + [make_plan() for _ in range(copies - 1)]
    xdt = torch.float32 if m.x.dtype == np.float32 else torch.float16
    xs = [torch.from_numpy(m.x).to(dev) for _ in range(copies)]
    ys = [torch.empty(m.n_rows, dtype=torch.float32, device=dev) for _ in range(copies)]
    assert xs[0].dtype == xdt
    stream = torch.cuda.Stream(device=dev)
    peak, peak_src = load_peak()

    steps = args.steps
    if not steps:   # ~0.1 s of work per region at 70% of peak (>= 3 us a step)
        est = max(nbytes / (0.7 * peak * 1e9), 3e-6)
        steps = min(20_000, max(200, int(0.1 / est)))
        steps = int(math.ceil(steps / copies) * copies)
    warmup = max(3, args.warmup)

    def launch(j):
        S.spmv_run(plans[j % copies], xs[j % copies], ys[j % copies], stream=stream)

    with torch.cuda.stream(stream):
        for j in range(warmup):
            launch(j)
    torch.cuda.synchronize(dev)

    # capture the timed steps into graphs of at most 4096 launches each
    graphs = []
    chunk = 4096
    for g0 in range(0, steps, chunk):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(g0, min(steps, g0 + chunk)):
                launch(j)
        graphs.append(g)
    with torch.cuda.stream(stream):   # one untimed replay (graph upload)
        for g in graphs[:1]:
            g.replay()
    torch.cuda.synchronize(dev)

    def replay():
        for g in graphs:
            g.replay()

    regions, clk = timed_regions(replay, stream, dev, pg, local, steps,
                                 max(nbytes / (0.7 * peak * 1e9), 1e-6),
                                 args.regions)
    ms = regions["median_ms"]
    sec_per_step, value, per_launch = job_throughput(nbytes, world, ms, steps)
    flops = m.n_elem * FEM_FLOPS_PER_ELEMENT if fmt == "fem" else 2 * m.nnz
    gflops = world * flops / sec_per_step / 1e9

    # end to end through the C ABI with pinned host buffers: batches of B
    # vectors through spmv_run_host_batch (each vector copied in, multiplied
    # and copied out inside the timed region; one vector's copies overlap its
    # neighbours' products), and the one-vector synchronous spmv_run_host
    x_host = torch.from_numpy(m.x).pin_memory().numpy()
    y_host = torch.empty(m.n_rows, dtype=torch.float32).pin_memory().numpy()
    vec_bytes = m.n_cols * m.x.dtype.itemsize + m.n_rows * 4
    B = int(min(16, max(2, (256 << 20) // max(vec_bytes, 1))))
    xb = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(m.x, (B, m.n_cols)))
                          ).pin_memory().numpy()
    yb = torch.empty((B, m.n_rows), dtype=torch.float32).pin_memory().numpy()

    def e2e_time(call, n_steps, per_call):
        for _ in range(3):
            call(0)
        if pg is not None:
            torch.distributed.barrier()
        t = time.perf_counter()
        for j in range(n_steps // per_call):
            call(j)
        t = (time.perf_counter() - t) / (n_steps // per_call * per_call)
        if pg is not None:
            tt = torch.tensor([t], device=dev)
            torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
            t = float(tt.item())
        return t

    e2e_steps = max(20, min(2000, int(0.5 / max(sec_per_step * 4, 1e-6))))
    e2e_sec = e2e_time(lambda j: S.spmv_run_host_batch(plans[j % copies], xb, yb, stream=stream),
                       max(e2e_steps, 4 * B), B)
    e2e_single_sec = e2e_time(
        lambda j: S.spmv_run_host(plans[j % copies], x_host, y_host, stream=stream),
        e2e_steps, 1)

    line = None
    if rank == 0:
        traffic = recorded_traffic(name, fmt, bool(info.get("segments", 0)))
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": ms / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if m.values.dtype == np.float32 else "f16",
            "data": "synthetic",
            "config": {"workload": desc, "format": fmt, "n_rows": m.n_rows,
                       "n_cols": m.n_cols, "nnz": m.nnz,
                       "stored_entries": int(info["n_entries"]),
                       "algorithmic_bytes": nbytes,
                       "bins_rows": info["rows_per_bin"],
                       "bins_tiles": info["tiles_per_bin"],
                       "grid": info["grid"], "x_in_smem": bool(info["x_in_smem"]),
                       "l2": (f"rotating {copies} resident copies, "
                              f"{copies * nbytes / 2**20:.0f} MiB "
                              + (">= 3x" if copies * nbytes >= 3 * l2 else
                                 "< L2: latency-bound, L2-resident,")
                              + f" L2 ({l2 / 2**20:.0f} MiB)"),
                       "timing": ("CUDA graphs of back-to-back spmv_run, CUDA "
                                  "events on the launching stream around each "
                                  "region of `steps` steps; value and "
                                  "ms_per_step from the median region"),
                       "regions": region_report(regions, steps),
                       "parallelism": f"replicas{world}"},
            "gflops": gflops,
            "roofline": ({"bound": "hbm", "achieved": per_launch, "peak": peak,
                          "unit": "GB/s", "frac": per_launch / peak,
                          "peak_source": peak_src, "traffic": traffic}
                         if fmt != "fem" else
                         {"bound": "alu", "achieved": gflops / world / 1e3,
                          "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s",
                          "frac": gflops / world / 1e3 / FP32_PEAK_TFLOPS,
                          "peak_source": "152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz",
                          "traffic": traffic,
                          "hbm_achieved_GBs": per_launch}),
            "e2e": {"value": world * nbytes / e2e_sec / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": int(m.n_cols * m.x.dtype.itemsize),
                    "d2h_bytes_per_step": int(m.n_rows * 4),
                    "ms_per_step": e2e_sec * 1e3,
                    "call": f"spmv_run_host_batch, {B} vectors per call",
                    "one_vector_call": {"value": world * nbytes / e2e_single_sec / 1e9,
                                        "ms_per_step": e2e_single_sec * 1e3,
                                        "call": "spmv_run_host (copy in, run, copy out, "
                                                "synchronize)"}},
            "gpu_launches": int(info["launches_per_run"]) * steps,
            "clocks": clk,
        }
        if world == 1 and not args.no_cpu_baseline:
            cpu_gbs, sample = oracle_baseline(m, fmt, args.cpu_budget)
            line["cpu_baseline"] = {"value": cpu_gbs, "unit": "GB/s", "cores": 1,
                                    "kind": "oracle", "sample": sample}
            par = parallel_baseline(m, fmt, args.cpu_budget / 2)
            if par is not None:
                line["cpu_baseline_all_cores"] = par
    for p in plans:
        S.spmv_plan_destroy(p)
    del xs, ys, graphs
    torch.cuda.empty_cache()
    return line


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps per timed region (default: ~0.1 s of work)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--regions", type=int, default=0,
                    help="timed regions (default: enough for ~0.6 s of timed "
                         "work, at least %d)" % MIN_REGIONS)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="one of %s, or 'all'" % ", ".join(WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pcg-loop", choices=["device", "host"], default="device",
                    help="CG lines: the solve's device-side loop (default), or host-driven "
                         "batches of direct launches (for per-kernel profiling)")
    args = ap.parse_args(argv)
    world, rank, local = dist_setup()
    if args.workload != "all" and args.workload not in WORKLOADS:
        ap.error(f"unknown workload {args.workload}")

    if args.impl == "reference":
        if args.workload == "all":
            for name in WORKLOADS:
                args.workload = name
                run_reference(args, world, rank)
            return 0
        return run_reference(args, world, rank)

    import torch
    pg = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist.group.WORLD
    names = list(WORKLOADS) if args.workload == "all" else [args.workload]
    for name in names:
        line = bench_one(args, name, world, rank, local, pg)
        if line is not None:
            print(json.dumps(line), flush=True)
    if pg is not None:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
