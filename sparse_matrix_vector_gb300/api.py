"""Python binding of the C ABI (include/spmv.h), same names as the C calls.

Only argument marshalling lives here: numpy arrays become host pointers,
torch CUDA tensors become device pointers and the current torch stream
becomes the cudaStream_t. Every step of y = A x runs in the library's
kernels; if the library is not built, the first call raises.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from . import _lib
from ._lib import (SPMV_DELTA_FEWEST_BYTES, SPMV_DELTA_SPARSITY_TABLE, SPMV_F16, SPMV_F32,
                   SPMV_FORMAT_CSR, SPMV_FORMAT_DELTA2, SPMV_FORMAT_DELTA4,
                   SPMV_FORMAT_DELTA8, SPMV_FORMAT_DELTA_AUTO, SPMV_FORMAT_AUTO,
                   SPMV_FORMAT_SELL)

FORMATS = {"csr": SPMV_FORMAT_CSR, "delta4": SPMV_FORMAT_DELTA4,
           "delta2": SPMV_FORMAT_DELTA2, "delta8": SPMV_FORMAT_DELTA8,
           "delta": SPMV_FORMAT_DELTA_AUTO, "sell": SPMV_FORMAT_SELL,
           "auto": SPMV_FORMAT_AUTO}
FORMAT_NAMES = {v: k for k, v in FORMATS.items()}
DELTA_POLICIES = {"fewest_bytes": SPMV_DELTA_FEWEST_BYTES,
                  "sparsity_table": SPMV_DELTA_SPARSITY_TABLE}


class SpmvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        msg = _lib.load().spmv_status_string(status).decode()
        name = _lib.STATUS_NAMES.get(self.status, str(status))
        super().__init__(f"{where}: {name} ({msg})")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise SpmvError(status, where)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _format_code(fmt) -> int:
    if isinstance(fmt, str):
        return FORMATS[fmt.lower()]
    return int(fmt)


@dataclass
class _HostCSR:
    """Keeps the contiguous host copies alive while the C call runs."""
    struct: _lib.spmv_csr
    keep: tuple


def _host_csr(row_ptr, col_idx, values, n_cols: int) -> _HostCSR:
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    vals = np.asarray(values)
    if vals.dtype == np.float16:
        dt = SPMV_F16
        v = np.ascontiguousarray(vals)
    elif vals.dtype == np.float32:
        dt = SPMV_F32
        v = np.ascontiguousarray(vals)
    else:
        raise TypeError("values must be float32 or float16")
    s = _lib.spmv_csr(n_rows=rp.shape[0] - 1, n_cols=int(n_cols),
                      nnz=int(ci.shape[0]), row_ptr=rp.ctypes.data,
                      col_idx=ci.ctypes.data if ci.size else None,
                      values=v.ctypes.data if v.size else None,
                      value_dtype=dt)
    return _HostCSR(s, (rp, ci, v))


def spmv_plan_options(**kw) -> _lib.spmv_plan_options:
    """Library defaults, overridden by keyword (tile_nnz, tile_rows,
    cta_row_min, split_row_min, split_chunk, x_smem, reduce, lanes,
    interleave, sell_sigma, csr_kernel, delta_kernel)."""
    o = _lib.spmv_plan_options()
    _lib.load().spmv_plan_options_init(ctypes.byref(o))
    for k, v in kw.items():
        if not hasattr(o, k) or k == "reserved":
            raise KeyError(k)
        setattr(o, k, int(v))
    return o


def _info_dict(info: _lib.spmv_plan_info) -> dict:
    d = {}
    for name, _t in info._fields_:
        if name == "reserved":
            continue
        v = getattr(info, name)
        d[name] = list(v) if hasattr(v, "__len__") else int(v)
    return d


def spmv_status_string(status: int) -> str:
    return _lib.load().spmv_status_string(int(status)).decode()


def spmv_abi_version() -> int:
    return int(_lib.load().spmv_abi_version())


@dataclass
class DeltaMatrix:
    """A DELTA matrix (deltas of `bits` bits) copied out of the library
    (numpy arrays)."""
    n_rows: int
    n_cols: int
    nnz: int
    row_ptr: np.ndarray   # int64[n_rows + 1]
    values: np.ndarray    # uint16[n_entries] (fp16 bit patterns)
    words: np.ndarray     # uint32[n_entries * bits / 32]
    n_gap_pads: int
    n_align_pads: int
    n_explicit_zeros: int
    bits: int = 4

    @property
    def n_entries(self) -> int:
        return int(self.row_ptr[-1]) if self.row_ptr.size else 0


def spmv_convert(row_ptr, col_idx, values, n_cols: int, bits: int = 4) -> DeltaMatrix:
    """CSR (fp16 values) -> DELTA with `bits`-bit deltas (2, 4 or 8) on the
    host, by the library's converter (spmv_convert_bits)."""
    h = _host_csr(row_ptr, col_idx, values, n_cols)
    d = _lib.spmv_delta()
    lib = _lib.load()
    _check(lib.spmv_convert_bits(ctypes.byref(h.struct), int(bits), ctypes.byref(d)),
           "spmv_convert_bits")
    try:
        n = int(d.n_entries)
        b = int(d.delta_bits)
        rp = np.ctypeslib.as_array(ctypes.cast(d.row_ptr, ctypes.POINTER(ctypes.c_int64)),
                                   shape=(d.n_rows + 1,)).copy()
        if n:
            vals = np.ctypeslib.as_array(
                ctypes.cast(d.values, ctypes.POINTER(ctypes.c_uint16)), shape=(n,)).copy()
            words = np.ctypeslib.as_array(
                ctypes.cast(d.words, ctypes.POINTER(ctypes.c_uint32)),
                shape=(n * b // 32,)).copy()
        else:
            vals = np.zeros(0, np.uint16)
            words = np.zeros(0, np.uint32)
        return DeltaMatrix(int(d.n_rows), int(d.n_cols), int(d.nnz), rp, vals,
                           words, int(d.n_gap_pads), int(d.n_align_pads),
                           int(d.n_explicit_zeros), b)
    finally:
        lib.spmv_delta_free(ctypes.byref(d))


def spmv_delta_select_bits(row_ptr, col_idx, values, n_cols: int,
                           policy="fewest_bytes"):
    """Delta width (2, 4 or 8) for a CSR matrix with fp16 values under
    `policy` ("fewest_bytes" or "sparsity_table"), and the entries each width
    would store: returns (bits, {2: n, 4: n, 8: n})."""
    h = _host_csr(row_ptr, col_idx, values, n_cols)
    code = DELTA_POLICIES[policy] if isinstance(policy, str) else int(policy)
    bits = ctypes.c_int32()
    entries = (ctypes.c_int64 * 3)()
    _check(_lib.load().spmv_delta_select_bits(ctypes.byref(h.struct), code,
                                              ctypes.byref(bits), entries),
           "spmv_delta_select_bits")
    return int(bits.value), {2: int(entries[0]), 4: int(entries[1]), 8: int(entries[2])}


@dataclass
class SellMatrix:
    """A sliced-ELL matrix copied out of the library (numpy arrays)."""
    n_rows: int
    n_cols: int
    nnz: int
    C: int
    sigma: int
    slice_ptr: np.ndarray   # int64[n_slices + 1]
    perm: np.ndarray        # int32[n_slices * C], -1 past the last row
    cols: np.ndarray        # int32[n_slots]
    values: np.ndarray      # float32 or float16 [n_slots]


def spmv_convert_sell(row_ptr, col_idx, values, n_cols: int, sigma: int = 1) -> SellMatrix:
    """CSR (fp32 or fp16 values) -> sliced ELL on the host, by the library's
    converter (spmv_convert_sell)."""
    h = _host_csr(row_ptr, col_idx, values, n_cols)
    sl = _lib.spmv_sell()
    lib = _lib.load()
    _check(lib.spmv_convert_sell(ctypes.byref(h.struct), int(sigma), ctypes.byref(sl)),
           "spmv_convert_sell")
    try:
        ns, slots = int(sl.n_slices), int(sl.n_slots)

        def arr(ptr, ctype, n, dtype):
            if n == 0:
                return np.zeros(0, dtype)
            return np.ctypeslib.as_array(ctypes.cast(ptr, ctypes.POINTER(ctype)),
                                         shape=(n,)).copy().view(dtype)
        vdt = np.float32 if sl.value_dtype == SPMV_F32 else np.float16
        vct = ctypes.c_uint32 if sl.value_dtype == SPMV_F32 else ctypes.c_uint16
        return SellMatrix(int(sl.n_rows), int(sl.n_cols), int(sl.nnz), int(sl.C),
                          int(sl.sigma),
                          arr(sl.slice_ptr, ctypes.c_int64, ns + 1, np.int64),
                          arr(sl.perm, ctypes.c_int32, ns * int(sl.C), np.int32),
                          arr(sl.cols, ctypes.c_int32, slots, np.int32),
                          arr(sl.values, vct, slots, vdt))
    finally:
        lib.spmv_sell_free(ctypes.byref(sl))


def spmv_select_format(row_ptr, col_idx, values, n_cols: int):
    """Format by the CV of the row lengths: returns (format name, sigma, cv)
    with format "sell" or "csr"."""
    h = _host_csr(row_ptr, col_idx, values, n_cols)
    fmt, sigma, cv = ctypes.c_int(), ctypes.c_int32(), ctypes.c_double()
    _check(_lib.load().spmv_select_format(ctypes.byref(h.struct), ctypes.byref(fmt),
                                          ctypes.byref(sigma), ctypes.byref(cv)),
           "spmv_select_format")
    return FORMAT_NAMES[int(fmt.value)], int(sigma.value), float(cv.value)


def spmv_plan_inspect(row_ptr, col_idx, values, n_cols: int, format="csr",
                      options=None) -> dict:
    """Host-only planner dry run (no device needed)."""
    h = _host_csr(row_ptr, col_idx, values, n_cols)
    info = _lib.spmv_plan_info()
    opts = ctypes.byref(options) if options is not None else None
    _check(_lib.load().spmv_plan_inspect(ctypes.byref(h.struct),
                                         _format_code(format), opts,
                                         ctypes.byref(info)),
           "spmv_plan_inspect")
    return _info_dict(info)


class Plan:
    """Owns a spmv_plan*; device memory is released by spmv_plan_destroy
    (or when the object is garbage collected)."""

    def __init__(self, handle: int, device: int):
        self._handle = ctypes.c_void_p(handle)
        self.device = device
        info = _lib.spmv_plan_info()
        _check(_lib.load().spmv_plan_get_info(self._handle, ctypes.byref(info)),
               "spmv_plan_get_info")
        self.info = _info_dict(info)
        self.x_dtype_code = SPMV_F32 if self.info["value_dtype"] == SPMV_F32 else SPMV_F16

    @property
    def handle(self):
        if self._handle is None or not self._handle.value:
            raise ValueError("plan has been destroyed")
        return self._handle

    @property
    def n_rows(self) -> int:
        return self.info["n_rows"]

    @property
    def n_cols(self) -> int:
        return self.info["n_cols"]

    def destroy(self) -> None:
        if self._handle is not None and self._handle.value:
            _lib.load().spmv_plan_destroy(self._handle)
        self._handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def _current_device() -> int:
    import torch
    return torch.cuda.current_device()


def spmv_plan_create(row_ptr, col_idx, values, n_cols: int, format="csr",
                     options=None) -> Plan:
    """Validate, plan and upload a CSR matrix on the current CUDA device."""
    h = _host_csr(row_ptr, col_idx, values, n_cols)
    out = ctypes.c_void_p()
    lib = _lib.load()
    if options is None:
        st = lib.spmv_plan_create(ctypes.byref(h.struct), _format_code(format),
                                  ctypes.byref(out))
    else:
        st = lib.spmv_plan_create_ex(ctypes.byref(h.struct), _format_code(format),
                                     ctypes.byref(options), ctypes.byref(out))
    _check(st, "spmv_plan_create")
    return Plan(out.value, _current_device())


def spmv_plan_create_fem(nex: int, ney: int, nez: int, rho, K0) -> Plan:
    """Plan the matrix-free stiffness operator of an nex x ney x nez hex mesh
    (element matrices rho[e] * K0) on the current CUDA device; x and y are
    fp32 with 3 (nex+1)(ney+1)(nez+1) entries."""
    r = np.ascontiguousarray(rho, dtype=np.float32)
    k = np.ascontiguousarray(K0, dtype=np.float32).reshape(-1)
    if k.size != 24 * 24:
        raise ValueError("K0 must hold 24 x 24 values")
    mesh = _lib.spmv_fem_mesh(nex=int(nex), ney=int(ney), nez=int(nez),
                              rho=r.ctypes.data if r.size else None, K0=k.ctypes.data)
    out = ctypes.c_void_p()
    _check(_lib.load().spmv_plan_create_fem(ctypes.byref(mesh), ctypes.byref(out)),
           "spmv_plan_create_fem")
    return Plan(out.value, _current_device())


def spmv_plan_create_delta(delta: DeltaMatrix, options=None) -> Plan:
    """Plan from an already converted DELTA matrix."""
    rp = np.ascontiguousarray(delta.row_ptr, dtype=np.int64)
    vals = np.ascontiguousarray(delta.values, dtype=np.uint16)
    words = np.ascontiguousarray(delta.words, dtype=np.uint32)
    d = _lib.spmv_delta(n_rows=delta.n_rows, n_cols=delta.n_cols, nnz=delta.nnz,
                        n_entries=int(rp[-1]) if rp.size else 0,
                        n_gap_pads=delta.n_gap_pads,
                        n_align_pads=delta.n_align_pads,
                        n_explicit_zeros=delta.n_explicit_zeros,
                        values=vals.ctypes.data if vals.size else None,
                        words=words.ctypes.data if words.size else None,
                        row_ptr=rp.ctypes.data, delta_bits=int(delta.bits))
    out = ctypes.c_void_p()
    opts = ctypes.byref(options) if options is not None else None
    _check(_lib.load().spmv_plan_create_delta(ctypes.byref(d), opts,
                                              ctypes.byref(out)),
           "spmv_plan_create_delta")
    return Plan(out.value, _current_device())


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev_ptr(t, n: int, dtype_code: int | None, what: str) -> int:
    if isinstance(t, int):
        return t
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor or a device pointer")
    if not t.is_contiguous() or t.numel() != n:
        raise ValueError(f"{what} must be contiguous with {n} elements")
    want = {SPMV_F32: torch.float32, SPMV_F16: torch.float16}[dtype_code]
    if t.dtype != want:
        raise TypeError(f"{what} must be {want}, got {t.dtype}")
    return t.data_ptr()


def spmv_run(plan: Plan, x, y, stream=None) -> None:
    """y = A x on the plan's device, asynchronous on `stream` (default: the
    current torch stream). x: fp32 (fp32 CSR) or fp16 tensor of n_cols;
    y: fp32 tensor of n_rows, overwritten."""
    xp = _dev_ptr(x, plan.n_cols, plan.x_dtype_code, "x")
    yp = _dev_ptr(y, plan.n_rows, SPMV_F32, "y")
    _check(_lib.load().spmv_run(plan.handle, xp, yp, _stream_handle(stream)),
           "spmv_run")


PCG_STATUS = {1: "converged", 2: "iteration limit", 3: "breakdown"}


def spmv_pcg_solve(plan: Plan, b, x, rel_tol: float = 1e-6, max_iter: int = 1000,
                   check_every: int = 16, diag=None, stream=None) -> dict:
    """Jacobi-preconditioned CG for A x = b on the plan's device: b and x
    are fp32 CUDA tensors of n (x: initial guess in, solution out); diag is
    the preconditioner's diagonal (default: the plan's own). Synchronizes
    the stream; returns iterations, status and ||r|| / ||b||."""
    n = plan.n_rows
    bp = _dev_ptr(b, n, SPMV_F32, "b")
    xp = _dev_ptr(x, n, SPMV_F32, "x")
    dp = None if diag is None else _dev_ptr(diag, n, SPMV_F32, "diag")
    res = _lib.spmv_pcg_result()
    _check(_lib.load().spmv_pcg_solve(plan.handle, dp, bp, xp, float(rel_tol), int(max_iter),
                                      int(check_every), _stream_handle(stream),
                                      ctypes.byref(res)),
           "spmv_pcg_solve")
    return {"iterations": int(res.iterations), "status": PCG_STATUS.get(int(res.status), "?"),
            "rel_residual": float(res.rel_residual)}


def spmv_run_host(plan: Plan, x_host: np.ndarray, y_host: np.ndarray,
                  stream=None) -> None:
    """End-to-end y = A x with host arrays (copies inside the call; returns
    after the stream has finished)."""
    want = np.float32 if plan.x_dtype_code == SPMV_F32 else np.float16
    if (x_host.dtype != want or not x_host.flags.c_contiguous
            or x_host.size != plan.n_cols):
        raise ValueError("x_host has the wrong dtype, size or layout")
    if (y_host.dtype != np.float32 or not y_host.flags.c_contiguous
            or y_host.size != plan.n_rows or not y_host.flags.writeable):
        raise ValueError("y_host must be a writeable contiguous float32 array")
    _check(_lib.load().spmv_run_host(plan.handle, x_host.ctypes.data,
                                     y_host.ctypes.data, _stream_handle(stream)),
           "spmv_run_host")


def spmv_run_host_batch(plan: Plan, x_host: np.ndarray, y_host: np.ndarray,
                        stream=None) -> None:
    """End-to-end y[i] = A x[i] for a batch of host vectors (x_host: count x
    n_cols of the plan's x dtype, y_host: count x n_rows float32, both
    C-contiguous); copies and products of neighbouring vectors overlap.
    Returns after the last y is in host memory."""
    want = np.float32 if plan.x_dtype_code == SPMV_F32 else np.float16
    if (x_host.dtype != want or not x_host.flags.c_contiguous or x_host.ndim != 2
            or x_host.shape[1] != plan.n_cols):
        raise ValueError("x_host must be a C-contiguous (count, n_cols) array of the plan's x dtype")
    count = x_host.shape[0]
    if (y_host.dtype != np.float32 or not y_host.flags.c_contiguous or y_host.ndim != 2
            or y_host.shape != (count, plan.n_rows) or not y_host.flags.writeable):
        raise ValueError("y_host must be a writeable C-contiguous (count, n_rows) float32 array")
    _check(_lib.load().spmv_run_host_batch(plan.handle, int(count), x_host.ctypes.data,
                                           y_host.ctypes.data, _stream_handle(stream)),
           "spmv_run_host_batch")


def spmv_csr_run_noalloc(n_rows: int, n_cols: int, row_ptr, col_idx, values,
                         x, y, stream=None) -> None:
    """Allocation-free y = A x on a CSR matrix held in caller-owned CUDA
    tensors (row_ptr/col_idx int32, values and x fp32 or fp16, y fp32), all
    contiguous and on the current CUDA device. For callers that may not
    allocate device memory; see include/spmv.h."""
    import torch
    for name, t in (("row_ptr", row_ptr), ("col_idx", col_idx)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    if (values.dtype not in (torch.float32, torch.float16) or not values.is_cuda
            or not values.is_contiguous()):
        raise TypeError("values must be a contiguous float32 or float16 CUDA tensor")
    code = SPMV_F32 if values.dtype == torch.float32 else SPMV_F16
    if row_ptr.numel() != n_rows + 1:
        raise ValueError("row_ptr must have n_rows + 1 elements")
    nnz = int(col_idx.numel())
    if values.numel() != nnz:
        raise ValueError("values and col_idx differ in length")
    xp = _dev_ptr(x, n_cols, code, "x")
    yp = _dev_ptr(y, n_rows, SPMV_F32, "y")
    here = torch.cuda.current_device()
    for name, t in (("row_ptr", row_ptr), ("col_idx", col_idx), ("values", values),
                    ("x", x), ("y", y)):
        if isinstance(t, torch.Tensor) and t.device.index != here:
            raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{here}")
    _check(_lib.load().spmv_csr_run_noalloc(
        n_rows, n_cols, nnz, row_ptr.data_ptr(), col_idx.data_ptr(),
        values.data_ptr(), code, xp, yp, _stream_handle(stream)),
        "spmv_csr_run_noalloc")


def spmv_plan_check(plan: Plan) -> None:
    _check(_lib.load().spmv_plan_check(plan.handle), "spmv_plan_check")


def spmv_plan_destroy(plan: Plan) -> None:
    plan.destroy()
