"""GB300-native sparse matrix-vector multiply y = A x (fp32 / fp16 CSR, sliced
ELL, the column-delta format with 2-, 4- or 8-bit deltas, and a matrix-free
hex-mesh stiffness operator) behind a C ABI, ``include/spmv.h``.

The compiled library is ``libspmv_gb300.so`` next to this file (built by
``sparse_matrix_vector_gb300.build``). This package only marshals arguments.
"""
from .api import (  # noqa: F401
    DeltaMatrix, Plan, SellMatrix, SpmvError, spmv_abi_version, spmv_convert,
    spmv_convert_sell, spmv_delta_select_bits, spmv_select_format,
    spmv_csr_run_noalloc,
    spmv_plan_check, spmv_plan_create, spmv_plan_create_delta, spmv_plan_create_fem,
    spmv_pcg_solve, spmv_plan_destroy, spmv_plan_inspect, spmv_plan_options, spmv_run,
    spmv_run_host, spmv_run_host_batch, spmv_status_string,
)
from ._lib import (  # noqa: F401
    SPMV_F16, SPMV_F32, SPMV_FORMAT_CSR, SPMV_FORMAT_DELTA2, SPMV_FORMAT_DELTA4,
    SPMV_FORMAT_DELTA8, SPMV_FORMAT_DELTA_AUTO, SPMV_FORMAT_SELL, SPMV_FORMAT_AUTO,
    SPMV_FORMAT_FEM,
)
