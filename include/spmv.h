/*
 * spmv.h -- C ABI of the GB300 sparse matrix-vector multiply library.
 *
 * The library computes y = A x on one CUDA device (sm_103a) for a sparse
 * matrix A stored either as
 *   - CSR (row_ptr / col_idx / values), values fp32 or fp16; or
 *   - DELTA4: fp16 values with 4-bit column deltas packed eight to a 32-bit
 *     word, zero-valued padding entries where a gap does not fit in 4 bits,
 *     and CSR-like row pointers over the stored entries (DELTA2 / DELTA8:
 *     the same with 2- or 8-bit deltas, 16 or 4 to a word); or
 *   - SELL: sliced ELLPACK, fp32 or fp16 values: rows cut into slices of
 *     SPMV_SELL_C rows, each slice padded with zeros to its longest row and
 *     stored column-major (optionally rows sorted by length first); or
 *   - FEM: the stiffness matrix of a structured hexahedral mesh, never
 *     assembled: y = sum over elements of rho_e K0 applied to the element's
 *     24 dofs (spmv_plan_create_fem).
 * x is fp32 for fp32 values and fp16 otherwise; y is always fp32 and every
 * product is accumulated in fp32.
 *
 * Sources (web pages, by title and section):
 *   [CSR]   "CUDA CSR SpMV optimisation" (codechina.net), section 2.1: the CSR
 *           arrays and the definition y[row] = sum over k in
 *           [row_ptr[row], row_ptr[row+1]) of values[k] * x[col_idx[k]],
 *           and a table comparing COO / CSR / ELL / HYB; section 2.2:
 *           one-time upload of the arrays with cudaMalloc and an
 *           asynchronous copy, kernel launches on a stream chosen by the
 *           format, and the choice among ELL / HYB / CSR by the coefficient
 *           of variation (CV) of the row lengths.
 *   [MACKO] "MACKO-SpMV" (maplevalley.com.cn), section 2.1: the format
 *           struct {values with zero placeholders, 4-bit deltas, row
 *           pointers} and its four encoding steps; section 2.2: the warp
 *           decode (prefix sum of deltas) and half2 multiply.
 *   [FEM]   "Fused FEM matvec" (bbs.csdn.net), section 2.1: y = K x as gather,
 *           element product and scatter-add; section 2.2: the three fused in
 *           one kernel; section 5.2: one element matrix shared by all
 *           elements (here scaled per element by a density, as in SIMP).
 *   [SPGEMM] "Hash-based multi-phase SpGEMM" (mlqm.cn), section 2.1.1: rows
 *           grouped by work into bins served by partial-warp, warp and
 *           block-per-row kernels; section 5.2: batching of tiny rows.
 *
 * Conventions for every call:
 *   - Host pointers are read only during the call; nothing keeps them.
 *   - Device pointers (x_dev, y_dev) are caller-owned CUDA device memory on
 *     the device the plan was created on.
 *   - Errors are returned as spmv_status; no call aborts, throws or prints.
 *   - A plan is not thread-safe: calls that use one plan must be ordered
 *     (one host thread, one stream or explicit stream ordering), because a
 *     run may use scratch memory owned by the plan.
 */
#ifndef SPMV_GB300_SPMV_H
#define SPMV_GB300_SPMV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPMV_ABI_VERSION 6

/* Rows per slice of the SELL format (one warp of the kernel per slice). */
#define SPMV_SELL_C 32

typedef enum spmv_status {
  SPMV_OK = 0,
  SPMV_ERR_INVALID_ARG = 1,      /* null pointer, negative size, bad enum   */
  SPMV_ERR_BAD_ROW_PTR = 2,      /* row_ptr[0] != 0, decreasing, or last != nnz */
  SPMV_ERR_COL_OUT_OF_RANGE = 3, /* a column (or decoded column) >= n_cols  */
  SPMV_ERR_UNSORTED_OR_DUPLICATE_COLS = 4, /* DELTA needs increasing cols  */
  SPMV_ERR_UNSUPPORTED = 5,      /* format / dtype combination not provided */
  SPMV_ERR_OUT_OF_MEMORY = 6,    /* host or device allocation failed        */
  SPMV_ERR_CUDA = 7,             /* a CUDA runtime call failed (no device…) */
  SPMV_ERR_TOO_LARGE = 8,        /* sizes exceed 32-bit device indexing     */
  SPMV_ERR_WRONG_DEVICE = 9,     /* current device differs from the plan's  */
  SPMV_ERR_DEVICE_STATUS = 10    /* a kernel reported an error in the plan's
                                    device status word (bounded wait expired) */
} spmv_status;

typedef enum spmv_dtype { SPMV_F32 = 0, SPMV_F16 = 1 } spmv_dtype;

typedef enum spmv_format {
  SPMV_FORMAT_CSR = 0,     /* [CSR] section 2.1                               */
  SPMV_FORMAT_DELTA4 = 1,  /* [MACKO] section 2.1, 4-bit deltas               */
  SPMV_FORMAT_DELTA2 = 2,  /* the same format with 2-bit deltas ([MACKO] 3.3) */
  SPMV_FORMAT_DELTA8 = 3,  /* the same format with 8-bit deltas ([MACKO] 3.3) */
  SPMV_FORMAT_DELTA_AUTO = 4, /* the width spmv_delta_select_bits picks under
                                 SPMV_DELTA_FEWEST_BYTES; plans and their info
                                 report the chosen width's format code      */
  SPMV_FORMAT_SELL = 5,   /* sliced ELL ([CSR] 2.1 ELL, in slices of
                             SPMV_SELL_C rows); sigma from the options      */
  SPMV_FORMAT_FEM = 7,    /* matrix-free hex-mesh stiffness operator; made
                             by spmv_plan_create_fem only                  */
  SPMV_FORMAT_AUTO = 6    /* CSR or SELL by the CV of the row lengths
                             (spmv_select_format), except that matrices
                             whose rows hold more than 128 or fewer than
                             16 nonzeros on average take CSR (a lane per
                             row serialises long rows; a SELL warp over
                             very short rows has too little to read);
                             plans and their info report the chosen
                             format                                         */
} spmv_format;

/* How spmv_delta_select_bits picks a delta width ([MACKO] section 3.3). */
typedef enum spmv_delta_policy {
  /* the width whose encoding stores the fewest bytes (values, deltas and
   * row pointers; padding included); ties go to the wider field */
  SPMV_DELTA_FEWEST_BYTES = 0,
  /* the sparsity table of [MACKO] 3.3 as printed, with s = 1 - nnz /
   * (n_rows * n_cols): s < 0.3 -> 8 bits, 0.3 <= s <= 0.7 -> 4 (the default
   * where the 2- and 4-bit ranges overlap), s > 0.7 -> 2 (the 1-bit width the
   * table gives above 0.9 is not provided; 2 is the nearest) */
  SPMV_DELTA_SPARSITY_TABLE = 1
} spmv_delta_policy;

/* A CSR matrix in HOST memory ([CSR] section 2.1).
 * row_ptr: n_rows+1 offsets, row_ptr[0] == 0, non-decreasing, last == nnz.
 * col_idx: nnz column indices in [0, n_cols). Any order and repeats are
 *          accepted for SPMV_FORMAT_CSR and SELL (repeats add up); the
 *          DELTA formats need strictly increasing columns inside every row.
 * values:  nnz elements of value_dtype (fp16 given as its 16-bit pattern). */
typedef struct spmv_csr {
  int32_t n_rows;
  int32_t n_cols;
  int64_t nnz;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  const void* values;
  spmv_dtype value_dtype;
} spmv_csr;

/* A column-delta matrix in HOST memory ([MACKO] section 2.1), as produced by
 * spmv_convert (4-bit deltas) or spmv_convert_bits (b = 2, 4 or 8 bits;
 * [MACKO] section 3.3 lists the widths). With D = 2^b - 1 and P = 32 / b
 * deltas per 32-bit word, each row is encoded, with the running column c
 * starting at 0 at the start of the row:
 *   for each nonzero (in increasing column order) at column j:
 *     d = j - c; while d > D emit (+0.0, D), c += D, d -= D;
 *     emit (value, d); c = j;
 *   then emit (+0.0, 0) until the row holds a multiple of P entries.
 * Entry e stores its value in values[e] and its delta in bits
 * b*(e%P)..b*(e%P)+b-1 of words[e/P] (for b = 4: nibble e%8 of word e/8).
 * row_ptr[r] is the index of the first entry of row r (always a multiple of
 * P). A stored +0.0 (bits 0x0000) is indistinguishable from padding;
 * decoding drops every such entry. */
typedef struct spmv_delta {
  int32_t n_rows;
  int32_t n_cols;
  int64_t nnz;              /* nonzeros encoded (entries that are not padding) */
  int64_t n_entries;        /* stored entries, padding included              */
  int64_t n_gap_pads;       /* padding entries inserted for gaps > D         */
  int64_t n_align_pads;     /* padding entries that round rows up to P       */
  int64_t n_explicit_zeros; /* input values equal to +0.0 (stored as such)   */
  uint16_t* values;         /* n_entries fp16 bit patterns                   */
  uint32_t* words;          /* n_entries / P words of packed deltas          */
  int64_t* row_ptr;         /* n_rows + 1 entry offsets                      */
  int32_t delta_bits;       /* b: 2, 4 or 8 (0 is read as 4)                 */
  int32_t reserved;
} spmv_delta;

/* A sliced-ELL matrix in HOST memory ([CSR] section 2.1, ELL in slices), as
 * produced by spmv_convert_sell. Rows are first put in sorted order: inside
 * each window of `sigma` consecutive rows, by decreasing length, rows of
 * equal length in their original order (sigma = 1: the original order). The
 * sorted rows are cut into slices of C = SPMV_SELL_C; slice s is as wide as
 * its longest row, w_s = (slice_ptr[s+1] - slice_ptr[s]) / C, and slot
 * (k, lane) of slice s, at slice_ptr[s] + k * C + lane, holds the k-th
 * stored entry (in CSR order) of the slice's lane-th row. Slots past a row's
 * length hold value 0 at the row's last column (column 0 for an empty row
 * and for lanes of the last slice that hold no row).
 * perm[s * C + lane] is the original row index of that lane's row, or -1. */
typedef struct spmv_sell {
  int32_t n_rows;
  int32_t n_cols;
  int64_t nnz;
  int32_t C;                /* SPMV_SELL_C                                   */
  int32_t sigma;            /* sorting window (1: rows in order)             */
  int64_t n_slices;         /* ceil(n_rows / C)                              */
  int64_t n_slots;          /* stored slots, padding included                */
  int64_t* slice_ptr;       /* n_slices + 1 slot offsets                     */
  int32_t* perm;            /* n_slices * C original rows (-1: none)         */
  int32_t* cols;            /* n_slots column indices                        */
  void* values;             /* n_slots elements of value_dtype               */
  spmv_dtype value_dtype;
  int32_t reserved;
} spmv_sell;

/* Planner knobs ([SPGEMM] section 2.1.1 grouping; [MACKO] section 3.3
 * dynamic scheduling). Zero / negative fields mean "library default". */
typedef struct spmv_plan_options {
  int32_t tile_nnz;      /* nonzero budget of a short-row tile             */
  int32_t tile_rows;     /* row budget of a short-row tile                 */
  int32_t cta_row_min;   /* rows longer than this get a CTA of their own   */
  int32_t split_row_min; /* rows longer than this are split across CTAs    */
  int32_t split_chunk;   /* nonzeros per chunk of a split row              */
  int32_t x_smem;        /* -1 auto, 0 never, 1 whenever x fits: stage x in
                            shared memory once per CTA                     */
  int32_t reduce;        /* short-row tiles: 0 auto (per tile, by a cost
                            model of its row lengths), 1 lanes mode (rows
                            summed by `lanes` lanes from shared memory),
                            2 walk mode (per-thread segmented sums)        */
  int32_t lanes;         /* lanes per row in forced lanes mode: 1..256
                            (rounded down to a power of two)               */
  int32_t interleave;    /* CSR order in which threads take a unit's
                            nonzeros for the x gathers: 0 auto, 1 chunks of
                            8 consecutive per thread, 2 element-interleaved
                            (a warp's lanes take consecutive nonzeros)     */
  int32_t sell_sigma;    /* SELL: rows are sorted by decreasing length inside
                            windows of this many rows before slicing; 1 keeps
                            the row order; 0 chooses by the CV of the row
                            lengths as spmv_select_format does             */
  int32_t csr_kernel;    /* CSR: 0 auto (warp segments when rows average at
                            least 256 nonzeros; else mixed warp segments
                            when the CV of the row lengths exceeds 2; else
                            CTA tiles), 1 CTA tiles
                            (the bins above), 2 warp segments (rows cut into
                            slices of at most 512 nonzeros, each warp a
                            contiguous share; [CSR] 4.1 warp per row),
                            3 mixed warp segments (runs of whole rows packed
                            256 nonzeros to a segment, [SPGEMM] 5.2;
                            longer rows in slices of 256)                  */
  int32_t delta_kernel;  /* DELTA decode ([MACKO] 2.2): 0 auto (several
                            lanes per word for 4-bit deltas, and for 2-bit
                            deltas unless more than 18% of the stored
                            entries are +0.0 padding), 1 a lane per packed
                            word, 2 several lanes per word (2- and 4-bit
                            deltas: 4 lanes per word for 4-bit, 8 for 2-bit,
                            each lane two entries, so a warp's gathers fall
                            in a narrow window of x; 8-bit deltas always
                            take a lane per word)                          */
  int32_t reserved[4];
} spmv_plan_options;

/* What the planner decided; filled by spmv_plan_inspect / spmv_plan_get_info.
 * Row bins ([SPGEMM] section 2.1.1, adapted to nonzeros per row; a short-row
 * tile hands every thread 8 consecutive nonzeros, so the bin says how many
 * threads cooperate on a row):
 *   0 sub-warp: <= 8 nonzeros (1-2 threads)
 *   1 warp:     9..256 nonzeros (up to 33 threads)
 *   2 CTA:      257..split_row_min nonzeros (up to the whole CTA)
 *   3 split:    longer rows, cut into chunks across CTAs
 * tiles_per_bin: [0] short-row tiles (any mix of bins 0-2), [1] unused,
 * [2] single-row tiles, [3] split chunks. */
typedef struct spmv_plan_info {
  int32_t n_rows;
  int32_t n_cols;
  int64_t nnz;
  int32_t format;
  int32_t value_dtype;
  int64_t n_entries;         /* stored entries (== nnz for CSR)            */
  int64_t n_tiles;           /* work units of one run                      */
  int64_t rows_per_bin[4];
  int64_t tiles_per_bin[4];
  int64_t n_split_rows;
  int32_t x_in_smem;         /* 1 when x is staged in shared memory        */
  int32_t grid;              /* CTAs of the main launch                    */
  int32_t block;             /* threads per CTA                            */
  int32_t launches_per_run;  /* kernel launches issued by one spmv_run     */
  int64_t matrix_bytes;      /* stored matrix: values + indices + row ptrs */
  int64_t aux_bytes;         /* planner tables and scratch on the device   */
  int64_t algorithmic_bytes; /* matrix_bytes + x read once + y written     */
  int64_t walk_tiles;        /* short-row tiles reduced in walk mode       */
  int64_t interleaved;       /* 1 if products are taken element-interleaved */
  int64_t segments;          /* 1 if the plan runs warp-owned row segments
                                (DELTA; CSR with long or irregular rows);
                                n_tiles then counts segments               */
  int64_t reserved[5];
} spmv_plan_info;

typedef struct spmv_plan spmv_plan;

/* Short English text for a status code (static storage). The pages have no
 * counterpart: status codes replace the exceptions and aborts of their
 * snippets. */
const char* spmv_status_string(spmv_status status);

/* Returns SPMV_ABI_VERSION of the built library. */
int32_t spmv_abi_version(void);

/* Fill *opts with "library default" in every field (sizes 0, x_smem -1,
 * reduce 0). The defaults themselves depend on the matrix's value type and
 * are chosen when the plan is made: a stage holds 2048 nonzeros (fp32 or
 * fp16), short-row tiles take up to 16 fewer, rows above half of that get
 * a tile of their own, and split chunks take up to a full stage. */
void spmv_plan_options_init(spmv_plan_options* opts);

/* [MACKO] section 2.1: convert a CSR matrix with fp16 values into DELTA4
 * on the host. The library allocates out->values, out->words and
 * out->row_ptr with malloc; release them with spmv_delta_free. On error
 * *out is left zeroed. Errors: INVALID_ARG, BAD_ROW_PTR, COL_OUT_OF_RANGE,
 * UNSORTED_OR_DUPLICATE_COLS, UNSUPPORTED (fp32 values), OUT_OF_MEMORY. */
spmv_status spmv_convert(const spmv_csr* csr, spmv_delta* out);

/* As spmv_convert, with deltas of `bits` bits (2, 4 or 8; anything else:
 * INVALID_ARG). */
spmv_status spmv_convert_bits(const spmv_csr* csr, int32_t bits, spmv_delta* out);

/* Pick a delta width (2, 4 or 8) for a CSR matrix with fp16 values under
 * `policy`. entries, if not NULL, receives the number of entries the
 * encoding would store at 2, 4 and 8 bits (padding included), counted
 * exactly without building it. Errors: as spmv_convert, and INVALID_ARG for
 * a NULL bits or an unknown policy. */
spmv_status spmv_delta_select_bits(const spmv_csr* csr, spmv_delta_policy policy,
                                   int32_t* bits, int64_t entries[3]);

/* [CSR] section 2.1, ELL in slices: lay a CSR matrix (fp32 or fp16 values;
 * any column order, repeats allowed) out as spmv_sell with sorting window
 * sigma >= 1. The library allocates the arrays with malloc; release them
 * with spmv_sell_free. On error *out is left zeroed. Errors: INVALID_ARG
 * (sigma < 1), BAD_ROW_PTR, COL_OUT_OF_RANGE, TOO_LARGE (more than 2^31 - 1
 * slots), OUT_OF_MEMORY. */
spmv_status spmv_convert_sell(const spmv_csr* csr, int32_t sigma, spmv_sell* out);

/* Free the arrays of a spmv_sell filled by spmv_convert_sell and zero it. */
void spmv_sell_free(spmv_sell* s);

/* [CSR] section 2.2: choose a format by the coefficient of variation of the
 * row lengths, CV = (population standard deviation) / mean (0 when the mean
 * is 0): CV < 0.3 -> SELL with sigma 1 (ELL); 0.3 <= CV <= 0.7 -> SELL with
 * sigma 1024 (rows sorted by length in windows: the page's hybrid ELL + COO
 * band, served by sorted slices); CV > 0.7 -> CSR (sigma 0). Any output
 * pointer may be NULL. Errors: INVALID_ARG, BAD_ROW_PTR. */
spmv_status spmv_select_format(const spmv_csr* csr, spmv_format* format, int32_t* sigma,
                               double* cv);

/* Free the arrays of a spmv_delta filled by spmv_convert and zero it. */
void spmv_delta_free(spmv_delta* d);

/* Host-only dry run of the planner: validates csr exactly as
 * spmv_plan_create does and reports the bins and tiles it would build,
 * without touching any CUDA device (device-dependent fields -- grid,
 * x_in_smem -- assume a 152-SM device). opts may be NULL. */
spmv_status spmv_plan_inspect(const spmv_csr* csr, spmv_format format,
                              const spmv_plan_options* opts,
                              spmv_plan_info* info);

/* Build a plan on the current CUDA device ([CSR] section 2.2): validate,
 * convert (DELTA, SELL), bin the rows, then copy the matrix and the planner's
 * tables into device memory owned by the plan. The caller may free its host
 * arrays as soon as this returns. Synchronous. On error *out is NULL. */
spmv_status spmv_plan_create(const spmv_csr* csr, spmv_format format,
                             spmv_plan** out);

/* As spmv_plan_create, with planner options (opts may be NULL). */
spmv_status spmv_plan_create_ex(const spmv_csr* csr, spmv_format format,
                                const spmv_plan_options* opts,
                                spmv_plan** out);

/* Build a column-delta plan directly from an already converted matrix (for
 * weights converted once ahead of time), at its delta_bits. Every stored
 * entry's decoded column must be < n_cols and row_ptr entries must be
 * multiples of 32 / delta_bits. */
spmv_status spmv_plan_create_delta(const spmv_delta* delta,
                                   const spmv_plan_options* opts,
                                   spmv_plan** out);

/* A structured hexahedral mesh for the matrix-free operator ([FEM] 2.1,
 * 5.2), in HOST memory. nex x ney x nez elements; element
 * e = ex + nex*(ey + ney*ez); node (i, j, k) = i + (nex+1)*(j + (ney+1)*k);
 * dof = 3*node + c (n = 3 * (nex+1)(ney+1)(nez+1) dofs). Element e's local
 * node b is at (ex, ey, ez) + corner b, corners in the order (0,0,0),
 * (1,0,0), (1,1,0), (0,1,0), (0,0,1), (1,0,1), (1,1,1), (0,1,1); local dof
 * 3*b + c. The element's matrix is rho[e] * K0. */
typedef struct spmv_fem_mesh {
  int32_t nex;
  int32_t ney;
  int32_t nez;
  int32_t reserved;
  const float* rho;  /* nex*ney*nez element densities (finite)             */
  const float* K0;   /* 24*24 element matrix, row-major (finite)           */
} spmv_fem_mesh;

/* Plan y = K x for K = sum_e P_e^T (rho_e K0) P_e without assembling K:
 * the plan copies rho to the device and K0 into itself. x and y are fp32,
 * n elements each; runs are deterministic (no atomics). info.nnz reports the
 * stored entries K would have if assembled. Errors: INVALID_ARG (a size < 1,
 * NULL arrays, non-finite values), TOO_LARGE (n > 2^31 - 4097), CUDA,
 * OUT_OF_MEMORY. */
spmv_status spmv_plan_create_fem(const spmv_fem_mesh* mesh, spmv_plan** out);

/* Outcome of spmv_pcg_solve. */
typedef struct spmv_pcg_result {
  int32_t iterations;    /* iterations taken                                */
  int32_t status;        /* 1 converged, 2 iteration limit reached,
                            3 breakdown (p . A p <= 0: A not SPD)           */
  double rel_residual;   /* ||r|| / ||b|| of the recurrence's residual      */
} spmv_pcg_result;

/* Jacobi-preconditioned conjugate gradients for A x = b ([FEM] 6.1), A the
 * square fp32 plan's operator (CSR, SELL or FEM; symmetric positive
 * definite), preconditioner the diagonal of A (diag_dev, n fp32 on the
 * device, or NULL for the plan's own diagonal; a zero entry leaves its row
 * unscaled). x_dev holds the initial guess and receives the solution; b_dev
 * is not written. Stops when ||r|| <= rel_tol ||b|| or after max_iter
 * iterations. Each iteration is the plan's product and two or three vector
 * kernels on `stream`. The iterations run as one CUDA graph with a
 * device-side loop (two iterations per pass; the direction kernel ends the
 * loop on convergence, the limit or a breakdown), kept in the plan for the
 * same b, x and diag, so the host waits once per solve. When `stream` is
 * the legacy default stream or is being captured, or the graph cannot be
 * built, the host runs batches of 4, then 8, then check_every (<= 0: 16)
 * iterations instead and checks the device-side state between them;
 * kernels after convergence inside a batch do nothing. The call
 * synchronizes the stream. Vectors are fp32 and the recurrence's scalars
 * fp64; the result is the same bits on every run.
 * Errors: INVALID_ARG (NULL pointers, non-square or non-fp32 plan, no
 * diagonal), OUT_OF_MEMORY, CUDA. */
spmv_status spmv_pcg_solve(spmv_plan* plan, const float* diag_dev, const float* b_dev,
                           float* x_dev, double rel_tol, int32_t max_iter, int32_t check_every,
                           void* stream, spmv_pcg_result* result);

/* Copy the plan's planner report into *info. */
spmv_status spmv_plan_get_info(const spmv_plan* plan, spmv_plan_info* info);

/* y = A x, asynchronously on `stream` (a cudaStream_t; NULL = legacy
 * default stream): the launch step of [CSR] 2.2 (the matrix is already
 * resident, so only kernels chosen by the plan's format run). x_dev: n_cols
 * elements (fp32 for fp32-value plans, fp16 otherwise), aligned to its
 * element size; y_dev: n_rows fp32, aligned to 4 bytes, fully overwritten
 * (rows without nonzeros get 0). x and y must not overlap. DELTA, SELL and
 * FEM plans multiply padding (or out-of-mesh) entries as 0 * x[c], so x
 * must be finite there (DELTA plans whose entries are more than 18% +0.0
 * skip those products altogether). Does not synchronize. Errors:
 * INVALID_ARG, WRONG_DEVICE, CUDA (launch failure). */
spmv_status spmv_run(spmv_plan* plan, const void* x_dev, float* y_dev,
                     void* stream);

/* End-to-end variant with HOST buffers: copies x_host (n_cols elements of
 * the plan's x type) into a plan-owned device buffer, runs y = A x, copies
 * y back into y_host (n_rows fp32) and synchronizes `stream`: the copy-in,
 * launch and copy-out of [CSR] 2.2 for the vectors. Pinned host memory gives
 * the fastest copies. Errors: INVALID_ARG (null buffer), WRONG_DEVICE,
 * CUDA. */
spmv_status spmv_run_host(spmv_plan* plan, const void* x_host, float* y_host,
                          void* stream);

/* The end-to-end product of `count` independent vectors with HOST buffers:
 * y_host[i*n_rows ..] = A x_host[i*n_cols ..] for i < count (x: the plan's x
 * type, y: fp32, both contiguous, vector after vector). The copy-in of one
 * vector, the product of the one before it and the copy-out of the one
 * before that run at the same time (two plan-owned staging pairs, the
 * products on `stream`, the copies on two streams of the plan's own, ordered
 * by events); returns after the last y is in host memory. Pinned host
 * memory gives the fastest copies and lets the copies overlap. The call
 * synchronizes, so it cannot be captured into a CUDA graph. The copy-in /
 * launch / copy-out of [CSR] 2.2, pipelined over a batch. Errors:
 * INVALID_ARG (count < 0, null buffer), WRONG_DEVICE, OUT_OF_MEMORY (the
 * second staging pair, first call only), CUDA. */
spmv_status spmv_run_host_batch(spmv_plan* plan, int32_t count, const void* x_host,
                                float* y_host, void* stream);

/* Allocation-free y = A x for a CSR matrix the caller already holds in
 * device memory (the pages have no counterpart: this entry point exists for
 * callers that may not allocate device memory -- a latency-critical loop
 * after its set-up phase, where cudaMalloc could synchronise the device; a
 * component inside a memory pool that owns all device memory; a plug-in
 * handed device buffers but no allocator. spmv_plan_create allocates, so
 * those callers cannot use plans).
 * row_ptr (n_rows+1), col_idx (nnz), values (nnz, value_dtype) and x (n_cols,
 * fp32 for SPMV_F32 values, fp16 for SPMV_F16) are caller-owned DEVICE
 * arrays on the current device and must form a valid CSR matrix (row_ptr
 * non-decreasing from 0 to nnz, columns in [0, n_cols)); their contents
 * are not validated, but each pointer is checked (cudaPointerGetAttributes,
 * which allocates nothing) to be device or managed memory of the current
 * device. Alignment: col_idx 16 bytes, values 16 (fp32) or 8 (fp16)
 * bytes, row_ptr and y 4 bytes. y (n_rows fp32) is overwritten. Runs two
 * kernels on `stream`; calls no allocating routine.
 * Scratch: a file-scope device array of 768 KiB (and a status word) per
 * device, shared by all
 * calls and held until the process exits; calls that overlap on the GPU
 * race on it, so order them (one stream). The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress); make that first call
 * before any stream capture.
 * Errors: INVALID_ARG (negative sizes, null or misaligned pointers, an
 * array that is not on the current device), TOO_LARGE (nnz > 134,217,728,
 * the scratch limit), CUDA. */
spmv_status spmv_csr_run_noalloc(int32_t n_rows, int32_t n_cols, int64_t nnz,
                                 const int32_t* row_ptr,
                                 const int32_t* col_idx, const void* values,
                                 spmv_dtype value_dtype, const void* x,
                                 float* y, void* stream);

/* Synchronize the plan's device and read its device status word: OK, or
 * DEVICE_STATUS if a kernel reported an error since the last check (the
 * word is cleared by this call). In a checked build (below) a column index
 * or row offset found out of range also sets it. */
spmv_status spmv_plan_check(spmv_plan* plan);

/* 1 if this library was built with SPMV_CHECKED=1, else 0. A checked build
 * (a separate build of the same sources, for debugging; the pages have no
 * counterpart: it stands in for a memory checker) makes the CSR kernels and
 * spmv_csr_run_noalloc test every column index against n_cols and every row
 * offset against its slice before using it; an index out of range is
 * replaced by a safe one and reported through the status word (no trap, no
 * access outside any buffer; the results are then not meaningful). */
int32_t spmv_checked_build(void);

/* Checked builds: synchronize the current device and read the status word
 * of spmv_csr_run_noalloc (kept in its scratch array): OK, or DEVICE_STATUS
 * if a call found an index out of range since the last check (the word is
 * cleared). Ordinary builds return OK at once. Allocates nothing. */
spmv_status spmv_noalloc_check(void);

/* Release the plan and its device memory (synchronizes the device first):
 * the cudaFree counterpart of [CSR] 2.2's one-time upload. NULL is
 * accepted. */
void spmv_plan_destroy(spmv_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* SPMV_GB300_SPMV_H */
