/*
 * All-core CPU baseline: the oracle's CSR loop and its column-delta walk,
 * with the rows shared out over OpenMP threads. Each row is still summed by
 * one thread in fp64, in stored order, exactly as the single-threaded oracle
 * does, so the results are the oracle's bit for bit.
 *
 * TEST AND BENCHMARK INFRASTRUCTURE ONLY. It is timed beside the GPU path as
 * a second reported CPU baseline (the benchmark's cpu_baseline leg); it is
 * not the parity oracle (that is spmv_oracle.c, single-threaded), and the
 * library under test shares nothing with it.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -shared -fPIC
 *
 * Sources followed (by page title and section):
 *  - "CUDA CSR SpMV optimisation" page, section 2.1: y[row] is the sum over
 *    k in [row_ptr[row], row_ptr[row+1]) of values[k] * x[col_idx[k]];
 *    section 1 contrasts a CPU and a GPU run of this product.
 *  - "MACKO-SpMV" page, section 2.1: the column-delta format (deltas of
 *    `bits` bits, 32 / bits to a 32-bit word, little field first, the running
 *    column restarting at 0 in every row); entries whose value bits are
 *    +0.0 are padding and are skipped.
 */
#include <omp.h>
#include <stdint.h>

/* Threads the parallel loops use. */
int omp_baseline_threads(void) { return omp_get_max_threads(); }

/* y = A x in fp64 for a CSR matrix (fp64 values and x), rows in parallel. */
int omp_csr_spmv(int64_t n_rows, const int64_t *row_ptr, const int64_t *col_idx,
                 const double *values, const double *x, double *y) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_rows; ++i) {
    double acc = 0.0;
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) acc = acc + values[k] * x[col_idx[k]];
    y[i] = acc;
  }
  return 0;
}

/* y = A x in fp64 for a matrix in the column-delta format: each row walks
 * its entries keeping the running column (value bits are fp16, widened
 * exactly through the table `half_to_double` of 65536 entries). */
int omp_delta_spmv(int64_t n_rows, const int64_t *entry_row_ptr, const uint16_t *values,
                   const uint32_t *words, int bits, const double *half_to_double,
                   const double *x, double *y) {
  if (bits != 2 && bits != 4 && bits != 8) return -2;
  const int64_t per_word = 32 / bits;
  const uint32_t mask = (1u << bits) - 1u;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_rows; ++i) {
    double acc = 0.0;
    int64_t col = 0;
    for (int64_t e = entry_row_ptr[i]; e < entry_row_ptr[i + 1]; ++e) {
      const uint32_t shift = (uint32_t)(bits * (e % per_word));
      col += (int64_t)((words[e / per_word] >> shift) & mask);
      if (values[e] != 0x0000u) acc = acc + half_to_double[values[e]] * x[col];
    }
    y[i] = acc;
  }
  return 0;
}
