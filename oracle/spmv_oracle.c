/*
 * Oracle: plain, slow, single-threaded CPU reference for sparse matrix-vector
 * multiply and for the 4-bit column-delta storage format.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load or call this code. The library under
 * test shares nothing with it: no header, no helper, no table.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -shared -fPIC
 * (FMA contraction off so that every product is rounded once to fp64 and
 * every sum is a plain fp64 addition, in index order).
 *
 * Sources followed (by page title and section):
 *  - "CUDA CSR SpMV optimisation" page (codechina.net), section 2.1: the scalar
 *    CSR kernel defines y[row] as the sum over k in [row_ptr[row],
 *    row_ptr[row+1]) of values[k] * x[col_idx[k]].
 *  - "MACKO-SpMV" page (maplevalley.com.cn), section 2.1: the format keeps
 *    values (with zero placeholders), 4-bit column deltas packed eight to a
 *    32-bit word, and CSR-like row pointers; encoding takes deltas between
 *    neighbouring columns (worked example [2,5,12,13] -> [2,3,7,1]), inserts a
 *    zero-valued entry whenever a gap does not fit in 4 bits, packs the
 *    nibbles, and aligns rows.
 * Readings taken where the page is silent or garbled:
 *  - a delta is stored as-is in 4 bits (codes 0..15); a gap of 16 or more
 *    first emits padding entries of value +0.0 and delta 15 until the rest
 *    fits (the only reading that reproduces the worked example);
 *  - the running column restarts at 0 at the start of every row;
 *  - entry e of the whole stream puts its nibble at bits 4*(e%8)..4*(e%8)+3
 *    of word e/8 (little-nibble-first);
 *  - row alignment: every row is padded with (+0.0, delta 0) entries to a
 *    multiple of 8 entries, so each row starts on a word boundary;
 *  - decoding drops every entry whose value bits are exactly 0x0000 (+0.0),
 *    since padding and a stored +0.0 cannot be told apart.
 */
#include <stdint.h>
#include <stddef.h>

#define DELTA_BITS 4
#define DELTA_MAX 15 /* largest code a 4-bit field holds */
#define ROW_ALIGN 8  /* entries per 32-bit word of nibbles */

/* y = A x and s = |A| |x| (elementwise products), fp64, in stored order.
 * Returns 0. Indices are trusted (tests build valid inputs). */
int oracle_csr_spmv(int64_t n_rows, const int64_t *row_ptr,
                    const int64_t *col_idx, const double *values,
                    const double *x, double *y, double *s) {
  for (int64_t i = 0; i < n_rows; ++i) {
    double acc = 0.0;
    double abs_acc = 0.0;
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
      double prod = values[k] * x[col_idx[k]];
      acc = acc + prod;
      abs_acc = abs_acc + (prod < 0.0 ? -prod : prod);
    }
    y[i] = acc;
    if (s) s[i] = abs_acc;
  }
  return 0;
}

/* Pass 1 of the encoder: number of stored entries per row.
 * out_row_ptr[n_rows+1] receives entry offsets. Returns 0, or -1 when a row's
 * columns are negative or not strictly increasing (the delta format needs
 * sorted, distinct columns). */
int oracle_delta_count(int64_t n_rows, const int64_t *row_ptr,
                       const int64_t *col_idx, int64_t *out_row_ptr,
                       int64_t *gap_pads, int64_t *align_pads) {
  int64_t total = 0, gaps = 0, aligns = 0;
  out_row_ptr[0] = 0;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t count = 0;
    int64_t prev = 0;
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
      int64_t c = col_idx[k];
      if (c < 0) return -1;
      if (k > row_ptr[i] && c <= col_idx[k - 1]) return -1;
      int64_t d = c - prev;
      while (d > DELTA_MAX) {
        count += 1; /* padding entry */
        gaps += 1;
        prev += DELTA_MAX;
        d -= DELTA_MAX;
      }
      count += 1; /* the nonzero itself */
      prev = c;
    }
    while (count % ROW_ALIGN != 0) {
      count += 1;
      aligns += 1;
    }
    total += count;
    out_row_ptr[i + 1] = total;
  }
  if (gap_pads) *gap_pads = gaps;
  if (align_pads) *align_pads = aligns;
  return 0;
}

static void put_entry(uint16_t *out_values, uint32_t *out_words, int64_t e,
                      uint16_t value_bits, uint32_t delta) {
  out_values[e] = value_bits;
  uint32_t shift = (uint32_t)(DELTA_BITS * (e % ROW_ALIGN));
  out_words[e / ROW_ALIGN] |= (delta & 0xFu) << shift;
}

/* Pass 2 of the encoder. out_row_ptr comes from oracle_delta_count; out_words
 * must be zero-filled by the caller (n_entries/8 words). value_bits are the
 * fp16 bit patterns of the CSR values. */
int oracle_delta_fill(int64_t n_rows, const int64_t *row_ptr,
                      const int64_t *col_idx, const uint16_t *value_bits,
                      const int64_t *out_row_ptr, uint16_t *out_values,
                      uint32_t *out_words) {
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t e = out_row_ptr[i];
    int64_t prev = 0;
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
      int64_t c = col_idx[k];
      int64_t d = c - prev;
      while (d > DELTA_MAX) {
        put_entry(out_values, out_words, e, 0x0000u, DELTA_MAX);
        e += 1;
        prev += DELTA_MAX;
        d -= DELTA_MAX;
      }
      put_entry(out_values, out_words, e, value_bits[k], (uint32_t)d);
      e += 1;
      prev = c;
    }
    while (e < out_row_ptr[i + 1]) {
      put_entry(out_values, out_words, e, 0x0000u, 0u);
      e += 1;
    }
  }
  return 0;
}

/* Decoder: walks each row's entries keeping the running column, drops entries
 * whose value bits are 0x0000. out_col/out_vals need room for n_entries;
 * out_row_ptr[n_rows+1] receives CSR offsets. Returns the number of kept
 * entries. */
int64_t oracle_delta_decode(int64_t n_rows, const int64_t *entry_row_ptr,
                            const uint16_t *values, const uint32_t *words,
                            int64_t *out_row_ptr, int64_t *out_col,
                            uint16_t *out_vals) {
  int64_t kept = 0;
  out_row_ptr[0] = 0;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t col = 0;
    for (int64_t e = entry_row_ptr[i]; e < entry_row_ptr[i + 1]; ++e) {
      uint32_t shift = (uint32_t)(DELTA_BITS * (e % ROW_ALIGN));
      uint32_t d = (words[e / ROW_ALIGN] >> shift) & 0xFu;
      col += (int64_t)d;
      if (values[e] != 0x0000u) {
        out_col[kept] = col;
        out_vals[kept] = values[e];
        kept += 1;
      }
    }
    out_row_ptr[i + 1] = kept;
  }
  return kept;
}
