/*
 * Oracle: plain, slow, single-threaded CPU reference for sparse matrix-vector
 * multiply and for the column-delta storage format (4-bit deltas, and the
 * 2- and 8-bit widths).
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
 *    fits (the only reading that reproduces the worked example); a width of
 *    b bits stores codes 0..2^b-1 and pads with delta 2^b-1 the same way;
 *  - the running column restarts at 0 at the start of every row;
 *  - entry e of the whole stream puts its nibble at bits 4*(e%8)..4*(e%8)+3
 *    of word e/8 (little-nibble-first); a b-bit field of entry e sits at bits
 *    b*(e%(32/b)) of word e/(32/b);
 *  - row alignment: every row is padded with (+0.0, delta 0) entries to a
 *    multiple of 8 entries (32/b for width b), so each row starts on a word
 *    boundary;
 *  - decoding drops every entry whose value bits are exactly 0x0000 (+0.0),
 *    since padding and a stored +0.0 cannot be told apart.
 */
#include <stdint.h>
#include <stddef.h>

/* Field width of the deltas: 4 bits ("MACKO-SpMV" 2.1) unless a caller of
 * the *_bits entry points asks for 2 or 8 ("MACKO-SpMV" 3.3 lists the
 * widths); a word of 32 bits then holds 32 / bits deltas, and rows are
 * aligned to whole words. */
#define DELTA_BITS 4

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

/* Pass 1 of the encoder: number of stored entries per row, for deltas of
 * `bits` bits (2, 4 or 8). out_row_ptr[n_rows+1] receives entry offsets.
 * Returns 0, -1 when a row's columns are negative or not strictly increasing
 * (the delta format needs sorted, distinct columns), or -2 for another
 * width. */
int oracle_delta_count_bits(int64_t n_rows, const int64_t *row_ptr,
                            const int64_t *col_idx, int bits, int64_t *out_row_ptr,
                            int64_t *gap_pads, int64_t *align_pads) {
  if (bits != 2 && bits != 4 && bits != 8) return -2;
  const int64_t dmax = ((int64_t)1 << bits) - 1; /* largest code a field holds */
  const int64_t per_word = 32 / bits;             /* fields per 32-bit word */
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
      while (d > dmax) {
        count += 1; /* padding entry */
        gaps += 1;
        prev += dmax;
        d -= dmax;
      }
      count += 1; /* the nonzero itself */
      prev = c;
    }
    while (count % per_word != 0) {
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

int oracle_delta_count(int64_t n_rows, const int64_t *row_ptr, const int64_t *col_idx,
                       int64_t *out_row_ptr, int64_t *gap_pads, int64_t *align_pads) {
  return oracle_delta_count_bits(n_rows, row_ptr, col_idx, DELTA_BITS, out_row_ptr, gap_pads,
                                 align_pads);
}

static void put_entry(uint16_t *out_values, uint32_t *out_words, int64_t e, int bits,
                      uint16_t value_bits, uint32_t delta) {
  const int64_t per_word = 32 / bits;
  out_values[e] = value_bits;
  uint32_t shift = (uint32_t)(bits * (e % per_word));
  out_words[e / per_word] |= (delta & ((1u << bits) - 1u)) << shift;
}

/* Pass 2 of the encoder. out_row_ptr comes from oracle_delta_count_bits with
 * the same width; out_words must be zero-filled by the caller
 * (n_entries * bits / 32 words). value_bits are the fp16 bit patterns of the
 * CSR values. */
int oracle_delta_fill_bits(int64_t n_rows, const int64_t *row_ptr, const int64_t *col_idx,
                           const uint16_t *value_bits, int bits, const int64_t *out_row_ptr,
                           uint16_t *out_values, uint32_t *out_words) {
  if (bits != 2 && bits != 4 && bits != 8) return -2;
  const int64_t dmax = ((int64_t)1 << bits) - 1;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t e = out_row_ptr[i];
    int64_t prev = 0;
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
      int64_t c = col_idx[k];
      int64_t d = c - prev;
      while (d > dmax) {
        put_entry(out_values, out_words, e, bits, 0x0000u, (uint32_t)dmax);
        e += 1;
        prev += dmax;
        d -= dmax;
      }
      put_entry(out_values, out_words, e, bits, value_bits[k], (uint32_t)d);
      e += 1;
      prev = c;
    }
    while (e < out_row_ptr[i + 1]) {
      put_entry(out_values, out_words, e, bits, 0x0000u, 0u);
      e += 1;
    }
  }
  return 0;
}

int oracle_delta_fill(int64_t n_rows, const int64_t *row_ptr, const int64_t *col_idx,
                      const uint16_t *value_bits, const int64_t *out_row_ptr,
                      uint16_t *out_values, uint32_t *out_words) {
  return oracle_delta_fill_bits(n_rows, row_ptr, col_idx, value_bits, DELTA_BITS, out_row_ptr,
                                out_values, out_words);
}

/* Decoder for deltas of `bits` bits: walks each row's entries keeping the
 * running column, drops entries whose value bits are 0x0000. out_col /
 * out_vals need room for n_entries; out_row_ptr[n_rows+1] receives CSR
 * offsets. Returns the number of kept entries. */
int64_t oracle_delta_decode_bits(int64_t n_rows, const int64_t *entry_row_ptr,
                                 const uint16_t *values, const uint32_t *words, int bits,
                                 int64_t *out_row_ptr, int64_t *out_col, uint16_t *out_vals) {
  const int64_t per_word = 32 / bits;
  const uint32_t mask = (1u << bits) - 1u;
  int64_t kept = 0;
  out_row_ptr[0] = 0;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t col = 0;
    for (int64_t e = entry_row_ptr[i]; e < entry_row_ptr[i + 1]; ++e) {
      uint32_t shift = (uint32_t)(bits * (e % per_word));
      uint32_t d = (words[e / per_word] >> shift) & mask;
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

int64_t oracle_delta_decode(int64_t n_rows, const int64_t *entry_row_ptr,
                            const uint16_t *values, const uint32_t *words,
                            int64_t *out_row_ptr, int64_t *out_col, uint16_t *out_vals) {
  return oracle_delta_decode_bits(n_rows, entry_row_ptr, values, words, DELTA_BITS,
                                  out_row_ptr, out_col, out_vals);
}
