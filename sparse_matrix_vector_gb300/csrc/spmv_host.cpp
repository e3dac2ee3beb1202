// Host half of the library: argument validation, the DELTA converter, the
// row-binning planner, plan lifetime and the run entry points.
//
// Sources (web pages, by title and section):
//   "CUDA CSR SpMV optimisation" (codechina.net), 2.1: CSR arrays and the
//     row sum that defines y; 2.2: upload once, then launch by format.
//   "MACKO-SpMV" (maplevalley.com.cn), 2.1: delta coding, zero padding for
//     gaps that do not fit the delta field, the fields packed into 32-bit
//     words, row alignment; the 2-, 4- and 8-bit field widths; 3.3:
//     splitting long rows ("dynamic scheduling").
//   "Hash-based multi-phase SpGEMM" (mlqm.cn), 2.1.1 and 2.2: rows grouped by
//     work into bins handled by partial-warp, warp and block-per-row
//     kernels; 5.2: batching of tiny rows.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <new>

#include "spmv_internal.h"

// The opaque handle of the public header.
struct spmv_plan {
  spmv::Plan impl;
};

namespace spmv {
namespace {

// Device indexing is 32-bit; keep clear of INT32_MAX so that padded spans
// (up to one vector past the end) never overflow.
constexpr int64_t kMaxIndex = (int64_t)INT32_MAX - 4096;
// CSR: x is gathered through L1 by default: staging it in shared memory
// costs a copy per CTA and, for the LLM shapes, a third of the CTAs per SM,
// and was measured slower on GB300 than L1-resident gathers.
constexpr size_t kXsAutoBytes = 0;
// DELTA: the producer / consumer kernel shares one shared-memory copy of x
// among three groups of warps; up to 32 KB of x (16,384 columns) two such
// CTAs still fit an SM, and gathers from shared memory beat L1 there
// (12288-column LLM matrices, 30/50/70/90%: 0.47/0.44/0.40/0.27 of HBM peak
// through L1, 0.47/0.46/0.48/0.30 from shared memory).
constexpr size_t kXsAutoBytesDelta = 32 * 1024;
constexpr size_t kXsMaxBytes = 160 * 1024;   // hard limit when forced
constexpr int kPadElems = 16;                // zero tail after device arrays
constexpr int kAssumedSms = 152;             // for host-only inspection
constexpr size_t kAssumedSmemOptin = 232448; // shared memory a CTA may opt in to (227 KB)

size_t dtype_size(spmv_dtype t) { return t == SPMV_F16 ? 2 : 4; }

bool valid_dtype(int t) { return t == SPMV_F32 || t == SPMV_F16; }
bool is_delta_format(int f) {
  return f == SPMV_FORMAT_DELTA4 || f == SPMV_FORMAT_DELTA2 || f == SPMV_FORMAT_DELTA8 ||
         f == SPMV_FORMAT_DELTA_AUTO;
}
bool valid_format(int f) {
  return f == SPMV_FORMAT_CSR || is_delta_format(f) || f == SPMV_FORMAT_SELL ||
         f == SPMV_FORMAT_AUTO;
}

int32_t format_delta_bits(int f) {
  return f == SPMV_FORMAT_DELTA2 ? 2 : f == SPMV_FORMAT_DELTA8 ? 8 : 4;
}

spmv_format delta_format(int32_t bits) {
  return bits == 2 ? SPMV_FORMAT_DELTA2 : bits == 8 ? SPMV_FORMAT_DELTA8 : SPMV_FORMAT_DELTA4;
}

// Structure checks shared by every entry point that takes a CSR matrix.
spmv_status validate_csr(const spmv_csr* m, bool need_sorted) {
  if (!m) return SPMV_ERR_INVALID_ARG;
  if (m->n_rows < 0 || m->n_cols < 0 || m->nnz < 0) return SPMV_ERR_INVALID_ARG;
  if (!valid_dtype(m->value_dtype)) return SPMV_ERR_INVALID_ARG;
  if (!m->row_ptr) return SPMV_ERR_INVALID_ARG;
  if (m->nnz > 0 && (!m->col_idx || !m->values)) return SPMV_ERR_INVALID_ARG;
  if (m->nnz > kMaxIndex) return SPMV_ERR_TOO_LARGE;
  const int32_t* rp = m->row_ptr;
  if (rp[0] != 0) return SPMV_ERR_BAD_ROW_PTR;
  for (int32_t r = 0; r < m->n_rows; ++r)
    if (rp[r + 1] < rp[r]) return SPMV_ERR_BAD_ROW_PTR;
  if ((int64_t)rp[m->n_rows] != m->nnz) return SPMV_ERR_BAD_ROW_PTR;
  for (int64_t k = 0; k < m->nnz; ++k) {
    int32_t c = m->col_idx[k];
    if (c < 0 || c >= m->n_cols) return SPMV_ERR_COL_OUT_OF_RANGE;
  }
  if (need_sorted) {
    for (int32_t r = 0; r < m->n_rows; ++r)
      for (int32_t k = rp[r] + 1; k < rp[r + 1]; ++k)
        if (m->col_idx[k] <= m->col_idx[k - 1])
          return SPMV_ERR_UNSORTED_OR_DUPLICATE_COLS;
  }
  return SPMV_OK;
}

// ------------------------------------------------------------ DELTA codec
// Deltas of b bits (2, 4 or 8): codes 0..2^b-1, 32/b to a word.
inline bool valid_delta_bits(int32_t b) { return b == 2 || b == 4 || b == 8; }
inline int64_t delta_cap(int32_t b) { return ((int64_t)1 << b) - 1; }
inline int64_t delta_per_word(int32_t b) { return 32 / b; }
inline int32_t delta_bits_of(const spmv_delta* d) { return d->delta_bits ? d->delta_bits : 4; }

// Stored entries of one row (before row alignment) under the encoding of
// the header comment.
int64_t delta_row_entries(const int32_t* cols, int32_t len, int64_t cap, int64_t* gaps) {
  int64_t n = 0, c = 0;
  for (int32_t k = 0; k < len; ++k) {
    int64_t gap = (int64_t)cols[k] - c;
    if (gap > cap) {
      int64_t pads = (gap - 1) / cap;
      n += pads;
      *gaps += pads;
    }
    n += 1;
    c = cols[k];
  }
  return n;
}

inline void emit(uint16_t* vals, uint32_t* words, int64_t e, int32_t b, uint16_t bits,
                 uint32_t code) {
  const int64_t per = delta_per_word(b);
  vals[e] = bits;
  words[e / per] |= code << ((uint32_t)b * (uint32_t)(e % per));
}

// Bytes the format stores: values, packed deltas, row pointers (int32 on
// the device).
inline int64_t delta_matrix_bytes(const spmv_delta& d) {
  const int32_t b = delta_bits_of(&d);
  return d.n_entries * 2 + d.n_entries * b / 8 + ((int64_t)d.n_rows + 1) * 4;
}

// Delta of stored entry e.
inline uint32_t delta_at(const uint32_t* words, int64_t e, int32_t b) {
  const int64_t per = delta_per_word(b);
  return (words[e / per] >> ((uint32_t)b * (uint32_t)(e % per))) & (uint32_t)delta_cap(b);
}

}  // namespace

Options resolve_options(const spmv_plan_options* o, spmv_dtype dtype) {
  Options r;
  const int cap = tile_cap(dtype);
  r.tile_nnz = cap - 16;
  r.tile_rows = kTileRowsCap;
  // a row too long to share a short-row tile with another of its length
  // gets a tile of its own (products summed in registers, no parking)
  r.cta_row_min = (cap - 16) / 2;
  r.split_row_min = cap;
  r.split_chunk = cap;
  r.x_smem = -1;
  r.reduce = -1;
  r.lanes_log2 = 0;
  r.interleave = 0;
  r.sell_sigma = 0;
  r.csr_kernel = 0;
  r.delta_kernel = 0;
  if (o) {
    if (o->csr_kernel >= 1 && o->csr_kernel <= 3) r.csr_kernel = o->csr_kernel;
    if (o->delta_kernel >= 1 && o->delta_kernel <= 2) r.delta_kernel = o->delta_kernel;
    if (o->interleave == 1 || o->interleave == 2) r.interleave = o->interleave;
    if (o->sell_sigma > 0) r.sell_sigma = o->sell_sigma;
    if (o->tile_nnz > 0) r.tile_nnz = std::min(o->tile_nnz, cap - 16);
    if (o->tile_rows > 0) r.tile_rows = std::min(o->tile_rows, kTileRowsCap);
    if (o->cta_row_min > 0) r.cta_row_min = o->cta_row_min;
    if (o->split_row_min > 0) r.split_row_min = o->split_row_min;
    if (o->split_chunk > 0) r.split_chunk = std::min(std::max(o->split_chunk, 64), cap);
    if (o->x_smem >= 0) r.x_smem = o->x_smem ? 1 : 0;
    if (o->reduce == 1) {
      r.reduce = 0;
      int l = 0;
      while ((2 << l) <= std::min(std::max(o->lanes, 1), kThreads)) ++l;
      r.lanes_log2 = l;
    } else if (o->reduce == 2) {
      r.reduce = 1;
    }
  }
  // a row that may sit in a short-row tile must fit one on its own, and a
  // row that is not split must fit one stage
  r.cta_row_min = std::min(r.cta_row_min, r.tile_nnz);
  r.split_row_min = std::min(std::max(r.split_row_min, r.cta_row_min), cap);
  return r;
}

// Reduction of a short-row tile. Lanes mode: products are parked in shared
// memory and each row is summed by g = 2^lg lanes; a warp pays, per pass of
// its rows, the slowest row's ceil(len / g) dependent additions plus lg
// shuffles. Walk mode: every thread sums its own 8 products by row and rows
// that cross threads are finished from per-thread carries; its cost is
// roughly fixed (binary search, walk, carries). Pick the cheaper one.
static int64_t lanes_cost(const int32_t* rp, int r0, int r1, int lg);

// Lanes-mode width for a tile: the g = 2^lg with the cheapest cost.
static uint32_t choose_lanes(const int32_t* rp, int r0, int r1) {
  int best_lg = 0;
  int64_t best = INT64_MAX;
  for (int lg = 0; lg <= 8; ++lg) {
    const int64_t c = lanes_cost(rp, r0, r1, lg);
    if (c < best) {
      best = c;
      best_lg = lg;
    }
  }
  return (uint32_t)best_lg << kLanesShift;
}

static uint32_t choose_reduction(const int32_t* rp, int r0, int r1) {
  const uint32_t lanes = choose_lanes(rp, r0, r1);
  const int64_t best = lanes_cost(rp, r0, r1, (int)(lanes >> kLanesShift));
  const int64_t walk_cost = 600;  // ~cycles: search, walk, carries, extra pass
  return best > walk_cost ? kStreamWalk : lanes;
}

// ~cycles of lanes mode with g = 2^lg: per warp, the sum over its passes of
// the slowest row's dependent additions plus shuffles and loads; the tile
// costs as much as its slowest warp.
static int64_t lanes_cost(const int32_t* rp, int r0, int r1, int lg) {
  const int R = r1 - r0;
  const int g = 1 << lg;
  const int per_pass = kThreads >> lg;
  if (lg > 5) {  // a row per group of g/32 warps, one barrier per pass
    int64_t t = 0;
    for (int p0 = 0; p0 < R; p0 += per_pass) {
      int64_t m = 0;
      for (int q = 0; q < per_pass && p0 + q < R; ++q)
        m = std::max<int64_t>(m, ((int64_t)rp[r0 + p0 + q + 1] - rp[r0 + p0 + q] + g - 1) / g);
      t += 4 * m + 8 * 5 + 40 + 100;
    }
    return t;
  }
  const int per_warp = 32 >> lg;
  int64_t worst = 0;
  for (int w = 0; w < kWarps; ++w) {
    int64_t t = 0;
    for (int p0 = 0; p0 < R; p0 += per_pass) {
      const int rs = p0 + w * per_warp;
      if (rs >= R) break;
      int64_t m = 0;
      for (int q = 0; q < per_warp && rs + q < R; ++q) {
        const int64_t len = rp[r0 + rs + q + 1] - rp[r0 + rs + q];
        m = std::max(m, (len + g - 1) / g);
      }
      t += 4 * m + 8 * lg + 40;
    }
    worst = std::max(worst, t);
  }
  return worst;
}

// Bin of a row by how many threads cooperate on it (nonzeros per row): a
// short-row tile gives every thread 8 consecutive nonzeros, so a row of <= 8
// spans at most 2 threads (sub-warp), <= 256 at most 33 (warp), a longer row
// up to the whole CTA; rows above split_row_min are split across CTAs.
static int row_bin(int64_t len, const Options& o) {
  if (len > o.split_row_min) return 3;
  if (len > 256) return 2;
  if (len > 8) return 1;
  return 0;
}

spmv_status plan_csr_tiles(int n_rows, const int32_t* rp, const Options& o,
                           int max_ctas, CsrTables* out, spmv_plan_info* info) {
  out->tiles.clear();
  out->splits.clear();
  out->cta_first.clear();
  out->n_chunks = 0;
  // Weight of a row: its nonzeros plus one (row pointer, y write). The
  // matrix is cut into G contiguous shares of equal weight, one per CTA
  // (persistent grid), and no short-row or single-row tile crosses a share
  // boundary, so every CTA gets the same amount of work.
  const int64_t total_w = (int64_t)rp[n_rows] + n_rows;
  constexpr int64_t kMinShare = 1024;
  const int G = (int)std::max<int64_t>(
      1, std::min<int64_t>(max_ctas, (total_w + kMinShare - 1) / kMinShare));
  auto boundary = [&](int b) { return (int64_t)((__int128)b * total_w / G); };
  int64_t cum = 0;  // weight of the tiles emitted so far
  int next_b = 1;
  // short-row tiles of a share are sized evenly: the share's weight over the
  // fewest tiles that respect tile_nnz
  int64_t target = 0;
  int64_t share_tiles = 0;  // planned short-row tiles left in this share
  auto share_target = [&]() {
    const int64_t left = (next_b < G ? boundary(next_b) : total_w) - cum;
    const int64_t cap = (int64_t)o.tile_nnz + 64;
    share_tiles = std::max<int64_t>(1, (left + cap - 1) / cap);
    return (left + share_tiles - 1) / share_tiles;
  };
  try {
    out->cta_first.push_back(0);
    target = share_target();
    auto mark = [&]() {
      bool moved = false;
      while (next_b < G && cum >= boundary(next_b)) {
        out->cta_first.push_back((int32_t)out->tiles.size());
        ++next_b;
        moved = true;
      }
      if (moved) target = share_target();
    };
    int r = 0;
    while (r < n_rows) {
      const int64_t len = (int64_t)rp[r + 1] - rp[r];
      if (len > o.split_row_min) {
        // the fewest chunks of at most split_chunk, all of (nearly) equal size
        const int64_t nch = (len + o.split_chunk - 1) / o.split_chunk;
        const int64_t per = (len + nch - 1) / nch;
        const int64_t sid = (int64_t)out->splits.size();
        if (sid > (int64_t)kSplitIdMask || out->n_chunks + nch > kMaxIndex)
          return SPMV_ERR_TOO_LARGE;
        out->splits.push_back({(int32_t)out->n_chunks, (int32_t)nch, rp[r], (int32_t)per});
        for (int64_t k = 0; k < nch; ++k) {
          mark();
          const int64_t b = rp[r] + k * per;
          const int64_t e = std::min<int64_t>(b + per, rp[r + 1]);
          const uint32_t flags = (k == 0 ? kSplitFirst : 0u) | (k == nch - 1 ? kSplitLast : 0u);
          out->tiles.push_back({r, (int32_t)b, (int32_t)e,
                                (int32_t)((kKindSplit << kKindShift) | flags |
                                          (uint32_t)sid)});
          cum += (e - b) + (k == 0 ? 1 : 0);
        }
        out->n_chunks += nch;
        info->rows_per_bin[3] += 1;
        info->tiles_per_bin[3] += nch;
        ++r;
        continue;
      }
      mark();
      if (len > o.cta_row_min) {
        out->tiles.push_back(
            {r, rp[r], rp[r + 1], (int32_t)(kKindRow << kKindShift)});
        info->rows_per_bin[row_bin(len, o)] += 1;
        info->tiles_per_bin[2] += 1;
        cum += len + 1;
        ++r;
        continue;
      }
      const int64_t limit = next_b < G ? boundary(next_b) : INT64_MAX;
      const int r0 = r;
      int64_t nz = 0, w = 0;
      while (r < n_rows && r - r0 < o.tile_rows) {
        const int64_t l = (int64_t)rp[r + 1] - rp[r];
        if (l > o.cta_row_min || nz + l > o.tile_nnz) break;
        // the last planned tile of a share takes whatever is left of it
        // a tile ends once it reaches its share's boundary (the row that
        // crosses it stays in); the last planned tile of a share takes
        // whatever is left of the share
        if (r > r0 && (cum + w >= limit || (share_tiles > 1 && w + l + 1 > target))) break;
        nz += l;
        w += l + 1;
        info->rows_per_bin[row_bin(l, o)] += 1;
        ++r;
      }
      // walk mode gives each thread 8 nonzeros, so larger tiles use lanes mode
      const bool walk_fits = nz <= kStreamTileCap;
      const uint32_t mode = (o.reduce == 1 && walk_fits) ? kStreamWalk
                            : o.reduce != -1 ? ((uint32_t)o.lanes_log2 << kLanesShift)
                            : walk_fits     ? choose_reduction(rp, r0, r)
                                            : choose_lanes(rp, r0, r);
      out->tiles.push_back({r0, rp[r0], rp[r],
                            (int32_t)((kKindStream << kKindShift) | mode | (uint32_t)(r - r0))});
      if (mode & kStreamWalk) info->walk_tiles += 1;
      info->tiles_per_bin[0] += 1;
      cum += w;
      --share_tiles;
    }
    while ((int)out->cta_first.size() <= G) out->cta_first.push_back((int32_t)out->tiles.size());
  } catch (const std::bad_alloc&) {
    return SPMV_ERR_OUT_OF_MEMORY;
  }
  if ((int64_t)out->tiles.size() > kMaxIndex) return SPMV_ERR_TOO_LARGE;
  info->n_tiles = (int64_t)out->tiles.size();
  info->n_split_rows = (int64_t)out->splits.size();
  info->grid = G;
  return SPMV_OK;
}

// Deal out->segs to at most max_warps warps as contiguous shares of equal
// weight, and set up the rows whose segments fall in more than one share: one
// partial per such warp (its piece), combined by the last to arrive. Packed
// segments (whole short rows) are never shared.
// Mark the segments of rows split into exactly two pieces (kSegCtlPair).
// Within each warp's share, move the piece of the row that continues into
// the next share to the front (kSegCtlPieceEnd on its last segment), so that
// a warp hands over both its pieces of shared rows early: a two-piece row's
// exchange then returns long before the warp needs its result at the end of
// the share, and the rows of more pieces are counted (kSegCtlCombine) while
// the warp still has whole rows to stream. The exchange and count used to
// sit at the end of every share, about 2 us before each CTA could exit.
void order_shares(SegTables* out, int n_warps) {
  std::vector<SegDesc>& sg = out->segs;
  for (size_t u = 0; u < sg.size(); ++u)
    if (out->seg_split[u] >= 0 && out->splits[(size_t)out->seg_split[u]].n_chunks == 2)
      sg[u].ctl |= kSegCtlPair;
  auto slice = [&](int64_t u) { return !(sg[(size_t)u].flags & kSegPacked); };
  auto split = [&](int64_t u) { return out->seg_split[(size_t)u] >= 0; };
  for (int g = 0; g < n_warps; ++g) {
    const int64_t a = out->warp_first[g], b = out->warp_first[g + 1];
    if (b - a < 2) continue;
    // the leading piece: a row begun by an earlier warp, segments [a, f]
    int64_t f = -1;
    if (split(a) && !(sg[(size_t)a].flags & kSegFirst)) {
      f = a;
      while (f + 1 < b && slice(f + 1) && sg[(size_t)(f + 1)].row == sg[(size_t)a].row) ++f;
      if (f == b - 1) continue;  // the share is one piece of one row
    }
    // the trailing piece: a row that a later warp finishes, segments [c, b)
    int64_t c = b;
    if (split(b - 1) && !(sg[(size_t)(b - 1)].flags & kSegLast)) {
      c = b - 1;
      while (c - 1 > f && c - 1 >= a && slice(c - 1) &&
             sg[(size_t)(c - 1)].row == sg[(size_t)(b - 1)].row)
        --c;
    }
    if (c < b && c > a) {
      std::rotate(sg.begin() + a, sg.begin() + c, sg.begin() + b);
      std::rotate(out->seg_split.begin() + a, out->seg_split.begin() + c,
                  out->seg_split.begin() + b);
      std::rotate(out->seg_slot.begin() + a, out->seg_slot.begin() + c,
                  out->seg_slot.begin() + b);
      const int64_t moved_end = a + (b - c) - 1;
      sg[(size_t)moved_end].ctl |= kSegCtlPieceEnd;
      sg[(size_t)(f >= 0 ? f + (b - c) : moved_end)].ctl |= kSegCtlCombine;
    } else if (c == b && f >= 0) {
      sg[(size_t)f].ctl |= kSegCtlCombine;
    }
  }
}

spmv_status deal_segments(const std::function<int64_t(const SegDesc&)>& weight, int max_warps,
                          int warps_per_cta, SegTables* out, spmv_plan_info* info) {
  constexpr int64_t kMinShare = 256;  // weight a warp should get at least
  const int64_t n_segs = (int64_t)out->segs.size();
  if (n_segs > kMaxIndex) return SPMV_ERR_TOO_LARGE;
  int64_t total_w = 0;
  for (const SegDesc& sg : out->segs) total_w += weight(sg);
  const int64_t want = std::max<int64_t>(1, (total_w + kMinShare - 1) / kMinShare);
  const int G = (int)std::max<int64_t>(1, std::min<int64_t>({(int64_t)max_warps, want,
                                                              std::max<int64_t>(n_segs, 1)}));
  const int grid = (G + warps_per_cta - 1) / warps_per_cta;
  const int n_warps = grid * warps_per_cta;
  out->warp_first.assign((size_t)n_warps + 1, (int32_t)n_segs);
  out->warp_first[0] = 0;
  {
    int64_t cum = 0;
    int g = 1;
    for (int64_t t = 0; t < n_segs; ++t) {
      while (g < G && cum >= (int64_t)((__int128)g * total_w / G)) out->warp_first[g++] = (int32_t)t;
      cum += weight(out->segs[(size_t)t]);
    }
    while (g < G) out->warp_first[g++] = (int32_t)n_segs;
  }
  out->seg_split.assign((size_t)n_segs, -1);
  out->seg_slot.assign((size_t)n_segs, -1);
  std::vector<int32_t> seg_warp((size_t)n_segs);
  for (int g = 0; g < n_warps; ++g)
    for (int32_t t = out->warp_first[g]; t < out->warp_first[g + 1]; ++t) seg_warp[t] = g;
  for (int64_t t = 0; t < n_segs;) {
    int64_t e = t + 1;
    if (!(out->segs[(size_t)t].flags & kSegPacked))
      while (e < n_segs && !(out->segs[(size_t)e].flags & kSegPacked) &&
             out->segs[(size_t)e].row == out->segs[(size_t)t].row)
        ++e;
    if (seg_warp[t] != seg_warp[e - 1]) {
      int32_t pieces = 0;
      for (int64_t u = t; u < e; ++u) {
        if (u > t && seg_warp[u] != seg_warp[u - 1]) ++pieces;
        out->seg_slot[(size_t)u] = (int32_t)out->n_chunks + pieces;
        out->seg_split[(size_t)u] = (int32_t)out->splits.size();
      }
      ++pieces;
      if (out->n_chunks + pieces > kMaxIndex) return SPMV_ERR_TOO_LARGE;
      out->splits.push_back({(int32_t)out->n_chunks, pieces, 0, 0});
      out->n_chunks += pieces;
    }
    t = e;
  }
  info->n_tiles = n_segs;
  info->n_split_rows = (int64_t)out->splits.size();
  info->grid = grid;
  return SPMV_OK;
}

spmv_status plan_segments(int32_t n_rows, const std::function<int64_t(int32_t)>& row_begin,
                          int64_t cap, int64_t seg_cost, int64_t entries_per_item,
                          int max_warps, int warps_per_cta, SegTables* out,
                          spmv_plan_info* info) {
  *out = SegTables();
  try {
    // cut every row into full segments of `cap` items and one shorter last
    // segment (full segments take the kernels' unpredicated path)
    for (int32_t r = 0; r < n_rows; ++r) {
      const int64_t i0 = row_begin(r), i1 = row_begin(r + 1), ni = i1 - i0;
      if (ni == 0) {
        out->empty_rows.push_back(r);
        info->rows_per_bin[0] += 1;
        continue;
      }
      if (i1 > INT32_MAX) return SPMV_ERR_TOO_LARGE;
      const int64_t n_s = (ni + cap - 1) / cap;
      const int64_t entries = ni * entries_per_item;
      info->rows_per_bin[n_s > 1 ? 3 : entries > 256 ? 2 : entries > 8 ? 1 : 0] += 1;
      for (int64_t k = 0; k < n_s; ++k) {
        const int64_t sb = i0 + k * cap, se = std::min(sb + cap, i1);
        const uint32_t flags = (k == 0 ? kSegFirst : 0u) | (k == n_s - 1 ? kSegLast : 0u);
        out->segs.push_back({r, (int32_t)sb, (int32_t)se, 0, flags});
      }
      (n_s > 1 ? info->tiles_per_bin[3] : info->tiles_per_bin[2]) += n_s;
    }
    return deal_segments([&](const SegDesc& sg) { return (int64_t)(sg.end - sg.begin) + seg_cost; },
                         max_warps, warps_per_cta, out, info);
  } catch (const std::bad_alloc&) {
    return SPMV_ERR_OUT_OF_MEMORY;
  }
}

// Mixed plans pack rows of at most this many nonzeros (longer rows are cut
// into slices of kCsrSegNnzMixed).
#ifndef SPMV_CSR_PACK_MAX
#define SPMV_CSR_PACK_MAX 256
#endif
constexpr int64_t kCsrPackRowMax = SPMV_CSR_PACK_MAX;

spmv_status plan_csr_mixed_segments(const spmv_csr* m, int max_warps, int warps_per_cta,
                                    SegTables* out, spmv_plan_info* info) {
  *out = SegTables();
  const int32_t* rp = m->row_ptr;
  const int64_t cap = kCsrSegNnzMixed;
  const int64_t pack_max = std::min<int64_t>(kCsrPackRowMax, cap);
  try {
    for (int32_t r = 0; r < m->n_rows;) {
      const int64_t len = (int64_t)rp[r + 1] - rp[r];
      if (len > pack_max) {  // a long row: slices of at most cap nonzeros
        const int64_t n_s = (len + cap - 1) / cap;
        info->rows_per_bin[n_s > 1 ? 3 : len > 256 ? 2 : 1] += 1;
        for (int64_t k = 0; k < n_s; ++k) {
          const int64_t sb = rp[r] + k * cap, se = std::min(sb + cap, (int64_t)rp[r + 1]);
          const uint32_t flags = (k == 0 ? kSegFirst : 0u) | (k == n_s - 1 ? kSegLast : 0u);
          out->segs.push_back({r, (int32_t)sb, (int32_t)se, 0, flags});
        }
        (n_s > 1 ? info->tiles_per_bin[3] : info->tiles_per_bin[2]) += n_s;
        ++r;
        continue;
      }
      // a run of whole rows (empty ones included), packed into one segment
      const int32_t r0 = r;
      int64_t nz = 0;
      while (r < m->n_rows && r - r0 < cap) {
        const int64_t l = (int64_t)rp[r + 1] - rp[r];
        if (l > pack_max || nz + l > cap) break;
        nz += l;
        info->rows_per_bin[l > 8 ? 1 : 0] += 1;
        ++r;
      }
      out->segs.push_back({r0, rp[r0], (int32_t)(rp[r0] + nz), r - r0, kSegPacked});
      info->tiles_per_bin[0] += 1;
    }
    // a packed segment's weight counts its rows too (the row sums)
    return deal_segments(
        [](const SegDesc& sg) {
          return (int64_t)(sg.end - sg.begin) + 32 + (sg.flags & kSegPacked ? 2 * sg.base : 0);
        },
        max_warps, warps_per_cta, out, info);
  } catch (const std::bad_alloc&) {
    return SPMV_ERR_OUT_OF_MEMORY;
  }
}

spmv_status plan_delta_segments(const spmv_delta* d, int max_warps, int warps_per_cta,
                                SegTables* out, spmv_plan_info* info) {
  const int64_t* rp = d->row_ptr;
  const int32_t bits = delta_bits_of(d);
  const int64_t per_word = 32 / bits;  // entries per word
  const uint32_t cap = (1u << bits) - 1u;
  // a segment's weight: its words plus a fixed cost (header, scans, copy)
  spmv_status s = plan_segments(
      d->n_rows, [&](int32_t r) { return rp[r] / per_word; }, delta_seg_words(bits), 16,
      per_word, max_warps, warps_per_cta, out, info);
  if (s != SPMV_OK) return s;
  // each segment's starting column: the running column of its row
  int32_t row = -1;
  int64_t col = 0, w = 0;
  for (SegDesc& sg : out->segs) {
    if (sg.row != row) {
      row = sg.row;
      col = 0;
      w = sg.begin;
    }
    for (; w < sg.begin; ++w) {
      const uint32_t word = d->words[w];
      for (int q = 0; q < per_word; ++q) col += (word >> (bits * q)) & cap;
    }
    if (col > INT32_MAX) return SPMV_ERR_TOO_LARGE;
    sg.base = (int32_t)col;
  }
  order_shares(out, (int)out->warp_first.size() - 1);  // after the bases (row order)
  return SPMV_OK;
}

namespace {

// ------------------------------------------------------------ CUDA helpers
struct DeviceGuard {
  int saved = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&saved) != cudaSuccess) return;
    ok = (saved == dev) || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (saved >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != saved)
      cudaSetDevice(saved);
  }
};

template <typename T>
spmv_status dev_alloc(T** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc((void**)p, bytes);
  if (e == cudaErrorMemoryAllocation) {
    cudaGetLastError();
    return SPMV_ERR_OUT_OF_MEMORY;
  }
  return e == cudaSuccess ? SPMV_OK : SPMV_ERR_CUDA;
}

// Allocate bytes_alloc, zero them, copy bytes_copy from host.
template <typename T>
spmv_status dev_upload(T** p, const void* host, size_t bytes_copy,
                       size_t bytes_alloc) {
  spmv_status s = dev_alloc(p, bytes_alloc);
  if (s != SPMV_OK) return s;
  if (cudaMemset(*p, 0, bytes_alloc ? bytes_alloc : 16) != cudaSuccess)
    return SPMV_ERR_CUDA;
  if (bytes_copy &&
      cudaMemcpy(*p, host, bytes_copy, cudaMemcpyHostToDevice) != cudaSuccess)
    return SPMV_ERR_CUDA;
  return SPMV_OK;
}

void free_plan(spmv_plan* plan) {
  if (!plan) return;
  Plan* p = &plan->impl;
  {
    DeviceGuard g(p->device);
    for (void* g : p->pcg_exec)
      if (g) cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(g));
    if (p->pcg_loop) cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(p->pcg_loop));
    for (void* e : p->batch_events)
      if (e) cudaEventDestroy(static_cast<cudaEvent_t>(e));
    for (void* q : p->batch_streams)
      if (q) cudaStreamDestroy(static_cast<cudaStream_t>(q));
    if (p->x_stage2) cudaFree(p->x_stage2);
    if (p->y_stage2) cudaFree(p->y_stage2);
    void* bufs[] = {p->row_ptr, p->col_idx,  p->values,   p->blocks,
                    p->tiles,   p->splits,   p->partials, p->counters, p->cells,
                    p->status,  p->x_stage,  p->y_stage,  p->cta_first,
                    p->row_split, p->perm, p->diag, p->pcg_work,
                    p->seg_off, p->empty_rows};
    for (void* b : bufs)
      if (b) cudaFree(b);
  }
  delete plan;
}

spmv_status bind_device(Plan* p) {
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    cudaGetLastError();
    return SPMV_ERR_CUDA;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount,
                             p->device) != cudaSuccess)
    return SPMV_ERR_CUDA;
  p->sm_count = sms;
  return SPMV_OK;
}

spmv_status common_buffers(Plan* p) {
  const size_t xs = p->dtype == SPMV_F32 ? 4 : 2;
  spmv_status s;
  if ((s = dev_upload(&p->status, nullptr, 0, 16)) != SPMV_OK) return s;
  if ((s = dev_alloc(&p->x_stage, (size_t)p->n_cols * xs + 16)) != SPMV_OK)
    return s;
  if ((s = dev_alloc(&p->y_stage, (size_t)p->n_rows * 4 + 16)) != SPMV_OK)
    return s;
  return SPMV_OK;
}

void fill_bytes(spmv_plan_info* info, size_t x_elem) {
  info->algorithmic_bytes = info->matrix_bytes +
                            (int64_t)info->n_cols * (int64_t)x_elem +
                            (int64_t)info->n_rows * 4;
}

// Shared memory the kernels' CTAs may hold per SM (dynamic + static + the
// runtime's per-CTA reservation) of the 256 KB that L1 and shared memory
// share. The carve-out is chosen in steps (..., 164, 196, 228 KB); above
// 196 KB, L1 is left with 28 KB, too few lines to keep the x gathers' misses
// in flight: random gathers from an L2-resident vector then run at half
// their rate (measured 0.46 against 0.94 per clock per SM), and fp32 CSR at
// 6 CTAs per SM ran 10-25% slower than at 5 on the Laplacian, FEM and
// power-law matrices.
constexpr size_t kSmemBudget = 196 * 1024;

// Order of the x gathers of a CSR matrix. With chunks of 8 consecutive
// nonzeros per thread, neighbouring lanes gather 8 nonzeros apart; where 8
// nonzeros of a row span more than 40 bytes of x, every lane of a warp-wide
// gather then touches its own sector, and taking the nonzeros
// element-interleaved (a warp's lanes on 32 consecutive nonzeros) cuts the
// L1 sectors per gather several-fold at the cost of scalar shared-memory
// accesses. Rows shorter than 32 nonzeros gain nothing: a warp's 32
// consecutive nonzeros then already span several rows. Measured on GB300
// (fraction of HBM peak, chunks / interleaved): FEM 0.716 / 0.769, LLM 70%
// 0.714 / 0.725, LLM 90% 0.504 / 0.533; Laplacian 0.709 / 0.660, LLM 30%
// 0.762 / 0.721, LLM 50% 0.727 / 0.698.
static bool csr_interleave_auto(const spmv_csr* m) {
  const int32_t* rp = m->row_ptr;
  const int32_t* ci = m->col_idx;
  double span = 0.0;  // sum over rows of (last column - first column)
  int64_t gaps = 0;   // sum over rows of (nonzeros - 1)
  const int step = std::max(1, m->n_rows / 4096);  // a sample of rows
  for (int r = 0; r < m->n_rows; r += step) {
    const int64_t len = (int64_t)rp[r + 1] - rp[r];
    if (len < 2) continue;
    int32_t lo = ci[rp[r]], hi = lo;
    for (int64_t k = rp[r]; k < rp[r + 1]; ++k) {
      lo = std::min(lo, ci[k]);
      hi = std::max(hi, ci[k]);
    }
    span += (double)hi - lo;
    gaps += len - 1;
  }
  if (m->n_rows == 0 || gaps == 0) return false;
  const double mean_len = (double)m->nnz / m->n_rows;
  const double span8_bytes = 7.0 * span / (double)gaps * (double)dtype_size(m->value_dtype);
  return mean_len >= 32.0 && span8_bytes >= 40.0;
}

// CSR with warp segments: the auto rule and the plan.
constexpr int64_t kCsrSegMinMeanRow = 256;  // rows averaging this many nonzeros or more

// Irregular row lengths (CV of the row lengths above this) take mixed
// segments: on the power-law matrix (CV 11.9) 28.9 us against 38.3 us for CTA
// tiles; regular short rows keep the tiles (5-point Laplacian 10.9 us against
// 15.2 us, hex-mesh stiffness 84 us against 164 us).
constexpr double kCsrMixedMinCv = 2.0;
double row_length_cv(const spmv_csr* m);

// 1: CTA tiles, 2: warp segments (long rows), 3: mixed segments
int csr_kernel_choice(const spmv_csr* m, const Options& o) {
  if (o.csr_kernel != 0) return o.csr_kernel;
  if (m->n_rows > 0 && m->nnz >= kCsrSegMinMeanRow * (int64_t)m->n_rows) return 2;
  return row_length_cv(m) > kCsrMixedMinCv ? 3 : 1;
}

// Device layout of a CSR segment plan: one block per segment, back to back in
// segment order, each a 32-byte header (SegHeader), for a packed run of short
// rows the rows' starts relative to the segment (int16), the segment's
// columns (padded to 16 bytes) and values (padded to 16 bytes).
spmv_status build_csr_seg_blocks(const spmv_csr* m, const SegTables& t, int stages,
                                 std::vector<uint4>* out, std::vector<int32_t>* seg_off) {
  const int vs = (int)dtype_size(m->value_dtype);
  const size_t n_segs = t.segs.size();
  auto packed_rows = [&](const SegDesc& sg) -> int64_t {
    return (sg.flags & kSegPacked) ? sg.base : 0;
  };
  try {
    seg_off->assign(n_segs + 1, 0);
    int64_t total = 0;  // in 16-byte steps
    for (size_t k = 0; k < n_segs; ++k) {
      (*seg_off)[k] = (int32_t)total;
      total += csr_seg_bytes((int64_t)t.segs[k].end - t.segs[k].begin, packed_rows(t.segs[k]),
                             vs) / 16;
      if (total > INT32_MAX) return SPMV_ERR_TOO_LARGE;
    }
    (*seg_off)[n_segs] = (int32_t)total;
    out->assign((size_t)total, make_uint4(0, 0, 0, 0));
  } catch (const std::bad_alloc&) {
    return SPMV_ERR_OUT_OF_MEMORY;
  }
  std::vector<int32_t> next(n_segs, -1);  // segment staged `stages` later by the same warp
  for (size_t g = 0; g + 1 < t.warp_first.size(); ++g)
    for (int32_t k = t.warp_first[g]; k + stages < t.warp_first[g + 1]; ++k) next[k] = k + stages;
  unsigned char* base = reinterpret_cast<unsigned char*>(out->data());
  const unsigned char* vals = static_cast<const unsigned char*>(m->values);
  for (size_t k = 0; k < n_segs; ++k) {
    const SegDesc& sg = t.segs[k];
    const int64_t nz = (int64_t)sg.end - sg.begin, R = packed_rows(sg);
    unsigned char* b = base + (size_t)(*seg_off)[k] * 16;
    SegHeader h{};
    h.base = (int32_t)R;
    h.row_flags = (uint32_t)sg.row | sg.flags;
    h.n_words = (int32_t)nz;
    h.split = t.seg_split[k];
    h.slot = t.seg_slot[k];
    h.ctl = t.segs[k].ctl;
    if (next[k] >= 0) {
      h.next_off = (*seg_off)[next[k]];
      h.next_bytes = ((*seg_off)[next[k] + 1] - (*seg_off)[next[k]]) * 16;
    }
    std::memcpy(b, &h, sizeof(h));
    unsigned char* p = b + kSegHeaderBytes;
    if (R > 0) {
      int16_t* rs = reinterpret_cast<int16_t*>(p);
      for (int64_t q = 0; q <= R; ++q) rs[q] = (int16_t)(m->row_ptr[sg.row + q] - sg.begin);
      p += delta_pad16((R + 1) * 2);
    }
    std::memcpy(p, m->col_idx + sg.begin, (size_t)nz * 4);
    std::memcpy(p + delta_pad16(nz * 4), vals + (size_t)sg.begin * vs, (size_t)nz * vs);
  }
  return SPMV_OK;
}

spmv_status create_csr_seg_plan(const spmv_csr* m, const Options& o, bool mixed, Plan* p) {
  spmv_plan_info& info = p->info;
  spmv_status s;
  const size_t vs = dtype_size(m->value_dtype);
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device) !=
      cudaSuccess)
    return SPMV_ERR_CUDA;
  const size_t xbytes = ((size_t)m->n_cols * vs + 15) / 16 * 16;
  const size_t rings = csr_seg_rings_bytes(m->value_dtype, mixed);
  const bool fits = rings + xbytes + 4096 <= (size_t)optin;
  p->x_smem = o.x_smem == 0 ? false : o.x_smem == 1 ? fits : (fits && xbytes <= kXsAutoBytesDelta);
  p->dyn_smem = rings + (p->x_smem ? xbytes : 0);
  if (csr_seg_set_smem_limit(p->dyn_smem) != 0) return SPMV_ERR_CUDA;
  const int occ = csr_seg_occupancy(m->value_dtype, p->x_smem, mixed, p->dyn_smem);
  if (occ <= 0) return SPMV_ERR_CUDA;
  const int wpc = csr_seg_warps_per_cta(m->value_dtype, mixed);
  SegTables t;
  s = mixed ? plan_csr_mixed_segments(m, p->sm_count * wpc, wpc, &t, &info)
            : plan_segments(
                  m->n_rows, [&](int32_t r) { return (int64_t)m->row_ptr[r]; }, kCsrSegNnzLong,
                  64, 1, p->sm_count * wpc, wpc, &t, &info);
  if (s != SPMV_OK) return s;
  order_shares(&t, (int)t.warp_first.size() - 1);
  p->csr_mixed = mixed;
  p->csr_segments = true;
  p->grid = info.grid;
  p->n_tiles = (int64_t)t.segs.size();
  std::vector<uint4> blocks;
  std::vector<int32_t> seg_off;
  if ((s = build_csr_seg_blocks(m, t, csr_seg_stages(m->value_dtype), &blocks, &seg_off)) !=
      SPMV_OK)
    return s;
  if ((s = dev_upload(&p->blocks, blocks.data(), blocks.size() * 16, blocks.size() * 16)) !=
      SPMV_OK)
    return s;
  if ((s = dev_upload(&p->seg_off, seg_off.data(), seg_off.size() * 4, seg_off.size() * 4)) !=
      SPMV_OK)
    return s;
  if ((s = dev_upload(&p->cta_first, t.warp_first.data(), t.warp_first.size() * 4,
                      t.warp_first.size() * 4)) != SPMV_OK)
    return s;
  if ((s = dev_upload(&p->empty_rows, t.empty_rows.data(), t.empty_rows.size() * 4,
                      t.empty_rows.size() * 4)) != SPMV_OK)
    return s;
  p->n_empty_rows = (int32_t)t.empty_rows.size();
  if ((s = dev_upload(&p->splits, t.splits.data(), t.splits.size() * sizeof(SplitInfo),
                      t.splits.size() * sizeof(SplitInfo))) != SPMV_OK)
    return s;
  if ((s = dev_upload(&p->partials, nullptr, 0, (size_t)t.n_chunks * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->counters, nullptr, 0, t.splits.size() * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->cells, nullptr, 0, t.splits.size() * 8)) != SPMV_OK) return s;
  if ((s = common_buffers(p)) != SPMV_OK) return s;
  info.x_in_smem = p->x_smem ? 1 : 0;
  info.block = wpc * 32;
  info.segments = 1;
  info.launches_per_run = m->n_rows > 0 ? 1 : 0;
  info.matrix_bytes = (int64_t)m->nnz * (int64_t)(vs + 4) + ((int64_t)m->n_rows + 1) * 4;
  // the blocks hold the columns and values plus headers and padding; the
  // row pointers are not kept on the device
  info.aux_bytes = (int64_t)(blocks.size() * 16) - (int64_t)m->nnz * (int64_t)(vs + 4) +
                   (int64_t)(seg_off.size() * 4 + t.warp_first.size() * 4 +
                             t.empty_rows.size() * 4 + t.splits.size() * (sizeof(SplitInfo) + 4) +
                             (size_t)t.n_chunks * 4);
  fill_bytes(&info, vs);
  return SPMV_OK;
}

spmv_status create_csr_plan(const spmv_csr* m, const Options& o, Plan* p) {
  CsrTables t;
  spmv_plan_info& info = p->info;
  spmv_status s;
  if ((s = bind_device(p)) != SPMV_OK) return s;
  const int kernel = csr_kernel_choice(m, o);
  if (kernel >= 2) return create_csr_seg_plan(m, o, kernel == 3, p);
  const size_t vs = dtype_size(m->value_dtype);
  const size_t xbytes = (size_t)m->n_cols * vs;
  p->x_smem = o.x_smem == 1 ? xbytes <= kXsMaxBytes
            : o.x_smem == -1 ? xbytes <= kXsAutoBytes : false;
  p->dyn_smem = (p->x_smem ? (xbytes + 15) / 16 * 16 : 0) +
                kStages * csr_stage_bytes(m->value_dtype);
  p->split_chunk = o.split_chunk;
  p->interleaved = o.interleave == 2 || (o.interleave == 0 && csr_interleave_auto(m));
  info.interleaved = p->interleaved ? 1 : 0;
  if (csr_set_smem_limit(p->dyn_smem) != 0) return SPMV_ERR_CUDA;
  // persistent grid: every CTA that fits on the device at once within the
  // shared-memory budget (so that L1 keeps at least 60 KB for the x gathers)
  const int occ = csr_kernel_occupancy(m->value_dtype, p->x_smem, p->interleaved, p->dyn_smem,
                                       kSmemBudget);
  if (occ <= 0) return SPMV_ERR_CUDA;
  s = plan_csr_tiles(m->n_rows, m->row_ptr, o, occ * p->sm_count, &t, &info);
  if (s != SPMV_OK) return s;
  p->n_tiles = (int64_t)t.tiles.size();
  p->grid = info.grid;
  const size_t nnz_alloc = (size_t)m->nnz + kPadElems;
  if ((s = dev_upload(&p->row_ptr, m->row_ptr, ((size_t)m->n_rows + 1) * 4,
                      ((size_t)m->n_rows + 1 + kPadElems) * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->col_idx, m->col_idx, (size_t)m->nnz * 4,
                      nnz_alloc * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->values, m->values, (size_t)m->nnz * vs,
                      nnz_alloc * vs)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->tiles, t.tiles.data(), t.tiles.size() * sizeof(Tile),
                      t.tiles.size() * sizeof(Tile))) != SPMV_OK) return s;
  if ((s = dev_upload(&p->cta_first, t.cta_first.data(), t.cta_first.size() * 4,
                      t.cta_first.size() * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->splits, t.splits.data(),
                      t.splits.size() * sizeof(SplitInfo),
                      t.splits.size() * sizeof(SplitInfo))) != SPMV_OK) return s;
  if ((s = dev_upload(&p->partials, nullptr, 0,
                      (size_t)t.n_chunks * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->counters, nullptr, 0,
                      t.splits.size() * 4)) != SPMV_OK) return s;
  if ((s = common_buffers(p)) != SPMV_OK) return s;
  info.x_in_smem = p->x_smem ? 1 : 0;
  info.grid = p->grid;
  info.block = kThreads;
  info.launches_per_run = p->n_tiles > 0 ? 1 : 0;
  info.matrix_bytes = (int64_t)m->nnz * (int64_t)(vs + 4) +
                      ((int64_t)m->n_rows + 1) * 4;
  info.aux_bytes = (int64_t)(t.tiles.size() * sizeof(Tile) +
                             t.splits.size() * (sizeof(SplitInfo) + 4) +
                             (size_t)t.n_chunks * 4 + t.cta_first.size() * 4);
  fill_bytes(&info, vs);
  return SPMV_OK;
}

spmv_status validate_delta(const spmv_delta* d, int64_t* nnz_out) {
  if (!d) return SPMV_ERR_INVALID_ARG;
  if (d->n_rows < 0 || d->n_cols < 0 || d->n_entries < 0 || !d->row_ptr)
    return SPMV_ERR_INVALID_ARG;
  if (d->n_entries > 0 && (!d->values || !d->words)) return SPMV_ERR_INVALID_ARG;
  const int32_t b = delta_bits_of(d);
  if (!valid_delta_bits(b)) return SPMV_ERR_INVALID_ARG;
  const int64_t per = delta_per_word(b);
  if (d->n_entries > kMaxIndex || (d->n_entries % per)) {
    return d->n_entries > kMaxIndex ? SPMV_ERR_TOO_LARGE : SPMV_ERR_BAD_ROW_PTR;
  }
  const int64_t* rp = d->row_ptr;
  if (rp[0] != 0 || rp[d->n_rows] != d->n_entries) return SPMV_ERR_BAD_ROW_PTR;
  int64_t nnz = 0;
  for (int32_t r = 0; r < d->n_rows; ++r) {
    if (rp[r + 1] < rp[r] || (rp[r] % per)) return SPMV_ERR_BAD_ROW_PTR;
    int64_t c = 0;
    for (int64_t e = rp[r]; e < rp[r + 1]; ++e) {
      c += delta_at(d->words, e, b);
      if (d->values[e] != 0) ++nnz;
    }
    if (rp[r + 1] > rp[r] && c >= d->n_cols) return SPMV_ERR_COL_OUT_OF_RANGE;
  }
  *nnz_out = nnz;
  return SPMV_OK;
}

// The diagonal of a square fp32 matrix (entries with column == row, repeats
// summed in stored order; 0 where a row has none), kept on the device for
// the Jacobi preconditioner of spmv_pcg_solve.
spmv_status upload_csr_diagonal(const spmv_csr* m, Plan* p) {
  std::vector<float> d;
  try {
    d.assign((size_t)m->n_rows, 0.f);
  } catch (const std::bad_alloc&) {
    return SPMV_ERR_OUT_OF_MEMORY;
  }
  const float* v = static_cast<const float*>(m->values);
  for (int32_t r = 0; r < m->n_rows; ++r)
    for (int32_t k = m->row_ptr[r]; k < m->row_ptr[r + 1]; ++k)
      if (m->col_idx[k] == r) d[r] += v[k];
  return dev_upload(&p->diag, d.data(), d.size() * 4, d.size() * 4 + 16);
}

// ------------------------------------------------------------ SELL
// "CUDA CSR SpMV optimisation" 2.1 (ELL) and 2.2 (choice by the CV of the
// row lengths); the layout is described with spmv_sell in the header.

constexpr int32_t kSellSigmaSorted = 1024;  // window of the middle CV band
constexpr int32_t kSellMaxMeanRow = 128;    // AUTO: longer rows on average go to CSR
// AUTO: rows shorter than this on average go to CSR too. A warp of SELL then
// reads only a few slots and exits after two latency rounds, while CSR's
// short-row tiles already read such rows with coalesced copies: on the
// 1000 x 999 5-point Laplacian (5 per row) CSR runs 10.8 us and SELL 11.5 us;
// on the hex-mesh stiffness matrix (78 per row) SELL runs 71 us and CSR 83 us.
constexpr int32_t kSellMinMeanRow = 16;

double row_length_cv(const spmv_csr* m) {
  if (m->n_rows == 0) return 0.0;
  const double mean = (double)m->nnz / (double)m->n_rows;
  if (mean == 0.0) return 0.0;
  double ss = 0.0;
  for (int32_t r = 0; r < m->n_rows; ++r) {
    const double d = (double)(m->row_ptr[r + 1] - m->row_ptr[r]) - mean;
    ss += d * d;
  }
  return std::sqrt(ss / (double)m->n_rows) / mean;
}

void choose_by_cv(double cv, spmv_format* f, int32_t* sigma) {
  if (cv < 0.3) {
    *f = SPMV_FORMAT_SELL;
    *sigma = 1;
  } else if (cv <= 0.7) {
    *f = SPMV_FORMAT_SELL;
    *sigma = kSellSigmaSorted;
  } else {
    *f = SPMV_FORMAT_CSR;
    *sigma = 0;
  }
}

// The sliced layout of a validated CSR matrix (arrays malloc'ed into *out).
spmv_status sell_layout(const spmv_csr* m, int32_t sigma, spmv_sell* out) {
  constexpr int C = SPMV_SELL_C;
  const int32_t n = m->n_rows;
  const int32_t* rp = m->row_ptr;
  std::vector<int32_t> order;
  try {
    order.resize((size_t)n);
  } catch (const std::bad_alloc&) {
    return SPMV_ERR_OUT_OF_MEMORY;
  }
  for (int32_t i = 0; i < n; ++i) order[i] = i;
  if (sigma > 1)
    for (int64_t w0 = 0; w0 < n; w0 += sigma) {
      const int64_t w1 = std::min<int64_t>(n, w0 + sigma);
      std::stable_sort(order.begin() + w0, order.begin() + w1, [&](int32_t a, int32_t b) {
        return rp[a + 1] - rp[a] > rp[b + 1] - rp[b];
      });
    }
  const int64_t n_slices = ((int64_t)n + C - 1) / C;
  out->slice_ptr = static_cast<int64_t*>(std::malloc((size_t)(n_slices + 1) * 8));
  out->perm = static_cast<int32_t*>(std::malloc((size_t)std::max<int64_t>(n_slices * C, 1) * 4));
  if (!out->slice_ptr || !out->perm) return SPMV_ERR_OUT_OF_MEMORY;
  out->slice_ptr[0] = 0;
  for (int64_t sl = 0; sl < n_slices; ++sl) {
    int64_t w = 0;
    for (int64_t q = sl * C; q < std::min<int64_t>((sl + 1) * C, n); ++q)
      w = std::max<int64_t>(w, rp[order[q] + 1] - rp[order[q]]);
    out->slice_ptr[sl + 1] = out->slice_ptr[sl] + w * C;
  }
  const int64_t slots = out->slice_ptr[n_slices];
  if (slots > kMaxIndex) return SPMV_ERR_TOO_LARGE;
  const size_t vs = dtype_size(m->value_dtype);
  out->cols = static_cast<int32_t*>(std::calloc((size_t)std::max<int64_t>(slots, 1), 4));
  out->values = std::calloc((size_t)std::max<int64_t>(slots, 1), vs);
  if (!out->cols || !out->values) return SPMV_ERR_OUT_OF_MEMORY;
  const unsigned char* src = static_cast<const unsigned char*>(m->values);
  unsigned char* dst = static_cast<unsigned char*>(out->values);
  for (int64_t q = 0; q < n_slices * C; ++q) {
    out->perm[q] = q < n ? order[q] : -1;
    if (q >= n) continue;
    const int32_t i = order[q];
    const int64_t sl = q / C, lane = q % C;
    const int64_t w = (out->slice_ptr[sl + 1] - out->slice_ptr[sl]) / C;
    const int64_t len = rp[i + 1] - rp[i];
    for (int64_t k = 0; k < w; ++k) {
      const int64_t at = out->slice_ptr[sl] + k * C + lane;
      if (k < len) {
        out->cols[at] = m->col_idx[rp[i] + k];
        std::memcpy(dst + at * vs, src + (rp[i] + k) * vs, vs);
      } else if (len > 0) {
        out->cols[at] = m->col_idx[rp[i + 1] - 1];  // value stays 0
      }
    }
  }
  out->n_rows = n;
  out->n_cols = m->n_cols;
  out->nnz = m->nnz;
  out->C = C;
  out->sigma = sigma;
  out->n_slices = n_slices;
  out->n_slots = slots;
  out->value_dtype = m->value_dtype;
  return SPMV_OK;
}

// Bytes the sliced layout stores: every slot's column and value, the slice
// offsets (int32 on the device) and, for sorted rows, the row of each lane.
int64_t sell_matrix_bytes(const spmv_sell& sl) {
  return sl.n_slots * (4 + (int64_t)dtype_size(sl.value_dtype)) + (sl.n_slices + 1) * 4 +
         (sl.sigma > 1 ? sl.n_slices * sl.C * 4 : 0);
}

void sell_info(const spmv_sell& sl, spmv_plan_info* info) {
  info->n_entries = sl.n_slots;
  info->n_tiles = sl.n_slices;
  info->tiles_per_bin[0] = sl.n_slices;
  info->rows_per_bin[1] = sl.n_rows;
  info->grid = (int32_t)((sl.n_slices + kSellSlicesPerCta - 1) / kSellSlicesPerCta);
  info->block = kSellSlicesPerCta * 32;
  info->launches_per_run = sl.n_rows > 0 ? 1 : 0;
  info->matrix_bytes = sell_matrix_bytes(sl);
  fill_bytes(info, dtype_size(sl.value_dtype));
}

spmv_status create_sell_plan(const spmv_sell* sl, Plan* p) {
  spmv_status s;
  if ((s = bind_device(p)) != SPMV_OK) return s;
  const size_t vs = dtype_size(sl->value_dtype);
  std::vector<int32_t> sp;
  try {
    sp.resize((size_t)sl->n_slices + 1);
  } catch (const std::bad_alloc&) {
    return SPMV_ERR_OUT_OF_MEMORY;
  }
  for (int64_t i = 0; i <= sl->n_slices; ++i) sp[i] = (int32_t)sl->slice_ptr[i];
  if ((s = dev_upload(&p->row_ptr, sp.data(), sp.size() * 4, sp.size() * 4)) != SPMV_OK)
    return s;
  if (sl->sigma > 1 &&
      (s = dev_upload(&p->perm, sl->perm, (size_t)sl->n_slices * sl->C * 4,
                      (size_t)sl->n_slices * sl->C * 4)) != SPMV_OK)
    return s;
  if ((s = dev_upload(&p->col_idx, sl->cols, (size_t)sl->n_slots * 4,
                      (size_t)sl->n_slots * 4 + 16)) != SPMV_OK)
    return s;
  if ((s = dev_upload(&p->values, sl->values, (size_t)sl->n_slots * vs,
                      (size_t)sl->n_slots * vs + 16)) != SPMV_OK)
    return s;
  if ((s = common_buffers(p)) != SPMV_OK) return s;
  p->n_tiles = sl->n_slices;
  p->n_entries = sl->n_slots;
  sell_info(*sl, &p->info);
  p->grid = p->info.grid;
  p->info.aux_bytes = 16;
  return SPMV_OK;
}

// Validate a CSR input for `format` and settle the automatic choices: the
// delta width (DELTA_AUTO), CSR or SELL by the CV of the row lengths (AUTO),
// and SELL's sorting window (options, else by the CV band; a SELL forced on
// a matrix whose CV points to CSR gets the sorted window).
spmv_status resolve_format(const spmv_csr* m, const Options& o, spmv_format* format,
                           int32_t* sigma) {
  const bool delta = is_delta_format(*format);
  spmv_status s = validate_csr(m, delta);
  if (s != SPMV_OK) return s;
  if (delta && m->value_dtype != SPMV_F16) return SPMV_ERR_UNSUPPORTED;
  *sigma = 0;
  if (*format == SPMV_FORMAT_DELTA_AUTO) {
    int32_t b = 4;
    if ((s = spmv_delta_select_bits(m, SPMV_DELTA_FEWEST_BYTES, &b, nullptr)) != SPMV_OK)
      return s;
    *format = delta_format(b);
  }
  if (*format == SPMV_FORMAT_AUTO || *format == SPMV_FORMAT_SELL) {
    spmv_format f;
    int32_t sg;
    choose_by_cv(row_length_cv(m), &f, &sg);
    // a lane per row serialises a long row's gathers, and very short rows
    // leave a SELL warp with too little to read: the CV band is taken only
    // for rows of kSellMinMeanRow to kSellMaxMeanRow stored entries on average
    const double nnz = (double)m->nnz, rows = (double)m->n_rows;
    if (*format == SPMV_FORMAT_AUTO)
      *format = (f == SPMV_FORMAT_SELL && (nnz > (double)kSellMaxMeanRow * rows ||
                                           nnz < (double)kSellMinMeanRow * rows))
                    ? SPMV_FORMAT_CSR
                    : f;
    if (*format == SPMV_FORMAT_SELL)
      *sigma = o.sell_sigma > 0 ? o.sell_sigma : (f == SPMV_FORMAT_SELL ? sg : kSellSigmaSorted);
  }
  return SPMV_OK;
}

// The data of one segment in the several-lanes-per-word layout (the block
// layout described with delta_wide_seg_bytes): nw words of b-bit fields and
// their values (32 / b halves a word) into `out`.
void write_delta_wide(int bits, const uint32_t* words, const uint16_t* values, int64_t nw,
                      unsigned char* out) {
  const int L = delta_wide_lanes(bits), W = delta_wide_step_words(bits);
  const int BW = delta_wide_block_words(bits), ob = delta_wide_off_bytes(bits);
  const int64_t per = 32 / bits, nb = nw / BW, nt = nw % BW;
  const uint32_t cap = (1u << bits) - 1u;
  std::vector<uint32_t> off2((size_t)nw);
  uint32_t o = 0;
  for (int64_t j = 0; j < nw; ++j) {
    off2[j] = o;
    for (int64_t q = 0; q < per; ++q) o += 2u * ((words[j] >> (bits * q)) & cap);
  }
  auto put_off = [ob](unsigned char* at, uint32_t v) {
    if (ob == 2) {
      const uint16_t h = (uint16_t)v;
      std::memcpy(at, &h, 2);
    } else {
      std::memcpy(at, &v, 4);
    }
  };
  // value word q (halves 2q, 2q + 1) of word j
  auto val32 = [values, per](int64_t j, int q) {
    uint32_t v;
    std::memcpy(&v, values + j * per + 2 * q, 4);
    return v;
  };
  unsigned char* bw = out;
  unsigned char* bo = bw + nb * W * 16;
  unsigned char* bv = bo + nb * W * 4 * ob;
  for (int64_t h = 0; h < nb; ++h)
    for (int g = 0; g < W; ++g)
      for (int k = 0; k < 4; ++k) {
        const int64_t j = (int64_t)BW * h + (int64_t)W * k + g;
        std::memcpy(bw + ((h * W + g) * 4 + k) * 4, words + j, 4);
        put_off(bo + ((h * W + g) * 4 + k) * ob, off2[j]);
        for (int q = 0; q < L; ++q) {
          const uint32_t v = val32(j, q);
          std::memcpy(bv + ((h * 32 + (int64_t)g * L + q) * 4 + k) * 4, &v, 4);
        }
      }
  unsigned char* tw = bv + nb * 512;
  unsigned char* to = tw + delta_pad16(nt * 4);
  unsigned char* tv = to + delta_pad16(nt * ob);
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t j = nb * BW + t;
    std::memcpy(tw + 4 * t, words + j, 4);
    put_off(to + ob * t, off2[j]);
  }
  std::memcpy(tv, values + nb * BW * per, (size_t)(nt * per) * 2);
}

// Device layout of a DELTA plan: one block per segment, back to back in
// segment order (so each warp's share is contiguous), each block a 32-byte
// header (SegHeader) and the segment's data. A lane per word: the words
// (padded to 16 bytes) and their values (padded to 16 bytes; at 2 bits each
// word's 32 bytes of values are split into two planes of 16-byte halves).
// Several lanes per word (wide): write_delta_wide. One bulk copy stages a
// block.
// seg_off receives every block's offset in 16-byte steps (n_segs + 1).
spmv_status build_delta_blocks(const spmv_delta* d, const SegTables& t, int stages, bool wide,
                               std::vector<uint4>* out, std::vector<int32_t>* seg_off) {
  const int32_t bits = delta_bits_of(d);
  const int64_t per = delta_per_word(bits);
  const size_t n_segs = t.segs.size();
  try {
    seg_off->assign(n_segs + 1, 0);
    int64_t total = 0;  // in 16-byte steps
    for (size_t k = 0; k < n_segs; ++k) {
      (*seg_off)[k] = (int32_t)total;
      const int64_t nw = (int64_t)t.segs[k].end - t.segs[k].begin;
      total += (wide ? delta_wide_seg_bytes(bits, nw) : delta_seg_bytes(bits, nw)) / 16;
      if (total > INT32_MAX) return SPMV_ERR_TOO_LARGE;
    }
    (*seg_off)[n_segs] = (int32_t)total;
    out->assign((size_t)total, make_uint4(0, 0, 0, 0));
  } catch (const std::bad_alloc&) {
    return SPMV_ERR_OUT_OF_MEMORY;
  }
  std::vector<int32_t> next((size_t)n_segs, -1);  // segment staged `stages` later by the same warp
  for (size_t g = 0; g + 1 < t.warp_first.size(); ++g)
    for (int32_t k = t.warp_first[g]; k + stages < t.warp_first[g + 1]; ++k) next[k] = k + stages;
  unsigned char* base = reinterpret_cast<unsigned char*>(out->data());
  for (size_t k = 0; k < n_segs; ++k) {
    const SegDesc& sg = t.segs[k];
    const int64_t wb = sg.begin, nw = (int64_t)sg.end - sg.begin;
    unsigned char* b = base + (size_t)(*seg_off)[k] * 16;
    SegHeader h{};
    h.base = sg.base;
    h.row_flags = (uint32_t)sg.row | sg.flags;
    h.n_words = (int32_t)nw;
    h.split = t.seg_split[k];
    h.slot = t.seg_slot[k];
    h.ctl = t.segs[k].ctl;
    if (next[k] >= 0) {
      h.next_off = (*seg_off)[next[k]];
      h.next_bytes = ((*seg_off)[next[k] + 1] - (*seg_off)[next[k]]) * 16;
    }
    std::memcpy(b, &h, sizeof(h));
    unsigned char* words = b + kSegHeaderBytes;
    const uint16_t* src = d->values + wb * per;
    if (wide) {
      write_delta_wide(bits, d->words + wb, src, nw, words);
      continue;
    }
    unsigned char* vals = words + delta_pad16(nw * 4);
    std::memcpy(words, d->words + wb, (size_t)nw * 4);
    if (bits == 2) {  // two planes: halves 0..7 of each word, then 8..15
      for (int64_t j = 0; j < nw; ++j) {
        std::memcpy(vals + 16 * j, src + 16 * j, 16);
        std::memcpy(vals + 16 * (nw + j), src + 16 * j + 8, 16);
      }
    } else {
      std::memcpy(vals, src, (size_t)(nw * per) * 2);
    }
  }
  return SPMV_OK;
}

// x in shared memory: by default when it is at most kXsAutoBytesDelta, and
// when forced as long as the warps' rings and x fit the CTA's shared memory.
// The DELTA decode of 2- and 4-bit deltas: several lanes per word, except
// for 2-bit deltas that are mostly padding (a lane per word, with the
// padding skip), or when a lane per word is asked for. LLM 12288^2 (us, a
// lane per word / several lanes per word): 4-bit deltas at 30 / 50 / 70 /
// 90% sparsity 55.5 / 52.4, 42.9 / 38.6, 29.6 / 27.4, 16.8 / 16.3; 2-bit
// deltas 57.8 / 51.3, 44.7 / 42.4, and with 35% and 73% padding at 70% and
// 90% 36.0 / 43.4, 28.3 / 36.4.
bool delta_wide_choice(const spmv_delta* d, const Options& o, bool skip_zero) {
  const int32_t b = delta_bits_of(d);
  if ((b != 4 && b != 2) || o.delta_kernel == 1) return false;
  return o.delta_kernel == 2 || b == 4 || !skip_zero;
}

bool delta_skip_zero_choice(const spmv_delta* d);

bool delta_x_fits(int bits, bool wide, int n_cols, int forced, size_t smem_optin) {
  const size_t xb = delta_x_smem_bytes(n_cols);
  const size_t reserve = 4096;  // static shared memory and the runtime's share
  const bool fits = delta_rings_bytes(bits, wide) + xb + reserve <= smem_optin;
  return forced == 1 ? fits : forced == -1 ? (fits && xb <= kXsAutoBytesDelta) : false;
}

// Share of +0.0 entries above which the DELTA kernel reads no x for them.
// LLM 12288^2 (share of +0.0 entries, us without / with the skip): 4-bit
// deltas at 90% sparsity (22%) 17.19 / 16.86; 2-bit at 90% (73%)
// 33.2 / 28.3, at 50% (13%) 44.7 / 45.4.
#ifndef SPMV_DELTA_SKIPZ_PCT
#define SPMV_DELTA_SKIPZ_PCT 18
#endif
constexpr int kDeltaSkipZeroPercent = SPMV_DELTA_SKIPZ_PCT;

// Entries stored as +0.0 (gap padding, row alignment, explicit zeros): when
// they are a noticeable share, the kernel variant that reads no x for them
// is used.
bool delta_skip_zero_choice(const spmv_delta* d) {
  int64_t zeros = 0;
  for (int64_t e = 0; e < d->n_entries; ++e) zeros += d->values[e] == 0;
  return zeros * 100 > d->n_entries * (int64_t)kDeltaSkipZeroPercent;
}

spmv_status create_delta_plan(const spmv_delta* d, const Options& o, Plan* p) {
  spmv_status s;
  spmv_plan_info& info = p->info;
  if ((uint32_t)d->n_rows > kSegRowMask) return SPMV_ERR_TOO_LARGE;
  // the kernel is chosen by the width the matrix was encoded with; the
  // plan's format code must name the same width
  p->delta_bits = delta_bits_of(d);
  if (p->format != delta_format(p->delta_bits)) return SPMV_ERR_INVALID_ARG;
  if ((s = bind_device(p)) != SPMV_OK) return s;
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device) !=
      cudaSuccess)
    return SPMV_ERR_CUDA;
  p->delta_skip_zero = delta_skip_zero_choice(d);
  p->delta_wide = delta_wide_choice(d, o, p->delta_skip_zero);
  p->x_smem = delta_x_fits(p->delta_bits, p->delta_wide, d->n_cols, o.x_smem, (size_t)optin);
  p->dyn_smem = delta_rings_bytes(p->delta_bits, p->delta_wide) +
                (p->x_smem ? delta_x_smem_bytes(d->n_cols) : 0);
  if (delta_set_smem_limit(p->delta_bits, p->delta_wide, p->dyn_smem) != 0) return SPMV_ERR_CUDA;
  const int occ = delta_kernel_occupancy(p->delta_bits, p->delta_wide, p->x_smem, p->dyn_smem);
  if (occ <= 0) return SPMV_ERR_CUDA;
  const int wpc = delta_warps_per_cta(p->delta_bits);
  SegTables t;
  const int per_sm = std::min(occ, delta_grid_per_sm(p->delta_bits));
  if ((s = plan_delta_segments(d, per_sm * p->sm_count * wpc, wpc, &t, &info)) != SPMV_OK)
    return s;
  p->grid = info.grid;
  p->n_tiles = (int64_t)t.segs.size();
  std::vector<uint4> blocks;
  std::vector<int32_t> seg_off;
  if ((s = build_delta_blocks(d, t, delta_stages(p->delta_bits), p->delta_wide, &blocks,
                              &seg_off)) != SPMV_OK)
    return s;
  if ((s = dev_upload(&p->blocks, blocks.data(), blocks.size() * 16,
                      blocks.size() * 16)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->seg_off, seg_off.data(), seg_off.size() * 4,
                      seg_off.size() * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->cta_first, t.warp_first.data(), t.warp_first.size() * 4,
                      t.warp_first.size() * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->empty_rows, t.empty_rows.data(), t.empty_rows.size() * 4,
                      t.empty_rows.size() * 4)) != SPMV_OK) return s;
  p->n_empty_rows = (int32_t)t.empty_rows.size();
  if ((s = dev_upload(&p->splits, t.splits.data(), t.splits.size() * sizeof(SplitInfo),
                      t.splits.size() * sizeof(SplitInfo))) != SPMV_OK) return s;
  if ((s = dev_upload(&p->partials, nullptr, 0, (size_t)t.n_chunks * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->counters, nullptr, 0, t.splits.size() * 4)) != SPMV_OK) return s;
  if ((s = dev_upload(&p->cells, nullptr, 0, t.splits.size() * 8)) != SPMV_OK) return s;
  if ((s = common_buffers(p)) != SPMV_OK) return s;
  info.x_in_smem = p->x_smem ? 1 : 0;
  info.block = wpc * 32;
  info.segments = 1;
  info.launches_per_run = d->n_rows > 0 ? 1 : 0;
  info.matrix_bytes = delta_matrix_bytes(*d);
  // the blocks hold the matrix's values and deltas, the segment headers and
  // the 16-byte alignment padding; the rest of them is auxiliary
  info.aux_bytes = (int64_t)(blocks.size() * 16) -
                   (info.matrix_bytes - ((int64_t)d->n_rows + 1) * 4) +
                   (int64_t)(seg_off.size() * 4 + t.warp_first.size() * 4 +
                             t.empty_rows.size() * 4 + t.splits.size() * (sizeof(SplitInfo) + 4) +
                             (size_t)t.n_chunks * 4);
  fill_bytes(&info, 2);
  return SPMV_OK;
}

// The plan's y = A x launch (skip: see launch_csr; dot: see launch_sell,
// SELL and FEM plans only).
int launch_product(const Plan& p, const void* x, float* y, void* stream, const int* skip,
                   float* dot = nullptr) {
  return p.format == SPMV_FORMAT_CSR    ? (p.csr_segments ? launch_csr_seg(p, x, y, stream, skip)
                                                         : launch_csr(p, x, y, stream, skip))
         : p.format == SPMV_FORMAT_SELL ? launch_sell(p, x, y, stream, skip, dot)
         : p.format == SPMV_FORMAT_FEM  ? launch_fem(p, x, y, stream, skip, dot)
                                        : launch_delta(p, x, y, stream);
}

}  // namespace
}  // namespace spmv

using namespace spmv;

extern "C" {

const char* spmv_status_string(spmv_status s) {
  switch (s) {
    case SPMV_OK: return "ok";
    case SPMV_ERR_INVALID_ARG: return "invalid argument";
    case SPMV_ERR_BAD_ROW_PTR: return "malformed row pointers";
    case SPMV_ERR_COL_OUT_OF_RANGE: return "column index out of range";
    case SPMV_ERR_UNSORTED_OR_DUPLICATE_COLS:
      return "columns not strictly increasing within a row";
    case SPMV_ERR_UNSUPPORTED: return "unsupported format / dtype combination";
    case SPMV_ERR_OUT_OF_MEMORY: return "out of memory";
    case SPMV_ERR_CUDA: return "CUDA runtime error";
    case SPMV_ERR_TOO_LARGE: return "sizes exceed 32-bit device indexing";
    case SPMV_ERR_WRONG_DEVICE: return "current device is not the plan's device";
    case SPMV_ERR_DEVICE_STATUS: return "a kernel reported an error";
  }
  return "unknown status";
}

int32_t spmv_abi_version(void) { return SPMV_ABI_VERSION; }

void spmv_plan_options_init(spmv_plan_options* o) {
  if (!o) return;
  // every size knob 0 = the default for the matrix's value type, chosen when
  // the plan is made (the stage holds more fp16 than fp32 nonzeros)
  std::memset(o, 0, sizeof(*o));
  o->x_smem = -1;
}

spmv_status spmv_convert_bits(const spmv_csr* m, int32_t b, spmv_delta* out) {
  if (!out) return SPMV_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  if (!valid_delta_bits(b)) return SPMV_ERR_INVALID_ARG;
  spmv_status s = validate_csr(m, true);
  if (s != SPMV_OK) return s;
  if (m->value_dtype != SPMV_F16) return SPMV_ERR_UNSUPPORTED;
  const int64_t cap = delta_cap(b), per = delta_per_word(b);
  const int32_t* rp = m->row_ptr;
  const uint16_t* v = static_cast<const uint16_t*>(m->values);
  int64_t* erp = static_cast<int64_t*>(std::malloc(((size_t)m->n_rows + 1) * 8));
  if (!erp) return SPMV_ERR_OUT_OF_MEMORY;
  int64_t total = 0, gaps = 0, aligns = 0;
  erp[0] = 0;
  for (int32_t r = 0; r < m->n_rows; ++r) {
    int64_t n = delta_row_entries(m->col_idx + rp[r], rp[r + 1] - rp[r], cap, &gaps);
    int64_t padded = (n + per - 1) / per * per;
    aligns += padded - n;
    total += padded;
    erp[r + 1] = total;
  }
  uint16_t* vals = static_cast<uint16_t*>(std::malloc((size_t)total * 2 + 16));
  uint32_t* words = static_cast<uint32_t*>(std::calloc((size_t)(total / per) + 1, 4));
  if (!vals || !words) {
    std::free(erp);
    std::free(vals);
    std::free(words);
    return SPMV_ERR_OUT_OF_MEMORY;
  }
  int64_t zeros = 0;
  for (int32_t r = 0; r < m->n_rows; ++r) {
    int64_t e = erp[r], c = 0;
    for (int32_t k = rp[r]; k < rp[r + 1]; ++k) {
      const int64_t col = m->col_idx[k];
      int64_t gap = col - c;
      for (; gap > cap; gap -= cap) emit(vals, words, e++, b, 0, (uint32_t)cap);
      emit(vals, words, e++, b, v[k], (uint32_t)gap);
      zeros += v[k] == 0;
      c = col;
    }
    while (e < erp[r + 1]) emit(vals, words, e++, b, 0, 0);
  }
  out->n_rows = m->n_rows;
  out->n_cols = m->n_cols;
  out->nnz = m->nnz;
  out->n_entries = total;
  out->n_gap_pads = gaps;
  out->n_align_pads = aligns;
  out->n_explicit_zeros = zeros;
  out->values = vals;
  out->words = words;
  out->row_ptr = erp;
  out->delta_bits = b;
  return SPMV_OK;
}

spmv_status spmv_convert(const spmv_csr* m, spmv_delta* out) {
  return spmv_convert_bits(m, 4, out);
}

spmv_status spmv_delta_select_bits(const spmv_csr* m, spmv_delta_policy policy, int32_t* bits,
                                   int64_t entries[3]) {
  if (!bits || (policy != SPMV_DELTA_FEWEST_BYTES && policy != SPMV_DELTA_SPARSITY_TABLE))
    return SPMV_ERR_INVALID_ARG;
  spmv_status s = validate_csr(m, true);
  if (s != SPMV_OK) return s;
  if (m->value_dtype != SPMV_F16) return SPMV_ERR_UNSUPPORTED;
  static const int32_t kWidths[3] = {2, 4, 8};
  int64_t n[3] = {0, 0, 0};
  for (int i = 0; i < 3; ++i) {
    const int32_t b = kWidths[i];
    const int64_t per = delta_per_word(b);
    for (int32_t r = 0; r < m->n_rows; ++r) {
      int64_t gaps = 0;
      const int64_t len = delta_row_entries(m->col_idx + m->row_ptr[r],
                                            m->row_ptr[r + 1] - m->row_ptr[r], delta_cap(b),
                                            &gaps);
      n[i] += (len + per - 1) / per * per;
    }
  }
  if (entries)
    for (int i = 0; i < 3; ++i) entries[i] = n[i];
  if (policy == SPMV_DELTA_SPARSITY_TABLE) {
    const double cells = (double)m->n_rows * (double)m->n_cols;
    const double sp = cells > 0 ? 1.0 - (double)m->nnz / cells : 0.0;
    *bits = sp < 0.3 ? 8 : (sp <= 0.7 ? 4 : 2);
    return SPMV_OK;
  }
  // stored bytes: 2 per entry for the values, b/8 per entry for the deltas
  // (row pointers are the same for every width); ties go to the wider field
  int best = 2;
  for (int i = 1; i >= 0; --i)
    if (n[i] * (16 + kWidths[i]) < n[best] * (16 + kWidths[best])) best = i;
  *bits = kWidths[best];
  return SPMV_OK;
}

spmv_status spmv_convert_sell(const spmv_csr* m, int32_t sigma, spmv_sell* out) {
  if (!out) return SPMV_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  if (sigma < 1) return SPMV_ERR_INVALID_ARG;
  spmv_status s = validate_csr(m, false);
  if (s != SPMV_OK) return s;
  s = sell_layout(m, sigma, out);
  if (s != SPMV_OK) spmv_sell_free(out);
  return s;
}

void spmv_sell_free(spmv_sell* sl) {
  if (!sl) return;
  std::free(sl->slice_ptr);
  std::free(sl->perm);
  std::free(sl->cols);
  std::free(sl->values);
  std::memset(sl, 0, sizeof(*sl));
}

spmv_status spmv_select_format(const spmv_csr* m, spmv_format* format, int32_t* sigma,
                               double* cv) {
  spmv_status s = validate_csr(m, false);
  if (s != SPMV_OK) return s;
  const double c = row_length_cv(m);
  spmv_format f;
  int32_t sg;
  choose_by_cv(c, &f, &sg);
  if (format) *format = f;
  if (sigma) *sigma = sg;
  if (cv) *cv = c;
  return SPMV_OK;
}

void spmv_delta_free(spmv_delta* d) {
  if (!d) return;
  std::free(d->values);
  std::free(d->words);
  std::free(d->row_ptr);
  std::memset(d, 0, sizeof(*d));
}

spmv_status spmv_plan_inspect(const spmv_csr* m, spmv_format format,
                              const spmv_plan_options* opts,
                              spmv_plan_info* info) {
  if (!info || !valid_format(format)) return SPMV_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  if (!m) return SPMV_ERR_INVALID_ARG;
  Options o = resolve_options(opts, m->value_dtype);
  int32_t sigma = 0;
  spmv_status s = resolve_format(m, o, &format, &sigma);
  if (s != SPMV_OK) return s;
  const bool delta = is_delta_format(format);
  info->n_rows = m->n_rows;
  info->n_cols = m->n_cols;
  info->nnz = m->nnz;
  info->format = format;
  info->value_dtype = m->value_dtype;
  info->block = kThreads;
  if (format == SPMV_FORMAT_SELL) {
    spmv_sell sl;
    if ((s = spmv_convert_sell(m, sigma, &sl)) != SPMV_OK) return s;
    sell_info(sl, info);
    info->aux_bytes = 16;
    spmv_sell_free(&sl);
    return SPMV_OK;
  }
  if (delta) {
    spmv_delta d;
    if ((s = spmv_convert_bits(m, format_delta_bits(format), &d)) != SPMV_OK) return s;
    if (d.n_entries > kMaxIndex) {
      spmv_delta_free(&d);
      return SPMV_ERR_TOO_LARGE;
    }
    const bool xs = delta_x_fits(format_delta_bits(format),
                                 delta_wide_choice(&d, o, delta_skip_zero_choice(&d)), m->n_cols,
                                 o.x_smem, kAssumedSmemOptin);
    const int wpc = delta_warps_per_cta(format_delta_bits(format));
    SegTables t;
    s = plan_delta_segments(&d, kAssumedSms * wpc, wpc, &t, info);
    info->block = wpc * 32;
    info->segments = 1;
    info->n_entries = d.n_entries;
    info->x_in_smem = xs ? 1 : 0;
    info->launches_per_run = m->n_rows > 0;
    info->matrix_bytes = delta_matrix_bytes(d);
    fill_bytes(info, 2);
    spmv_delta_free(&d);
    return s;
  }
  const size_t vsz = dtype_size(m->value_dtype);
  const int kernel = csr_kernel_choice(m, o);
  if (kernel >= 2) {
    const bool mixed = kernel == 3;
    const int wpc = csr_seg_warps_per_cta(m->value_dtype, mixed);
    SegTables t;
    s = mixed ? plan_csr_mixed_segments(m, kAssumedSms * wpc, wpc, &t, info)
              : plan_segments(
                    m->n_rows, [&](int32_t r) { return (int64_t)m->row_ptr[r]; },
                    kCsrSegNnzLong, 64, 1, kAssumedSms * wpc, wpc, &t, info);
    if (s != SPMV_OK) return s;
    info->block = wpc * 32;
    info->segments = 1;
    info->n_entries = m->nnz;
    const size_t xbytes = ((size_t)m->n_cols * vsz + 15) / 16 * 16;
    const bool fits =
        csr_seg_rings_bytes(m->value_dtype, mixed) + xbytes + 4096 <= kAssumedSmemOptin;
    info->x_in_smem = o.x_smem == 0 ? 0 : o.x_smem == 1 ? fits : (fits && xbytes <= kXsAutoBytesDelta);
    info->launches_per_run = m->n_rows > 0;
    info->matrix_bytes = m->nnz * (int64_t)(vsz + 4) + ((int64_t)m->n_rows + 1) * 4;
    fill_bytes(info, vsz);
    return SPMV_OK;
  }
  CsrTables t;
  s = plan_csr_tiles(m->n_rows, m->row_ptr, o, 5 * kAssumedSms, &t, info);
  if (s != SPMV_OK) return s;
  info->interleaved = (o.interleave == 2 || (o.interleave == 0 && csr_interleave_auto(m))) ? 1 : 0;
  const size_t vs = dtype_size(m->value_dtype);
  info->n_entries = m->nnz;
  info->x_in_smem = o.x_smem != 0 && (size_t)m->n_cols * vs <=
                    (o.x_smem == 1 ? kXsMaxBytes : kXsAutoBytes);

  info->launches_per_run = info->n_tiles > 0;
  info->matrix_bytes = m->nnz * (int64_t)(vs + 4) + ((int64_t)m->n_rows + 1) * 4;
  info->aux_bytes = (int64_t)(t.tiles.size() * sizeof(Tile) +
                              t.splits.size() * (sizeof(SplitInfo) + 4) +
                              (size_t)t.n_chunks * 4 + t.cta_first.size() * 4);
  fill_bytes(info, vs);
  return SPMV_OK;
}

spmv_status spmv_plan_create_ex(const spmv_csr* m, spmv_format format,
                                const spmv_plan_options* opts,
                                spmv_plan** out) {
  if (!out) return SPMV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!valid_format(format) || !m) return SPMV_ERR_INVALID_ARG;
  Options o = resolve_options(opts, m->value_dtype);
  int32_t sigma = 0;
  spmv_status s = resolve_format(m, o, &format, &sigma);
  if (s != SPMV_OK) return s;
  const bool delta = is_delta_format(format);
  spmv_plan* plan = new (std::nothrow) spmv_plan();
  if (!plan) return SPMV_ERR_OUT_OF_MEMORY;
  Plan* p = &plan->impl;
  p->format = format;
  p->dtype = m->value_dtype;
  p->n_rows = m->n_rows;
  p->n_cols = m->n_cols;
  p->nnz = m->nnz;
  p->info.n_rows = m->n_rows;
  p->info.n_cols = m->n_cols;
  p->info.nnz = m->nnz;
  p->info.format = format;
  p->info.value_dtype = m->value_dtype;
  if (format == SPMV_FORMAT_SELL) {
    spmv_sell sl;
    s = spmv_convert_sell(m, sigma, &sl);
    if (s == SPMV_OK) {
      s = create_sell_plan(&sl, p);
      spmv_sell_free(&sl);
    }
  } else if (delta) {
    spmv_delta d;
    s = spmv_convert_bits(m, format_delta_bits(format), &d);
    if (s == SPMV_OK) {
      if (d.n_entries > kMaxIndex) {
        s = SPMV_ERR_TOO_LARGE;
      } else {
        p->n_entries = d.n_entries;
        p->info.n_entries = d.n_entries;
        s = create_delta_plan(&d, o, p);
      }
      spmv_delta_free(&d);
    }
  } else {
    p->n_entries = m->nnz;
    p->info.n_entries = m->nnz;
    s = create_csr_plan(m, o, p);
  }
  if (s == SPMV_OK && !delta && m->value_dtype == SPMV_F32 && m->n_rows == m->n_cols)
    s = upload_csr_diagonal(m, p);
  if (s != SPMV_OK) {
    free_plan(plan);
    return s;
  }
  *out = plan;
  return SPMV_OK;
}

spmv_status spmv_plan_create(const spmv_csr* m, spmv_format format,
                             spmv_plan** out) {
  return spmv_plan_create_ex(m, format, nullptr, out);
}

spmv_status spmv_plan_create_delta(const spmv_delta* d,
                                   const spmv_plan_options* opts,
                                   spmv_plan** out) {
  if (!out) return SPMV_ERR_INVALID_ARG;
  *out = nullptr;
  int64_t nnz = 0;
  spmv_status s = validate_delta(d, &nnz);
  if (s != SPMV_OK) return s;
  Options o = resolve_options(opts, SPMV_F16);
  spmv_plan* plan = new (std::nothrow) spmv_plan();
  if (!plan) return SPMV_ERR_OUT_OF_MEMORY;
  Plan* p = &plan->impl;
  p->format = delta_format(delta_bits_of(d));
  p->dtype = SPMV_F16;
  p->n_rows = d->n_rows;
  p->n_cols = d->n_cols;
  p->nnz = nnz;
  p->n_entries = d->n_entries;
  p->info.n_rows = d->n_rows;
  p->info.n_cols = d->n_cols;
  p->info.nnz = nnz;
  p->info.format = p->format;
  p->info.value_dtype = SPMV_F16;
  p->info.n_entries = d->n_entries;
  s = create_delta_plan(d, o, p);
  if (s != SPMV_OK) {
    free_plan(plan);
    return s;
  }
  *out = plan;
  return SPMV_OK;
}

spmv_status spmv_plan_create_fem(const spmv_fem_mesh* mesh, spmv_plan** out) {
  if (!out) return SPMV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!mesh || !mesh->rho || !mesh->K0 || mesh->nex < 1 || mesh->ney < 1 || mesh->nez < 1)
    return SPMV_ERR_INVALID_ARG;
  const int64_t nnx = (int64_t)mesh->nex + 1, nny = (int64_t)mesh->ney + 1,
                nnz = (int64_t)mesh->nez + 1;
  const int64_t n_nodes = nnx * nny * nnz;
  if (3 * n_nodes > kMaxIndex) return SPMV_ERR_TOO_LARGE;
  const int64_t n_elem = (int64_t)mesh->nex * mesh->ney * mesh->nez;
  for (int q = 0; q < 24 * 24; ++q)
    if (!std::isfinite(mesh->K0[q])) return SPMV_ERR_INVALID_ARG;
  for (int64_t e = 0; e < n_elem; ++e)
    if (!std::isfinite(mesh->rho[e])) return SPMV_ERR_INVALID_ARG;
  spmv_plan* plan = new (std::nothrow) spmv_plan();
  if (!plan) return SPMV_ERR_OUT_OF_MEMORY;
  Plan* p = &plan->impl;
  p->format = SPMV_FORMAT_FEM;
  p->dtype = SPMV_F32;
  p->n_rows = p->n_cols = (int)(3 * n_nodes);
  // the stored entries the assembled matrix would have: node pairs that share
  // an element, 9 per pair, 3 m - 2 neighbours summed along an axis of m nodes
  p->nnz = 9 * (3 * nnx - 2) * (3 * nny - 2) * (3 * nnz - 2);
  p->n_tiles = n_nodes;
  p->fem_dims[0] = mesh->nex;
  p->fem_dims[1] = mesh->ney;
  p->fem_dims[2] = mesh->nez;
  std::memcpy(p->fem_k0, mesh->K0, sizeof(p->fem_k0));
  spmv_plan_info& info = p->info;
  info.n_rows = info.n_cols = p->n_rows;
  info.nnz = p->nnz;
  info.format = SPMV_FORMAT_FEM;
  info.value_dtype = SPMV_F32;
  info.n_tiles = n_nodes;
  info.block = kFemThreads;
  info.launches_per_run = 1;
  info.matrix_bytes = n_elem * 4 + 24 * 24 * 4;
  fill_bytes(&info, 4);
  spmv_status s = bind_device(p);
  if (s == SPMV_OK) s = dev_upload(&p->values, mesh->rho, (size_t)n_elem * 4, (size_t)n_elem * 4);
  if (s == SPMV_OK) s = common_buffers(p);
  if (s == SPMV_OK) {
    // the diagonal, for the Jacobi preconditioner: every element adds
    // rho_e K0[d][d] at each of its local dofs d (element order, fp64, one
    // rounding to fp32)
    std::vector<double> dd;
    std::vector<float> d;
    try {
      dd.assign((size_t)(3 * n_nodes), 0.0);
      d.resize(dd.size());
    } catch (const std::bad_alloc&) {
      s = SPMV_ERR_OUT_OF_MEMORY;
    }
    static const int kCx[8] = {0, 1, 1, 0, 0, 1, 1, 0}, kCy[8] = {0, 0, 1, 1, 0, 0, 1, 1};
    for (int64_t e = 0; s == SPMV_OK && e < n_elem; ++e) {
      const int64_t ex = e % mesh->nex, ey = (e / mesh->nex) % mesh->ney,
                    ez = e / ((int64_t)mesh->nex * mesh->ney);
      for (int b = 0; b < 8; ++b) {
        const int64_t nd = (ex + kCx[b]) + nnx * ((ey + kCy[b]) + nny * (ez + (b >= 4)));
        for (int c = 0; c < 3; ++c)
          dd[3 * nd + c] += (double)mesh->rho[e] * (double)mesh->K0[(3 * b + c) * 25];
      }
    }
    for (size_t q = 0; s == SPMV_OK && q < d.size(); ++q) d[q] = (float)dd[q];
    if (s == SPMV_OK) s = dev_upload(&p->diag, d.data(), d.size() * 4, d.size() * 4 + 16);
  }
  if (s != SPMV_OK) {
    free_plan(plan);
    return s;
  }
  p->grid = (int)((n_nodes + kFemThreads - 1) / kFemThreads);
  info.grid = p->grid;
  info.aux_bytes = 16;
  *out = plan;
  return SPMV_OK;
}

// Iterations in one pass of the device-side loop's body; the ones after
// convergence skip themselves. On the hex-mesh system (686k unknowns,
// matrix-free, 10 iterations) 1 and 2 measured 25.8 and 24.3 us per
// iteration (each pass of the loop costs about 1.5 us); 4 was no faster
// than 2.
#ifndef SPMV_PCG_BODY
#define SPMV_PCG_BODY 2
#endif
constexpr int kPcgBodyIterations = SPMV_PCG_BODY;

spmv_status spmv_pcg_solve(spmv_plan* plan, const float* diag, const float* b, float* x,
                           double rel_tol, int32_t max_iter, int32_t check_every, void* stream,
                           spmv_pcg_result* result) {
  if (!plan || !result) return SPMV_ERR_INVALID_ARG;
  std::memset(result, 0, sizeof(*result));
  Plan& p = plan->impl;
  if (p.dtype != SPMV_F32 || p.n_rows != p.n_cols || is_delta_format(p.format))
    return SPMV_ERR_INVALID_ARG;
  const float* d = diag ? diag : p.diag;
  if (p.n_rows > 0 && (!b || !x || !d)) return SPMV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPMV_ERR_CUDA;
  if (dev != p.device) return SPMV_ERR_WRONG_DEVICE;
  if (p.n_rows == 0) {
    result->status = kPcgConverged;
    return SPMV_OK;
  }
  spmv_status s;
  if (!p.pcg_work &&
      (s = dev_alloc(&p.pcg_work, pcg_work_bytes(p.n_rows, p.grid))) != SPMV_OK)
    return s;
  const size_t vec = ((size_t)p.n_rows * 4 + 255) / 256 * 256;
  float* pv = reinterpret_cast<float*>(p.pcg_work + 2 * vec);
  float* qv = reinterpret_cast<float*>(p.pcg_work + 3 * vec);
  PcgScalars* sc_dev =
      reinterpret_cast<PcgScalars*>(p.pcg_work + 4 * vec + 3 * kPcgBlocks * sizeof(float));
  // SELL and FEM products also hand over p . q per CTA: no step-length kernel
  const bool fused = pcg_fused_dot(p);
  float* pq_dev = fused ? reinterpret_cast<float*>(p.pcg_work + 4 * vec +
                                                   3 * kPcgBlocks * sizeof(float) + 256)
                        : nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PcgScalars sc{};
  sc.tol2 = rel_tol * rel_tol;
  sc.max_iter = max_iter;
  if (cudaMemcpyAsync(sc_dev, &sc, sizeof(sc), cudaMemcpyHostToDevice, st) != cudaSuccess)
    return SPMV_ERR_CUDA;
  if ((s = spmv_run(plan, x, qv, stream)) != SPMV_OK) return s;  // q = A x0
  if (launch_pcg(0, p, b, x, d, stream) != 0) return SPMV_ERR_CUDA;
  // Batches of 4, then 8, then check_every (default 16) iterations: short
  // solves stop within a few iterations of convergence, long ones pay one
  // host check per check_every iterations.
  const int full = check_every > 0 ? check_every : 16;
  // the products skip themselves once the solve is done (the device flag)
  const int* done_flag = &sc_dev->done;
  // one iteration's vector kernels after the product; cond goes to the
  // direction kernel, which decides whether the loop goes on
  auto launch_vectors = [&](unsigned long long cond) -> bool {
    if (!fused && launch_pcg(1, p, b, x, d, stream) != 0) return false;
    return launch_pcg(2, p, b, x, d, stream) == 0 && launch_pcg(3, p, b, x, d, stream, cond) == 0;
  };
  auto enqueue_batch = [&](int n_it) -> spmv_status {
    for (int k = 0; k < n_it; ++k)
      if (launch_product(p, pv, qv, stream, done_flag, pq_dev) != 0 || !launch_vectors(0))
        return SPMV_ERR_CUDA;
    return SPMV_OK;
  };
  // A batch is 4 launches per iteration; replaying it as one CUDA graph
  // takes the host's launch cost out of the loop. The graphs bake in b, x
  // and the diagonal, so they are kept for the next solve with the same
  // ones. The legacy default stream cannot be captured, nor can a stream the
  // caller is already capturing: those take the direct launches.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool graphable = st != nullptr && cudaStreamIsCapturing(st, &cap) == cudaSuccess &&
                         cap == cudaStreamCaptureStatusNone;
  cudaGetLastError();
  const void* key[3] = {b, x, d};
  if (p.pcg_key[0] != key[0] || p.pcg_key[1] != key[1] || p.pcg_key[2] != key[2]) {
    for (int g = 0; g < Plan::kPcgGraphs; ++g) {
      if (p.pcg_exec[g]) cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(p.pcg_exec[g]));
      p.pcg_exec[g] = nullptr;
      p.pcg_batch[g] = 0;
    }
    if (p.pcg_loop) cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(p.pcg_loop));
    p.pcg_loop = nullptr;
    p.pcg_loop_failed = false;
    for (int q = 0; q < 3; ++q) p.pcg_key[q] = key[q];
  }
  // The whole loop on the device: a graph whose while node runs
  // kPcgBodyIterations iterations (each the product and its vector kernels)
  // as long as the last direction kernel says so (it stops the loop on
  // convergence, the iteration limit or a breakdown; iterations after that
  // inside the same pass skip themselves), so the host waits once per
  // solve. Built once per b, x and diag; a device or driver that refuses it
  // leaves the batches below.
  if (graphable && !p.pcg_loop && !p.pcg_loop_failed) {
    cudaGraph_t g = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaGraphConditionalHandle h = 0;
    bool ok = cudaGraphCreate(&g, 0) == cudaSuccess &&
              cudaGraphConditionalHandleCreate(&h, g, 1, cudaGraphCondAssignDefault) ==
                  cudaSuccess;
    cudaGraphNodeParams np{};
    cudaGraphNode_t node = nullptr;
    if (ok) {
      np.type = cudaGraphNodeTypeConditional;
      np.conditional.handle = h;
      np.conditional.type = cudaGraphCondTypeWhile;
      np.conditional.size = 1;
      ok = cudaGraphAddNode(&node, g, nullptr, nullptr, 0, &np) == cudaSuccess;
    }
    if (ok) {
      cudaGraph_t body = np.conditional.phGraph_out[0];
      ok = cudaStreamBeginCaptureToGraph(st, body, nullptr, nullptr, 0,
                                         cudaStreamCaptureModeThreadLocal) == cudaSuccess;
      if (ok) {
        bool launched = true;
        for (int u = 0; u < kPcgBodyIterations && launched; ++u)
          launched = launch_product(p, pv, qv, stream, done_flag, pq_dev) == 0 &&
                     launch_vectors(u + 1 == kPcgBodyIterations ? (unsigned long long)h : 0ull);
        ok = cudaStreamEndCapture(st, &body) == cudaSuccess && launched;
      }
    }
    if (ok) ok = cudaGraphInstantiate(&exec, g, 0) == cudaSuccess;
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    if (ok && exec) {
      p.pcg_loop = exec;
    } else {
      if (exec) cudaGraphExecDestroy(exec);
      p.pcg_loop_failed = true;
    }
  }
  if (p.pcg_loop && max_iter > 0) {
    if (cudaGraphLaunch(static_cast<cudaGraphExec_t>(p.pcg_loop), st) != cudaSuccess ||
        cudaMemcpyAsync(&sc, sc_dev, sizeof(sc), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return SPMV_ERR_CUDA;
    result->iterations = sc.iter;
    result->status = sc.done ? sc.done : kPcgMaxIter;
    result->rel_residual = sc.bb > 0 ? std::sqrt(sc.rr / sc.bb) : std::sqrt(sc.rr);
    return SPMV_OK;
  }
  // the graph of a batch length, captured on first use (null: launch directly)
  auto graph_for = [&](int n_it) -> cudaGraphExec_t {
    if (!graphable) return nullptr;
    int slot = -1;
    for (int g = 0; g < Plan::kPcgGraphs; ++g)
      if (p.pcg_batch[g] == n_it && p.pcg_exec[g])
        return static_cast<cudaGraphExec_t>(p.pcg_exec[g]);
      else if (slot < 0 && !p.pcg_exec[g])
        slot = g;
    if (slot < 0) return nullptr;
    cudaGraph_t gr = nullptr;
    cudaGraphExec_t exec = nullptr;
    if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
      const spmv_status e = enqueue_batch(n_it);
      const cudaError_t ce = cudaStreamEndCapture(st, &gr);
      if (e != SPMV_OK || ce != cudaSuccess || !gr ||
          cudaGraphInstantiate(&exec, gr, 0) != cudaSuccess)
        exec = nullptr;
      if (gr) cudaGraphDestroy(gr);
    }
    cudaGetLastError();  // a failed capture leaves the direct launches
    if (exec) {
      p.pcg_exec[slot] = exec;
      p.pcg_batch[slot] = n_it;
    }
    return exec;
  };
  for (int64_t it = 0;;) {
    // the first batch goes out unchecked: if x0 already solves the system,
    // the device flag makes it a run of no-ops
    if (it > 0 || max_iter <= 0) {
      if (cudaMemcpyAsync(&sc, sc_dev, sizeof(sc), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
          cudaStreamSynchronize(st) != cudaSuccess)
        return SPMV_ERR_CUDA;
      if (sc.done || it >= max_iter) break;
    }
    const int n_it = it == 0 ? std::min(4, full) : (it == std::min(4, full) ? std::min(8, full) : full);
    cudaGraphExec_t exec = graph_for(n_it);
    if (exec) {
      if (cudaGraphLaunch(exec, st) != cudaSuccess) return SPMV_ERR_CUDA;
    } else if ((s = enqueue_batch(n_it)) != SPMV_OK) {
      return s;
    }
    it += n_it;
  }
  result->iterations = sc.iter;
  result->status = sc.done ? sc.done : kPcgMaxIter;
  result->rel_residual = sc.bb > 0 ? std::sqrt(sc.rr / sc.bb) : std::sqrt(sc.rr);
  return SPMV_OK;
}

spmv_status spmv_plan_get_info(const spmv_plan* plan, spmv_plan_info* info) {
  if (!plan || !info) return SPMV_ERR_INVALID_ARG;
  *info = plan->impl.info;
  return SPMV_OK;
}

static spmv_status check_run_args(const Plan& p, const void* x, const float* y,
                                  size_t* x_elem) {
  const size_t xs =
      p.dtype == SPMV_F32 ? 4 : 2;
  *x_elem = xs;
  if ((p.n_cols > 0 && !x) || (p.n_rows > 0 && !y)) return SPMV_ERR_INVALID_ARG;
  if (((uintptr_t)x % xs) || ((uintptr_t)y % 4)) return SPMV_ERR_INVALID_ARG;
  const uintptr_t x0 = (uintptr_t)x, x1 = x0 + (uintptr_t)p.n_cols * xs;
  const uintptr_t y0 = (uintptr_t)y, y1 = y0 + (uintptr_t)p.n_rows * 4;
  if (p.n_cols > 0 && p.n_rows > 0 && x0 < y1 && y0 < x1)
    return SPMV_ERR_INVALID_ARG;
  return SPMV_OK;
}

spmv_status spmv_run(spmv_plan* plan, const void* x, float* y, void* stream) {
  if (!plan) return SPMV_ERR_INVALID_ARG;
  Plan& p = plan->impl;
  size_t xs;
  spmv_status s = check_run_args(p, x, y, &xs);
  if (s != SPMV_OK) return s;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPMV_ERR_CUDA;
  if (dev != p.device) return SPMV_ERR_WRONG_DEVICE;
  if (p.n_rows == 0) return SPMV_OK;
  int rc = launch_product(p, x, y, stream, nullptr);
  return rc == 0 ? SPMV_OK : SPMV_ERR_CUDA;
}

spmv_status spmv_run_host(spmv_plan* plan, const void* x_host, float* y_host,
                          void* stream) {
  if (!plan) return SPMV_ERR_INVALID_ARG;
  Plan& p = plan->impl;
  if ((p.n_cols > 0 && !x_host) || (p.n_rows > 0 && !y_host))
    return SPMV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPMV_ERR_CUDA;
  if (dev != p.device) return SPMV_ERR_WRONG_DEVICE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t xs =
      p.dtype == SPMV_F32 ? 4 : 2;
  if (p.n_cols > 0 &&
      cudaMemcpyAsync(p.x_stage, x_host, (size_t)p.n_cols * xs,
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return SPMV_ERR_CUDA;
  spmv_status s = spmv_run(plan, p.x_stage, p.y_stage, stream);
  if (s != SPMV_OK) return s;
  if (p.n_rows > 0 &&
      cudaMemcpyAsync(y_host, p.y_stage, (size_t)p.n_rows * 4,
                      cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SPMV_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? SPMV_OK : SPMV_ERR_CUDA;
}

spmv_status spmv_run_host_batch(spmv_plan* plan, int32_t count, const void* x_host,
                                float* y_host, void* stream) {
  if (!plan || count < 0) return SPMV_ERR_INVALID_ARG;
  Plan& p = plan->impl;
  if (count == 0) return SPMV_OK;
  if ((p.n_cols > 0 && !x_host) || (p.n_rows > 0 && !y_host)) return SPMV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPMV_ERR_CUDA;
  if (dev != p.device) return SPMV_ERR_WRONG_DEVICE;
  const size_t xs = p.dtype == SPMV_F32 ? 4 : 2;
  const size_t xb = (size_t)p.n_cols * xs, yb = (size_t)p.n_rows * 4;
  spmv_status s;
  // the second staging pair, the two copy streams and the events, once per plan
  if (!p.x_stage2) {
    if ((s = dev_alloc(&p.x_stage2, xb + 16)) != SPMV_OK) return s;
    if ((s = dev_alloc(&p.y_stage2, yb + 16)) != SPMV_OK) return s;
  }
  for (void*& q : p.batch_streams)
    if (!q) {
      cudaStream_t c = nullptr;
      if (cudaStreamCreateWithFlags(&c, cudaStreamNonBlocking) != cudaSuccess) return SPMV_ERR_CUDA;
      q = c;
    }
  for (void*& e : p.batch_events)
    if (!e) {
      cudaEvent_t c = nullptr;
      if (cudaEventCreateWithFlags(&c, cudaEventDisableTiming) != cudaSuccess) return SPMV_ERR_CUDA;
      e = c;
    }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t s_in = static_cast<cudaStream_t>(p.batch_streams[0]);
  cudaStream_t s_out = static_cast<cudaStream_t>(p.batch_streams[1]);
  auto ev = [&](int k) { return static_cast<cudaEvent_t>(p.batch_events[k]); };
  // events 0-1: copy-in of slot 0 / 1 done; 2-3: product done; 4-5: copy-out
  // done; 6: the caller's earlier work on `stream`
  void* xst[2] = {p.x_stage, p.x_stage2};
  float* yst[2] = {p.y_stage, p.y_stage2};
  const unsigned char* xh = static_cast<const unsigned char*>(x_host);
  bool ok = cudaEventRecord(ev(6), st) == cudaSuccess &&
            cudaStreamWaitEvent(s_in, ev(6), 0) == cudaSuccess &&
            cudaStreamWaitEvent(s_out, ev(6), 0) == cudaSuccess;
  // vector i: copy in on s_in, product on `stream`, copy out on s_out; slot
  // i % 2 is reused by vector i + 2 only after vector i's product has read
  // it (copy-in) and its y has been copied out (product)
  for (int32_t i = 0; ok && i < count; ++i) {
    const int sl = i & 1;
    if (i >= 2) ok = cudaStreamWaitEvent(s_in, ev(2 + sl), 0) == cudaSuccess;
    ok = ok && (xb == 0 || cudaMemcpyAsync(xst[sl], xh + (size_t)i * xb, xb,
                                           cudaMemcpyHostToDevice, s_in) == cudaSuccess) &&
         cudaEventRecord(ev(sl), s_in) == cudaSuccess &&
         cudaStreamWaitEvent(st, ev(sl), 0) == cudaSuccess &&
         (i < 2 || cudaStreamWaitEvent(st, ev(4 + sl), 0) == cudaSuccess);
    if (!ok) break;
    if ((s = spmv_run(plan, xst[sl], yst[sl], stream)) != SPMV_OK) return s;
    ok = cudaEventRecord(ev(2 + sl), st) == cudaSuccess &&
         cudaStreamWaitEvent(s_out, ev(2 + sl), 0) == cudaSuccess &&
         (yb == 0 || cudaMemcpyAsync(y_host + (size_t)i * p.n_rows, yst[sl], yb,
                                     cudaMemcpyDeviceToHost, s_out) == cudaSuccess) &&
         cudaEventRecord(ev(4 + sl), s_out) == cudaSuccess;
  }
  // every stream drained, also after a failed enqueue
  const bool drained = cudaStreamSynchronize(s_in) == cudaSuccess &&
                       cudaStreamSynchronize(st) == cudaSuccess &&
                       cudaStreamSynchronize(s_out) == cudaSuccess;
  return ok && drained ? SPMV_OK : SPMV_ERR_CUDA;
}

spmv_status spmv_plan_check(spmv_plan* plan) {
  if (!plan) return SPMV_ERR_INVALID_ARG;
  Plan& p = plan->impl;
  DeviceGuard g(p.device);
  if (!g.ok) return SPMV_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPMV_ERR_CUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, p.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPMV_ERR_CUDA;
  if (word != 0) {
    cudaMemset(p.status, 0, 4);
    return SPMV_ERR_DEVICE_STATUS;
  }
  return SPMV_OK;
}

void spmv_plan_destroy(spmv_plan* plan) {
  if (!plan) return;
  free_plan(plan);
}

}  // extern "C"
