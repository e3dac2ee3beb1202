// Internal declarations shared by the host planner (spmv_host.cpp) and the
// device kernels (spmv_csr.cu, spmv_delta.cu). Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <functional>
#include <vector>

#include "../../include/spmv.h"

namespace spmv {

// ---------------------------------------------------------------- checked builds
// SPMV_CHECKED=1 (a separate build of the library, for debugging) makes the
// CSR kernels and the allocation-free entry point test every column index
// against the column count and every row offset against its slice before
// using it. An index out of range is replaced by a safe one (column 0; the
// nearest end of the slice) and the kernel records kStatusBadIndex in the
// device status word: results are then wrong but no access leaves its
// buffer, and nothing traps. Ordinary builds compile the checks away.
#ifndef SPMV_CHECKED
#define SPMV_CHECKED 0
#endif
constexpr bool kChecked = SPMV_CHECKED != 0;
constexpr int32_t kStatusBadIndex = 3;
// A column as a checked build uses it: c if 0 <= c < n, else 0 (bad set).
__host__ __device__ constexpr int checked_col(int c, int n, bool* bad) {
  return ((unsigned)c < (unsigned)n) ? c : (*bad = true, 0);
}
// An offset as a checked build uses it: clamped into [lo, hi] (bad set when
// it was outside).
__host__ __device__ constexpr int checked_offset(int v, int lo, int hi, bool* bad) {
  return v < lo ? (*bad = true, lo) : v > hi ? (*bad = true, hi) : v;
}

// ---------------------------------------------------------------- geometry
constexpr int kThreads = 256;            // CTA size of every kernel
constexpr int kWarps = kThreads / 32;
// CSR kernel: every work unit holds at most kTileCap nonzeros; its column,
// value and row-pointer slices are staged in shared memory by TMA bulk
// copies through a ring of kStages buffers.
#ifndef SPMV_TILE_CAP
#define SPMV_TILE_CAP 2048
#endif
#ifndef SPMV_STAGES
#define SPMV_STAGES 2
#endif
#ifndef SPMV_TILE_CAP_F16
#define SPMV_TILE_CAP_F16 2048
#endif
// Stage capacity in nonzeros, per value type. Larger fp16 stages (2560,
// 3072) measured slower on the same plans: the shared memory they take from
// the L1 carve-out is what caches the gathered x.
constexpr int kTileCap = SPMV_TILE_CAP;
constexpr int kTileCapF16 = SPMV_TILE_CAP_F16;
constexpr int tile_cap(spmv_dtype t) { return t == SPMV_F16 ? kTileCapF16 : kTileCap; }
// A short-row tile gives each thread one chunk of 8 consecutive nonzeros, so
// its aligned span (start rounded down to 8) must fit kThreads * 8.
// (walk mode; lanes mode takes any tile that fits a stage, tile_cap - 16).
constexpr int kStreamTileCap = (kTileCap < kThreads * 8 ? kTileCap : kThreads * 8) - 16;
constexpr int kTileRowsCap = 512;        // rows of a short-row tile
constexpr int kStages = SPMV_STAGES;
constexpr int kSellSlicesPerCta = 8;  // SELL: one warp per slice
constexpr int kFemThreads = 128;      // matrix-free FEM: one thread per node
constexpr int kPcgThreads = 256;      // conjugate gradients: vector kernels
constexpr int kPcgBlocks = 608;       // at most 4 blocks per SM of 152 (grid-stride)
constexpr int kPcgConverged = 1, kPcgMaxIter = 2, kPcgBreakdown = 3;

// Device-side scalars of a conjugate-gradient solve.
struct PcgScalars {
  double rz, rr, bb, alpha, beta, tol2;
  double rz_prev;  // rz at the start of the current iteration
  int iter, max_iter, done, arrived;
};
// DELTA kernel ("MACKO-SpMV" 2.2): rows are cut into segments of at most
// delta_seg_words(b) packed words; every warp of the grid owns a contiguous
// share of the segments and stages them through its own ring of shared-memory
// buffers, one bulk copy per segment. Lane l decodes words l, l + 32, ... of a
// segment (delta_lane_words(b) of them at most).
constexpr int delta_lane_words(int bits) { return bits == 2 ? 2 : 4; }
constexpr int delta_seg_words(int bits) { return 32 * delta_lane_words(bits); }
constexpr int kSegHeaderBytes = 32;
constexpr int64_t delta_pad16(int64_t b) { return (b + 15) & ~(int64_t)15; }
// Bytes of the device block of a segment of n_w words of b-bit deltas: the
// header, the words (padded to 16 bytes) and their values (32 / b halves a
// word, padded to 16 bytes).
constexpr int64_t delta_seg_bytes(int bits, int64_t n_w) {
  return kSegHeaderBytes + delta_pad16(n_w * 4) + delta_pad16(n_w * (64 / bits));
}
// The several-lanes-per-word layout (2- and 4-bit deltas). Each word has a
// doubled column offset, from the segment's starting column, of the entry
// before it: uint16 for 4-bit deltas (at most 2 x 127 words x 120 = 30,480;
// 2 bytes a word where 4 would add a fifth to the block: LLM 12288^2 at 30%
// sparsity 51.3 -> 48.6 us), uint32 for 2-bit deltas (their words carry 36
// bytes; uint16 measured no faster). L lanes share a word (4 for 4-bit
// deltas, 8 for 2-bit), a warp-wide step covers W = 32 / L words, and the
// words are stored in blocks of four steps (4 W words) so that a lane loads
// a block's words, offsets and values with three vector loads:
//   block h, lane l = g L + q (g = l / L, q = l % L), step k < 4 covers word
//   j = 4 W h + W k + g, whose 32-bit value word q the lane multiplies:
//   words   uint32 [h][g][k]      (16 bytes per (h, g))
//   offsets uint16/32 [h][g][k]
//   values  uint32 [h][l][k]      (16 bytes per (h, l))
// The n_w mod 4 W words after the last whole block follow in plain order:
// their words, their offsets (each part padded to 16 bytes) and their
// values (L uint32 a word).
constexpr int delta_wide_off_bytes(int bits) { return bits == 4 ? 2 : 4; }
static_assert(2 * (delta_seg_words(4) - 1) * 8 * 15 < 65536,
              "a 4-bit segment's doubled word offsets fit uint16");
constexpr int delta_wide_lanes(int bits) { return bits == 4 ? 4 : 8; }
constexpr int delta_wide_step_words(int bits) { return 32 / delta_wide_lanes(bits); }
constexpr int delta_wide_block_words(int bits) { return 4 * delta_wide_step_words(bits); }
constexpr int64_t delta_wide_block_bytes(int bits) {
  return delta_wide_block_words(bits) * (4 + delta_wide_off_bytes(bits) + 64 / bits);
}
constexpr int64_t delta_wide_seg_bytes(int bits, int64_t n_w) {
  const int64_t nb = n_w / delta_wide_block_words(bits), nt = n_w % delta_wide_block_words(bits);
  return kSegHeaderBytes + nb * delta_wide_block_bytes(bits) + delta_pad16(nt * 4) +
         delta_pad16(nt * delta_wide_off_bytes(bits)) + nt * (64 / bits);
}
// The largest block of a segment (its ring buffer's size).
constexpr int64_t delta_wide_seg_bytes_max(int bits) {
  int64_t m = 0;
  for (int64_t n = 0; n <= delta_seg_words(bits); ++n)
    m = delta_wide_seg_bytes(bits, n) > m ? delta_wide_seg_bytes(bits, n) : m;
  return m;
}
// Segment header (DELTA, and CSR with long rows), the first 32 bytes of its
// block:
//   base       DELTA: column before the segment's first entry; CSR: rows of
//              a packed run (0 for a slice)
//   row_flags  row | kSegFirst (first segment of the row) | kSegLast (last)
//   n_words    items in the segment (DELTA: packed words; CSR: nonzeros)
//   split      index into the split table when the row's segments are shared
//              by several warps, else -1
//   next_off   the block that this warp stages S segments later: offset in
//   next_bytes 16-byte steps and size in bytes (0 when there is none)
//   slot       for a split row: the partial-sum slot of this warp's piece
//   ctl        kSegCtlPieceEnd: the last segment of this warp's piece of a
//              split row that is not the row's last segment (the warp
//              reduces and parks its piece here); kSegCtlCombine: every
//              piece of this warp is parked after this segment (the warp
//              counts them and combines the rows it completes here);
//              kSegCtlPair: the row is split into exactly two pieces (they
//              meet in one 64-bit exchange, see the kernels)
struct SegHeader {
  int32_t base;
  uint32_t row_flags;
  int32_t n_words;
  int32_t split;
  int32_t next_off;
  int32_t next_bytes;
  int32_t slot;
  int32_t ctl;
};
constexpr int32_t kSegCtlPieceEnd = 1;
constexpr int32_t kSegCtlCombine = 2;
constexpr int32_t kSegCtlPair = 4;
static_assert(sizeof(SegHeader) == kSegHeaderBytes, "segment header is 32 bytes");
constexpr uint32_t kSegFirst = 1u << 31;
constexpr uint32_t kSegLast = 1u << 30;
constexpr uint32_t kSegPacked = 1u << 29;  // CSR: a run of whole short rows (see below)
constexpr uint32_t kSegRowMask = (1u << 29) - 1u;
// CSR segments, two plans:
//  long rows  -- every segment a slice of at most kCsrSegNnzLong nonzeros of
//                one row;
//  mixed rows -- runs of consecutive rows (at most kCsrSegNnzMixed nonzeros
//                and as many rows in all) packed into one segment
//                (kSegPacked; base = rows), and slices of at most
//                kCsrSegNnzMixed of the rows longer than that.
// A block is the header, for a packed segment its rows' starts relative to
// the segment (int16, rows + 1, padded to 16 bytes), the columns (padded to
// 16 bytes) and the values (padded to 16 bytes).
constexpr int kCsrSegNnzLong = 512;
constexpr int kCsrSegNnzMixed = 256;
constexpr int64_t csr_seg_bytes(int64_t nnz, int64_t packed_rows, int value_bytes) {
  return kSegHeaderBytes + (packed_rows ? delta_pad16((packed_rows + 1) * 2) : 0) +
         delta_pad16(nnz * 4) + delta_pad16(nnz * value_bytes);
}

// Tile descriptor (one int4 per work unit of the CSR kernel).
//   short-row tile: {row_begin, nnz_begin, nnz_end, KIND_STREAM | WALK? | lg << 16 | rows}
//                   (WALK: reduce by per-thread walk; else 2^lg lanes per row)
//   CTA-row tile:   {row,       nnz_begin, nnz_end, KIND_ROW}
//   split chunk:    {row,       nnz_begin, nnz_end, KIND_SPLIT | FIRST? | LAST? | split_id}
//                   (FIRST / LAST: the chunk is the row's first / last one)
constexpr uint32_t kKindShift = 30;
constexpr uint32_t kKindStream = 0u;
constexpr uint32_t kKindRow = 1u;
constexpr uint32_t kKindSplit = 2u;
constexpr uint32_t kRowsMask = 0xFFFFu;  // rows of a short-row tile
constexpr uint32_t kLanesShift = 16;     // log2(lanes per row), 4 bits (1..256 lanes)
constexpr uint32_t kStreamWalk = 1u << 20;
constexpr uint32_t kSplitFirst = 1u << 29;
constexpr uint32_t kSplitLast = 1u << 28;
constexpr uint32_t kSplitIdMask = (1u << 28) - 1u;

struct Tile {
  int32_t a, b, c, d;
};

// A row whose sum is assembled from partial sums.
//   CSR:    {first slot, chunks, row_ptr[row] (chunk k starts at row_begin +
//            k * per_chunk), nonzeros per chunk}
//   DELTA:  {first slot, pieces (warps whose shares hold part of the row),
//            0, 0}; a segment's header names its warp's piece
struct SplitInfo {
  int32_t first_slot;  // index of the first partial sum in the scratch array
  int32_t n_chunks;    // partial sums to wait for
  int32_t row_begin;
  int32_t reserved;
};

// Effective planner settings (defaults filled, limits applied).
struct Options {
  int tile_nnz;
  int tile_rows;
  int cta_row_min;
  int split_row_min;
  int split_chunk;
  int x_smem;  // -1 auto, 0 off, 1 on
  int reduce;  // short-row tiles: -1 per-tile choice, 0 lanes mode, 1 walk mode
  int lanes_log2;  // lanes mode when forced
  int interleave;  // CSR products: 0 auto, 1 chunks of 8, 2 element-interleaved
  int sell_sigma;  // SELL sorting window, 0: by the CV of the row lengths
  int csr_kernel;  // CSR: 0 auto, 1 CTA tiles, 2 warp segments (long rows), 3 mixed
  int delta_kernel;  // DELTA: 0 auto, 1 a lane per word, 2 several lanes per word (2/4-bit)
};

Options resolve_options(const spmv_plan_options* o, spmv_dtype dtype);

// Host-side result of planning a CSR matrix.
struct CsrTables {
  std::vector<Tile> tiles;
  std::vector<SplitInfo> splits;
  std::vector<int32_t> cta_first;  // CTA b runs tiles [cta_first[b], cta_first[b+1])
  int64_t n_chunks = 0;
};

// Cut the rows into work units and deal them to at most `max_ctas` CTAs as
// contiguous blocks of equal weight (nonzeros + rows).
spmv_status plan_csr_tiles(int n_rows, const int32_t* row_ptr,
                           const Options& opt, int max_ctas, CsrTables* out,
                           spmv_plan_info* info);

// One segment of a warp-segment plan (DELTA, or CSR with long rows), as the
// planner cuts it: a slice [begin, end) of one row's items (packed words for
// DELTA, nonzeros for CSR).
struct SegDesc {
  int32_t row;
  int32_t begin, end;
  int32_t base;      // DELTA: column before the first entry
  uint32_t flags;    // kSegFirst / kSegLast
  int32_t ctl = 0;   // kSegCtlPieceEnd / kSegCtlCombine
};

// Host-side result of cutting rows into segments and dealing them to warps.
struct SegTables {
  std::vector<SegDesc> segs;
  std::vector<int32_t> warp_first;  // warp g runs segments [warp_first[g], warp_first[g+1])
  std::vector<int32_t> seg_split;   // per segment: index into splits, or -1
  std::vector<int32_t> seg_slot;    // per segment of a split row: its warp's partial slot
  std::vector<SplitInfo> splits;    // {first_slot, pieces, 0, 0}
  std::vector<int32_t> empty_rows;  // rows without stored entries (y = 0)
  int64_t n_chunks = 0;             // partial-sum slots over all split rows
};

// Cut every row's items [row_begin(r), row_begin(r + 1)) into segments of at
// most `cap` (full ones first) and deal them to at most `max_warps` warps as
// contiguous shares of equal weight (items + seg_cost per segment).
spmv_status plan_segments(int32_t n_rows, const std::function<int64_t(int32_t)>& row_begin,
                          int64_t cap, int64_t seg_cost, int64_t entries_per_item,
                          int max_warps, int warps_per_cta, SegTables* out,
                          spmv_plan_info* info);
spmv_status plan_delta_segments(const spmv_delta* d, int max_warps, int warps_per_cta,
                                SegTables* out, spmv_plan_info* info);
spmv_status plan_csr_mixed_segments(const spmv_csr* m, int max_warps, int warps_per_cta,
                                    SegTables* out, spmv_plan_info* info);

// Device resources of a plan.
struct Plan {
  int device = -1;
  int sm_count = 0;
  spmv_format format = SPMV_FORMAT_CSR;
  spmv_dtype dtype = SPMV_F32;
  int n_rows = 0, n_cols = 0;
  int64_t nnz = 0, n_entries = 0;
  bool x_smem = false;
  int delta_bits = 4;          // DELTA: bits per column delta (2, 4 or 8)
  bool delta_skip_zero = false;  // DELTA: +0.0 entries (padding) read no x
  bool delta_wide = false;       // DELTA: several lanes per word (2- and 4-bit deltas)
  bool interleaved = false;  // CSR: products element-interleaved over the CTA
  bool csr_segments = false;  // CSR: warp-owned row segments
  bool csr_mixed = false;     // CSR segments: packed short rows + slices of long ones
  bool x_aligned16 = false;
  int grid = 0;
  size_t dyn_smem = 0;
  int64_t n_tiles = 0;
  int split_chunk = 0;

  // matrix (device)
  int32_t* row_ptr = nullptr;   // CSR offsets, DELTA entry offsets, SELL slot offsets
  int32_t* col_idx = nullptr;   // CSR and SELL columns
  void* values = nullptr;       // fp32 / fp16 (CSR, SELL)
  unsigned char* blocks = nullptr;  // DELTA: one block per segment
  int32_t* seg_off = nullptr;       // DELTA: block offsets (16-byte steps), n_segs + 1
  int32_t* empty_rows = nullptr;    // DELTA: rows without stored entries
  int32_t n_empty_rows = 0;
  // planner tables and scratch (device)
  Tile* tiles = nullptr;
  SplitInfo* splits = nullptr;
  int32_t* cta_first = nullptr;   // CSR: first tile per CTA; DELTA: first segment per warp
  int32_t* row_split = nullptr;
  int32_t* perm = nullptr;       // SELL: original row per slice lane (null: in order)
  // matrix-free FEM: elements per axis and the element matrix (the device
  // holds the densities in `values`)
  int fem_dims[3] = {0, 0, 0};
  // square fp32 plans: the matrix diagonal (Jacobi preconditioner) and the
  // conjugate-gradient workspace, allocated by the first solve
  float* diag = nullptr;
  unsigned char* pcg_work = nullptr;
  // captured batches of CG iterations (cudaGraphExec_t), one per batch
  // length, and the b, x and diag they were captured for
  static constexpr int kPcgGraphs = 3;
  void* pcg_exec[kPcgGraphs] = {nullptr, nullptr, nullptr};
  int pcg_batch[kPcgGraphs] = {0, 0, 0};
  const void* pcg_key[3] = {nullptr, nullptr, nullptr};
  // the whole iteration loop as one graph with a device-side while node
  // (cudaGraphExec_t), for the same b, x and diag as pcg_key
  void* pcg_loop = nullptr;
  bool pcg_loop_failed = false;
  float fem_k0[24 * 24] = {};
  float* partials = nullptr;    // one per split chunk
  int32_t* counters = nullptr;  // one per split row, zero between runs
  // segment plans: one exchange cell per split row, zero between runs
  unsigned long long* cells = nullptr;
  int32_t* status = nullptr;    // device status word
  // staging for spmv_run_host
  void* x_stage = nullptr;
  float* y_stage = nullptr;
  // spmv_run_host_batch: a second staging pair, the copy-in and copy-out
  // streams and, per staging slot, the events that order them (copy-in done,
  // product done, copy-out done); created on first use
  void* x_stage2 = nullptr;
  float* y_stage2 = nullptr;
  void* batch_streams[2] = {nullptr, nullptr};
  void* batch_events[7] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};

  spmv_plan_info info{};
};

// Kernel-side entry points (spmv_csr.cu, spmv_delta.cu).
int csr_kernel_occupancy(spmv_dtype dtype, bool x_smem, bool il, size_t dyn_smem,
                         size_t budget);
size_t csr_stage_bytes(spmv_dtype dtype);
int csr_set_smem_limit(size_t dyn);
int delta_warps_per_cta(int bits);      // warps of a DELTA CTA (each with its own ring)
// `wide`: the several-lanes-per-word kernel (2- and 4-bit deltas)
int delta_stages(int bits);              // ring depth per warp
int delta_grid_per_sm(int bits);         // CTAs per SM the grid uses (at most)
size_t delta_rings_bytes(int bits, bool wide);  // every stage of every warp of a CTA
size_t delta_x_smem_bytes(int n_cols);
int delta_set_smem_limit(int bits, bool wide, size_t dyn);
int delta_kernel_occupancy(int bits, bool wide, bool x_smem, size_t dyn_smem);
// `skip`: a device flag read at launch (after the kernels the launch depends
// on); when it is set the product is skipped (conjugate gradients, after
// convergence). nullptr for ordinary runs.
int launch_csr(const Plan& p, const void* x, float* y, void* stream, const int* skip = nullptr);
// CSR with warp-owned segments (spmv_csr_seg.cu), long-row or mixed plans.
int csr_seg_warps_per_cta(spmv_dtype dtype, bool mixed);
int csr_seg_stages(spmv_dtype dtype);
size_t csr_seg_rings_bytes(spmv_dtype dtype, bool mixed);
int csr_seg_set_smem_limit(size_t dyn);
int csr_seg_occupancy(spmv_dtype dtype, bool x_smem, bool mixed, size_t dyn_smem);
int launch_csr_seg(const Plan& p, const void* x, float* y, void* stream,
                   const int* skip = nullptr);
int launch_delta(const Plan& p, const void* x, float* y, void* stream);
// `dot` (SELL and FEM plans, square): when set, every CTA also writes its
// rows' x . y to dot[blockIdx] (the step length of conjugate gradients).
int launch_sell(const Plan& p, const void* x, float* y, void* stream, const int* skip = nullptr,
                float* dot = nullptr);
int launch_fem(const Plan& p, const void* x, float* y, void* stream, const int* skip = nullptr,
               float* dot = nullptr);
// Conjugate gradients (spmv_pcg.cu): workspace bytes for n unknowns, and one
// of its kernels (stage 0 init, 1 step length, 2 updates, 3 direction).
size_t pcg_work_bytes(int n, int product_grid);
// Whether the plan's product kernel can hand over p . q itself (SELL, FEM).
inline bool pcg_fused_dot(const Plan& p) {
  return p.format == SPMV_FORMAT_SELL || p.format == SPMV_FORMAT_FEM;
}
// `cond`: a conditional-node handle that the direction kernel sets to 0 once
// the solve is done and to 1 otherwise (0: no conditional node).
int launch_pcg(int stage, const Plan& p, const float* b, float* x, const float* diag,
               void* stream, unsigned long long cond = 0);

}  // namespace spmv
