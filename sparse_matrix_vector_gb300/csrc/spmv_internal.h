// Internal declarations shared by the host planner (spmv_host.cpp) and the
// device kernels (spmv_kernels.cu). Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "../../include/spmv.h"

namespace spmv {

// ---------------------------------------------------------------- geometry
constexpr int kThreads = 256;            // CTA size of every kernel
constexpr int kWarps = kThreads / 32;
constexpr int kVec = 4;                  // col_idx elements per 16-byte load
constexpr int kStreamVecs = 2;           // 4-element vectors per thread per tile
// A short-row tile holds at most this many nonzeros: its aligned span of
// kVec-element vectors must fit kThreads * kStreamVecs vectors.
constexpr int kMaxTileNnz = kThreads * kVec * kStreamVecs - (kVec - 1);
constexpr int kMaxTileRows = 1024;       // row offsets staged in shared memory
constexpr int kProdCap = kThreads * kVec * kStreamVecs;  // products per tile
constexpr int kRowUnroll = 2;            // vectors in flight per thread, long rows
constexpr int kDeltaWordsPerRound = kThreads;  // one 32-bit delta word per thread

// Tile descriptor (one int4 per work unit of the CSR kernel).
//   short-row tile: {row_begin, nnz_begin, nnz_end, KIND_STREAM | lg << 16 | rows}
//   CTA-row tile:   {row,       nnz_begin, nnz_end, KIND_ROW}
//   split chunk:    {row,       nnz_begin, nnz_end, KIND_SPLIT | split_id}
constexpr uint32_t kKindShift = 30;
constexpr uint32_t kKindStream = 0u;
constexpr uint32_t kKindRow = 1u;
constexpr uint32_t kKindSplit = 2u;
constexpr uint32_t kLanesShift = 16;     // log2(lanes per row), 3 bits
constexpr uint32_t kRowsMask = 0xFFFFu;  // rows of a short-row tile
constexpr uint32_t kSplitIdMask = (1u << kKindShift) - 1u;

struct Tile {
  int32_t a, b, c, d;
};

struct SplitInfo {
  int32_t first_slot;  // index of chunk 0's partial sum in the scratch array
  int32_t n_chunks;
};

// Effective planner settings (defaults filled, limits applied).
struct Options {
  int tile_nnz;
  int tile_rows;
  int cta_row_min;
  int split_row_min;
  int split_chunk;
  int x_smem;  // -1 auto, 0 off, 1 on
  int lanes;   // 0 auto
};

Options resolve_options(const spmv_plan_options* o);

// Host-side result of planning a CSR matrix.
struct CsrTables {
  std::vector<Tile> tiles;
  std::vector<SplitInfo> splits;
  int64_t n_chunks = 0;
};

spmv_status plan_csr_tiles(int n_rows, const int32_t* row_ptr,
                           const Options& opt, CsrTables* out,
                           spmv_plan_info* info);

// Device resources of a plan.
struct Plan {
  int device = -1;
  int sm_count = 0;
  spmv_format format = SPMV_FORMAT_CSR;
  spmv_dtype dtype = SPMV_F32;
  int n_rows = 0, n_cols = 0;
  int64_t nnz = 0, n_entries = 0;
  bool x_smem = false;
  bool x_aligned16 = false;
  int grid = 0;
  size_t dyn_smem = 0;
  int64_t n_tiles = 0;
  int split_chunk = 0;

  // matrix (device)
  int32_t* row_ptr = nullptr;   // CSR offsets or DELTA4 entry offsets
  int32_t* col_idx = nullptr;   // CSR only
  void* values = nullptr;       // fp32 / fp16 (CSR) or fp16 (DELTA4)
  uint32_t* words = nullptr;    // DELTA4 packed deltas
  // planner tables and scratch (device)
  Tile* tiles = nullptr;
  SplitInfo* splits = nullptr;
  float* partials = nullptr;    // one per split chunk
  int32_t* counters = nullptr;  // one per split row, zero between runs
  int32_t* status = nullptr;    // device status word
  // staging for spmv_run_host
  void* x_stage = nullptr;
  float* y_stage = nullptr;

  spmv_plan_info info{};
};

// Kernel-side entry points (spmv_kernels.cu).
int csr_kernel_occupancy(spmv_dtype dtype, bool x_smem, size_t dyn_smem);
int delta_kernel_occupancy(bool x_smem, size_t dyn_smem);
int set_kernel_smem_limits(size_t csr_dyn, size_t delta_dyn);
int launch_csr(const Plan& p, const void* x, float* y, void* stream);
int launch_delta(const Plan& p, const void* x, float* y, void* stream);

}  // namespace spmv
