// CSR kernel of y = A x for sm_103a (fp32 or fp16 values, int32 columns).
//
// CSR kernel: persistent CTAs walk contiguous blocks of the work units and
// stream each unit's column, value and row-pointer slices into shared memory
// with TMA bulk copies (cp.async.bulk + mbarrier), keeping kStages units in
// flight per CTA. Work units come from the host planner:
//   short-row tile  -- a run of consecutive rows (<= 2032 nonzeros): every
//                      thread multiplies 8 consecutive staged nonzeros by the
//                      gathered x; rows are then summed either by 2^lg lanes
//                      from shared memory (lanes mode, regular rows) or by a
//                      per-thread walk with carries across threads (walk
//                      mode, irregular rows) -- sub-warp / warp / CTA bins;
//   CTA-row tile    -- one row of up to 2048 nonzeros, CTA-wide reduction;
//   split chunk     -- a 2048-nonzero slice of a longer row; a CTA adds the
//                      consecutive chunks it owns in per-thread registers;
//                      a row shared by several CTAs is finished through
//                      plan-owned scratch by the CTA that completes it
//                      (atomic chunk count), in chunk order.
// Sources: "CUDA CSR SpMV optimisation" (codechina.net) 2.1 (row sum), 3.1
// (read-only path and shared-memory staging of x), 3.2 (vector loads), 4.1
// (warp per row with shuffle reduction); "Hash-based multi-phase SpGEMM"
// (mlqm.cn) 2.1.1 / 2.2 (rows binned to partial-warp, warp and block-per-row
// kernels); "MACKO-SpMV" (maplevalley.com.cn) 3.3 (splitting long rows).
//
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "spmv_device.cuh"
#include "spmv_internal.h"

namespace spmv {
namespace {

// x gathered through shared memory (staged) or the read-only path.
template <bool XS>
__device__ __forceinline__ float gather(const float* xg, const float* xs, int c) {
  return XS ? xs[c] : __ldg(xg + c);
}
template <bool XS>
__device__ __forceinline__ float gather(const __half* xg, const __half* xs, int c) {
  return __half2float(XS ? xs[c] : __ldg(xg + c));
}

// ------------------------------------------------------------ CSR kernel
struct CsrArgs {
  const int32_t* __restrict__ row_ptr;
  const int32_t* __restrict__ col;
  const void* __restrict__ val;
  const void* __restrict__ x;
  float* __restrict__ y;
  const int4* __restrict__ tiles;
  const int32_t* __restrict__ cta_first;
  int n_tiles;
  int n_cols;
  const SplitInfo* __restrict__ splits;
  float* partials;
  int32_t* counters;
  int split_chunk;
  int32_t* status;
  const int* skip;  // when set and nonzero at launch: do nothing (a finished solve)
};

// Shared-memory stage of one work unit: the columns and values of its
// nonzero span (aligned out to multiples of 8 elements) and, for a short-row
// tile, its row pointers (aligned out to multiples of 4).
template <typename VT>
struct Stage;
#ifndef SPMV_CSR_CTAS_F16
#define SPMV_CSR_CTAS_F16 6
#endif
#ifndef SPMV_CSR_CTAS_F32
#define SPMV_CSR_CTAS_F32 5
#endif
template <typename VT>
constexpr int kCsrCtasPerSm = sizeof(VT) == 2 ? SPMV_CSR_CTAS_F16 : SPMV_CSR_CTAS_F32;
template <typename VT>
struct Stage {
  static constexpr int kCap = sizeof(VT) == 2 ? kTileCapF16 : kTileCap;
  static constexpr int kColBytes = (kCap + 16) * 4;
  static constexpr int kValBytes = ((kCap + 16) * (int)sizeof(VT) + 15) / 16 * 16;
  static constexpr int kRpBytes = (kTileRowsCap + 8) * 4;
  static constexpr int kBytes = kColBytes + kValBytes + kRpBytes;
};

__device__ __forceinline__ bool is_sentinel(const int4& d) { return d.w == -1; }

// Thread 0: start the TMA copies of the work unit with descriptor d into a
// stage (valid == false marks the stage as the end of this CTA's work and
// completes its barrier phase).
template <typename VT>
__device__ __forceinline__ void issue_tile(const CsrArgs& a, unsigned char* stage,
                                           uint64_t* bar, int4* desc, bool valid,
                                           const int4 d, uint64_t pol) {
  if (!valid) {
    *desc = make_int4(0, 0, 0, -1);
    mbar_arrive(bar);
    return;
  }
  *desc = d;
  const int a0 = d.y & ~7, a1 = (d.z + 7) & ~7;
  const uint32_t ncol = (uint32_t)(a1 - a0) * 4u;
  const uint32_t nval = (uint32_t)(a1 - a0) * (uint32_t)sizeof(VT);
  uint32_t nrp = 0;
  int ra0 = 0;
  if (((uint32_t)d.w >> kKindShift) == kKindStream) {
    const int R = (int)((uint32_t)d.w & kRowsMask);
    ra0 = d.x & ~3;
    nrp = (uint32_t)((((d.x + R + 1) + 3) & ~3) - ra0) * 4u;
  }
  const uint32_t total = ncol + nval + nrp;
  if (total == 0) {
    mbar_arrive(bar);
    return;
  }
  mbar_arrive_expect_tx(bar, total);
  if (ncol) bulk_g2s(stage, a.col + a0, ncol, bar, pol);
  if (nval)
    bulk_g2s(stage + Stage<VT>::kColBytes, static_cast<const VT*>(a.val) + a0, nval, bar, pol);
  if (nrp)
    bulk_g2s(stage + Stage<VT>::kColBytes + Stage<VT>::kValBytes, a.row_ptr + ra0, nrp, bar,
             pol);
}

// Eight staged values starting at element 8c, widened to fp32.
__device__ __forceinline__ void stage_vals8(const float* v, int c, float (&o)[8]) {
  const float4 a = reinterpret_cast<const float4*>(v)[2 * c];
  const float4 b = reinterpret_cast<const float4*>(v)[2 * c + 1];
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void stage_vals8(const __half* v, int c, float (&o)[8]) {
  const uint4 a = reinterpret_cast<const uint4*>(v)[c];
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    __half2 p;
    *reinterpret_cast<uint32_t*>(&p) = w[h];
    const float2 f = __half22float2(p);
    o[2 * h] = f.x;
    o[2 * h + 1] = f.y;
  }
}

// Products of the 8 staged nonzeros of chunk c (elements outside
// [lo_rel, hi_rel) give 0 and gather nothing).
template <typename VT, typename XT, bool XS>
__device__ __forceinline__ void chunk_products(const int* s_col, const VT* s_val, int c,
                                               int lo_rel, int hi_rel, const XT* xg,
                                               const XT* xs, float (&p)[8]) {
  const int4 c0 = reinterpret_cast<const int4*>(s_col)[2 * c];
  const int4 c1 = reinterpret_cast<const int4*>(s_col)[2 * c + 1];
  const int cols[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  float v[8];
  stage_vals8(s_val, c, v);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int el = 8 * c + q;
    p[q] = (el >= lo_rel && el < hi_rel) ? v[q] * gather<XS>(xg, xs, cols[q]) : 0.f;
  }
}

// Value of staged element el, widened to fp32.
__device__ __forceinline__ float staged_val(const float* v, int el) { return v[el]; }
__device__ __forceinline__ float staged_val(const __half* v, int el) {
  return __half2float(v[el]);
}

// Staged element el of thread t, step k < 8, element-interleaved over the
// CTA: a warp-wide step spans 32 consecutive nonzeros, so its x gathers fall
// in few sectors.
__device__ __forceinline__ int strided_el(int base, int k) {
  return base + (int)threadIdx.x + kThreads * k;
}

// Products of the staged elements strided_el(base, k), k < 8 (0 outside
// [lo_rel, hi_rel)). All eight gathers are issued before any product is used.
template <typename VT, typename XT, bool XS>
__device__ __forceinline__ void strided_products(const int* s_col, const VT* s_val, int base,
                                                 int lo_rel, int hi_rel, const XT* xg,
                                                 const XT* xs, float (&p)[8]) {
  float xv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int el = strided_el(base, k);
    xv[k] = (el >= lo_rel && el < hi_rel) ? gather<XS>(xg, xs, s_col[el]) : 0.f;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int el = strided_el(base, k);
    p[k] = (el >= lo_rel && el < hi_rel) ? staged_val(s_val, el) * xv[k] : 0.f;
  }
}

// Short-row tile from a stage, lanes mode (rows of similar length): every
// thread multiplies its 8 staged nonzeros by the gathered x and parks the
// products in place of the staged columns; then each row is summed by
// g = 2^lg lanes and a shuffle reduction (g = 64..256: by g / 32 warps, whose
// sums meet in shared memory).
template <typename VT, typename XT, bool XS, bool IL>
__device__ __forceinline__ void stream_tile_lanes(const CsrArgs& a, const int4 d,
                                                  unsigned char* stage, const XT* xs,
                                                  float* s_red) {
  const int tid = threadIdx.x;
  const int r0 = d.x, s = d.y, e = d.z;
  const int R = (int)((uint32_t)d.w & kRowsMask);
  const int lg = (int)(((uint32_t)d.w >> kLanesShift) & 15u);
  const int a0 = s & ~7;
  const int s_rel = s - a0, e_rel = e - a0;
  const int n8 = (e_rel + 7) >> 3;
  int* s_col = reinterpret_cast<int*>(stage);
  const VT* s_val = reinterpret_cast<const VT*>(stage + Stage<VT>::kColBytes);
  const int* s_rp =
      reinterpret_cast<const int*>(stage + Stage<VT>::kColBytes + Stage<VT>::kValBytes) +
      (r0 - (r0 & ~3));
  float* s_prod = reinterpret_cast<float*>(s_col);  // products replace the columns
  const XT* xg = static_cast<const XT*>(a.x);
  if (IL) {
    // the tile spans at most kThreads * 8 elements; each thread replaces
    // exactly the columns it read with their products
    float p[8];
    strided_products<VT, XT, XS>(s_col, s_val, 0, s_rel, e_rel, xg, xs, p);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int el = strided_el(0, k);
      if (el < e_rel) s_prod[el] = p[k];
    }
  } else {
    for (int c = tid; c < n8; c += kThreads) {
      float p[8];
      chunk_products<VT, XT, XS>(s_col, s_val, c, s_rel, e_rel, xg, xs, p);
      reinterpret_cast<float4*>(s_prod)[2 * c] = make_float4(p[0], p[1], p[2], p[3]);
      reinterpret_cast<float4*>(s_prod)[2 * c + 1] = make_float4(p[4], p[5], p[6], p[7]);
    }
  }
  __syncthreads();
  const int g = 1 << lg;
  const int per_pass = kThreads >> lg;
  const int grp = tid >> lg, lig = tid & (g - 1);
  for (int base = 0; base < R; base += per_pass) {
    const int r = base + grp;
    float acc = 0.f;
    if (r < R) {
      const int b = s_rp[r] - a0, en = s_rp[r + 1] - a0;
#pragma unroll 4
      for (int i = b + lig; i < en; i += g) acc += s_prod[i];
    }
    if (lg <= 5) {
      for (int o = g >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lig == 0 && r < R) a.y[r0 + r] = acc;
    } else {  // a group of g / 32 warps per row: warp sums, then the group's first thread
      acc = warp_sum(acc);
      if ((tid & 31) == 0) s_red[tid >> 5] = acc;
      __syncthreads();
      if (lig == 0 && r < R) {
        float t = 0.f;
        for (int w = 0; w < (g >> 5); ++w) t += s_red[(tid >> 5) + w];
        a.y[r0 + r] = t;
      }
      __syncthreads();
    }
  }
}

// Short-row tile from a stage, walk mode (rows of any lengths): rows
// [r0, r0+R), nonzeros [s, e). Thread t owns the 8 staged nonzeros [8t, 8t+8) (stage-relative; the stage
// starts at s rounded down to 8) and keeps their products in registers. It
// finds the row of its first nonzero by binary search over the staged row
// pointers and walks its 8 nonzeros: a row that starts and ends inside its
// range is written to y at once; the partial of a row that continues past
// its range is a carry; the thread where a row that began in an earlier
// thread ends adds the carries of the threads the row spans, which a
// segmented scan over the CTA (shuffles within warps, warp totals through
// shared memory) has summed. Rows without nonzeros are written as 0 by a
// separate pass. Work per thread is bounded whatever the row lengths are.
template <typename VT, typename XT, bool XS>
__device__ __forceinline__ void stream_tile_walk(const CsrArgs& a, const int4 d,
                                                 unsigned char* stage, const XT* xs,
                                                 float* s_carry) {
  const int tid = threadIdx.x;
  const int r0 = d.x, s = d.y, e = d.z;
  const int R = (int)((uint32_t)d.w & kRowsMask);
  const int a0 = s & ~7;
  const int s_rel = s - a0, e_rel = e - a0;
  const int* s_col = reinterpret_cast<const int*>(stage);
  const VT* s_val = reinterpret_cast<const VT*>(stage + Stage<VT>::kColBytes);
  // B[r] = row_ptr[r0 + r] - a0, for r in [0, R]
  const int* s_rp =
      reinterpret_cast<const int*>(stage + Stage<VT>::kColBytes + Stage<VT>::kValBytes) +
      (r0 - (r0 & ~3));
  const XT* xg = static_cast<const XT*>(a.x);
  float* y = a.y + r0;

  const int lo = max(8 * tid, s_rel), hi = min(8 * tid + 8, e_rel);
  // Carries: a row that runs past this thread's nonzeros leaves its partial
  // sum in v; head is false only for a thread that lies wholly inside a row
  // begun by an earlier thread. A segmented inclusive scan of (v, head) over
  // the CTA then hands a thread that ends such a row the sum of that row's
  // carries, in a fixed order and in O(log) steps whatever the row's length.
  float v = 0.f;
  bool head = true;
  bool closes = false;  // this thread ends a row that began in an earlier thread
  int close_row = 0;
  float close_val = 0.f;
  if (lo < hi) {
    float p[8];
    chunk_products<VT, XT, XS>(s_col, s_val, tid, s_rel, e_rel, xg, xs, p);
    // row containing nonzero lo: the largest r < R with B[r] <= lo
    int l = 0, h = R - 1;
    while (l < h) {
      const int mid = (l + h + 1) >> 1;
      if (s_rp[mid] - a0 <= lo)
        l = mid;
      else
        h = mid - 1;
    }
    int row = l;
    int row_end = s_rp[row + 1] - a0;
    bool inside = (s_rp[row] - a0) >= lo;
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = 8 * tid + q;
      if (j >= lo && j < hi) {
        if (j >= row_end) {  // the current row ended just before j
          if (inside) {
            y[row] = acc;
          } else {
            closes = true;
            close_row = row;
            close_val = acc;
          }
          do {
            ++row;
            row_end = s_rp[row + 1] - a0;
          } while (row_end <= j);  // skip rows without nonzeros
          inside = true;
          acc = 0.f;
        }
        acc += p[q];
      }
    }
    if (row_end > hi) {  // the row goes on in the next thread(s)
      v = acc;
      head = inside;
    } else if (inside) {
      y[row] = acc;
    } else {
      closes = true;
      close_row = row;
      close_val = acc;
    }
  }
  for (int r = tid; r < R; r += kThreads)
    if (s_rp[r] == s_rp[r + 1]) y[r] = 0.f;
  // warp-level segmented scan: (u, hu) (+) (v, h) = (h ? v : u + v, hu | h)
  const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
  for (int dd = 1; dd < 32; dd <<= 1) {
    const float uv = __shfl_up_sync(0xffffffffu, v, dd);
    const int uh = __shfl_up_sync(0xffffffffu, head ? 1 : 0, dd);
    if (lane >= dd && !head) {
      v += uv;
      head = uh != 0;
    }
  }
  int* s_head = reinterpret_cast<int*>(s_carry + kWarps);
  if (lane == 31) {
    s_carry[wid] = v;
    s_head[wid] = head ? 1 : 0;
  }
  __syncthreads();
  // the scan's value entering this warp: earlier warps' totals, segmented
  float pv = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < kWarps; ++w2)
    if (w2 < wid) pv = s_head[w2] ? s_carry[w2] : pv + s_carry[w2];
  const float full = head ? v : v + pv;
  float before = __shfl_up_sync(0xffffffffu, full, 1);
  if (lane == 0) before = pv;
  if (closes) y[close_row] = before + close_val;
}

// Checked builds: before a staged unit is used, every column is tested
// against n_cols and every staged row offset of a short-row tile is clamped
// into the tile's nonzeros (the first and last exactly to its ends), so a
// corrupt index can neither gather outside x nor walk outside the stage.
template <typename VT>
__device__ __noinline__ void check_stage(const CsrArgs& a, const int4 d, unsigned char* stage) {
  bool bad = false;
  const int a0 = d.y & ~7;
  int* s_col = reinterpret_cast<int*>(stage);
  for (int el = d.y - a0 + (int)threadIdx.x; el < d.z - a0; el += kThreads)
    s_col[el] = checked_col(s_col[el], a.n_cols, &bad);
  if (((uint32_t)d.w >> kKindShift) == kKindStream) {
    const int R = (int)((uint32_t)d.w & kRowsMask);
    int* s_rp = reinterpret_cast<int*>(stage + Stage<VT>::kColBytes + Stage<VT>::kValBytes) +
                (d.x - (d.x & ~3));
    for (int r = threadIdx.x; r <= R; r += kThreads) {
      const int v = checked_offset(s_rp[r], d.y, d.z, &bad);
      s_rp[r] = r == 0 ? d.y : r == R ? d.z : v;
      if ((r == 0 && v != d.y) || (r == R && v != d.z)) bad = true;
    }
  }
  if (bad) atomicExch(a.status, kStatusBadIndex);
  __syncthreads();
}

// Per-thread partial sum of a staged slice [b, e) of one row.
template <typename VT, typename XT, bool XS, bool IL>
__device__ __forceinline__ float chunk_sum(const CsrArgs& a, const int4 d,
                                           unsigned char* stage, const XT* xs) {
  const int a0 = d.y & ~7;
  const int lo_rel = d.y - a0, hi_rel = d.z - a0;
  const int n8 = (hi_rel + 7) >> 3;
  const int* s_col = reinterpret_cast<const int*>(stage);
  const VT* s_val = reinterpret_cast<const VT*>(stage + Stage<VT>::kColBytes);
  const XT* xg = static_cast<const XT*>(a.x);
  float acc = 0.f;
  if (IL) {
    for (int base = 0; base < hi_rel; base += 8 * kThreads) {
      float p[8];
      strided_products<VT, XT, XS>(s_col, s_val, base, lo_rel, hi_rel, xg, xs, p);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc += p[q];
    }
  } else {
    for (int c = threadIdx.x; c < n8; c += kThreads) {
      float p[8];
      chunk_products<VT, XT, XS>(s_col, s_val, c, lo_rel, hi_rel, xg, xs, p);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc += p[q];
    }
  }
  return acc;
}

// Thread 0, at the end of this CTA's piece of split row `row` (its chunks
// starting at nonzero b0 and ending with the chunk that starts at b): if the
// piece is the whole row, write y; otherwise publish the piece's partial at
// the slot of its first chunk and count its chunks. The CTA that completes the
// count adds all slots of the row in chunk order (slots of other pieces'
// interior chunks hold 0), writes y, and clears the slots and the counter for
// the next run. Only rows that cross a CTA boundary take this path.
__device__ __forceinline__ void split_publish(const CsrArgs& a, int row, int sid,
                                              bool whole, int b0, int b, float part) {
  if (whole) {
    a.y[row] = part;
    return;
  }
  const SplitInfo si = a.splits[sid];
  const int k0 = (b0 - si.row_begin) / si.reserved;
  const int k = (b - si.row_begin) / si.reserved;
  a.partials[si.first_slot + k0] = part;
  __threadfence();
  const int add = k - k0 + 1;
  const int before = atomicAdd(a.counters + sid, add);
  if (before + add == si.n_chunks) {
    __threadfence();
    float sum = 0.f;
    for (int j = 0; j < si.n_chunks; ++j) {
      sum += __ldcg(a.partials + si.first_slot + j);
      a.partials[si.first_slot + j] = 0.f;
    }
    a.y[row] = sum;
    a.counters[sid] = 0;
  }
}

// Persistent CSR kernel: each CTA walks its contiguous block of work units;
// thread 0 keeps kStages units in flight (TMA bulk copies into a ring of shared
// memory stages) while the CTA computes the oldest one.
// Register budget: as many CTAs per SM as the planner's shared-memory budget
// lets in (5 with fp32 stages, 6 with fp16 ones).
template <typename VT, typename XT, bool XS, bool IL>
__global__ void __launch_bounds__(kThreads, kCsrCtasPerSm<VT>) csr_kernel(const CsrArgs a) {
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  __shared__ __align__(8) uint64_t s_bar[kStages];
  __shared__ int4 s_desc[kStages];
  __shared__ float s_red[kWarps];
  __shared__ float s_carry[2 * kWarps];  // walk mode: warp totals and head flags
  unsigned char* stages = dyn_smem;
  // this CTA's contiguous block of work units (equal weight per CTA)
  const int u_begin = __ldg(a.cta_first + blockIdx.x);
  const int u_end = __ldg(a.cta_first + blockIdx.x + 1);
  XT* xs = reinterpret_cast<XT*>(dyn_smem + kStages * Stage<VT>::kBytes);
  const int tid = threadIdx.x;
  uint64_t pol = 0;
  int4 next_d = make_int4(0, 0, 0, 0);  // thread 0: descriptor of the next unit to issue
  int next_u = u_begin;                 // thread 0: that unit
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&s_bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    pol = policy_evict_first();
    int4 d0[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s)
      d0[s] = next_u + s < u_end ? __ldg(a.tiles + next_u + s) : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int s = 0; s < kStages; ++s)
      issue_tile<VT>(a, stages + s * Stage<VT>::kBytes, &s_bar[s], &s_desc[s],
                     next_u + s < u_end, d0[s], pol);
    next_u += kStages;
    // the descriptor for the next refill is loaded one unit ahead, so the
    // refill never waits for it
    if (next_u < u_end) next_d = __ldg(a.tiles + next_u);
    pdl_launch_dependents();
  }
  // Everything above reads only plan-owned data (tiles and the matrix, which
  // no kernel writes); x, y and the split scratch are touched only after the
  // kernels this launch depends on have completed.
  pdl_wait();
  if (a.skip && *a.skip) {  // let the copies issued above land, then leave
    if (tid == 0)
      for (int s = 0; s < kStages; ++s) mbar_wait_bounded(&s_bar[s], 0u);
    return;
  }
  if (XS) stage_x<XT>(xs, static_cast<const XT*>(a.x), a.n_cols);
  bool aborted = false;
  float row_acc = 0.f;  // this thread's share of the current split-row piece
  int piece_b0 = -1;    // first nonzero of that piece, -1 when none is open
  bool piece_first = false;
  int i = 0;  // work units consumed; each consumption re-issues its stage
  for (;; ++i) {
    const int s = i % kStages;
    const uint32_t parity = (uint32_t)(i / kStages) & 1u;
    const bool ok = mbar_wait_bounded(&s_bar[s], parity);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const int4 d = s_desc[s];
    if (is_sentinel(d)) break;
    unsigned char* stage = stages + s * Stage<VT>::kBytes;
    const uint32_t w = (uint32_t)d.w;
    const uint32_t kind = w >> kKindShift;
    if (kChecked) check_stage<VT>(a, d, stage);
    if (kind == kKindStream) {
      if (w & kStreamWalk)
        stream_tile_walk<VT, XT, XS>(a, d, stage, xs, s_carry);
      else
        stream_tile_lanes<VT, XT, XS, IL>(a, d, stage, xs, s_red);
    } else if (kind == kKindRow) {
      const float part = cta_sum(chunk_sum<VT, XT, XS, IL>(a, d, stage, xs), s_red);
      if (tid == 0) a.y[d.x] = part;
    } else {
      if (piece_b0 < 0) {
        piece_b0 = d.y;
        piece_first = (w & kSplitFirst) != 0;
      }
      row_acc += chunk_sum<VT, XT, XS, IL>(a, d, stage, xs);
      const bool last = (w & kSplitLast) != 0;
      if (last || u_begin + i == u_end - 1) {  // row ends, or this CTA's share does
        const float part = cta_sum(row_acc, s_red);
        if (tid == 0)
          split_publish(a, d.x, (int)(w & kSplitIdMask), piece_first && last, piece_b0, d.y,
                        part);
        row_acc = 0.f;
        piece_b0 = -1;
      }
    }
    __syncthreads();  // stage s is free again
    if (tid == 0) {
      fence_proxy_async_smem();
      const bool valid = next_u < u_end;
      issue_tile<VT>(a, stage, &s_bar[s], &s_desc[s], valid, next_d, pol);
      ++next_u;
      if (next_u < u_end) next_d = __ldg(a.tiles + next_u);
    }
  }
  if (tid == 0 && aborted) {
    atomicExch(a.status, 1);
    // let copies still in flight land before the CTA's shared memory goes:
    // stage s was filled 1 + #{j < i : j % kStages == s} times
    for (int s = 0; s < kStages; ++s) {
      const int fills = 1 + (i > s ? (i - 1 - s) / kStages + 1 : 0);
      mbar_wait_bounded(&s_bar[s], (uint32_t)(fills - 1) & 1u);
    }
  }
}

template <typename VT, typename XT, bool XS>
const void* csr_fn(bool il) {
  return il ? reinterpret_cast<const void*>(&csr_kernel<VT, XT, XS, true>)
            : reinterpret_cast<const void*>(&csr_kernel<VT, XT, XS, false>);
}

template <typename VT>
constexpr size_t stage_bytes() {
  return (size_t)Stage<VT>::kBytes;
}

const void* csr_entry(spmv_dtype dt, bool xs, bool il) {
  if (dt == SPMV_F32)
    return xs ? csr_fn<float, float, true>(il) : csr_fn<float, float, false>(il);
  return xs ? csr_fn<__half, __half, true>(il) : csr_fn<__half, __half, false>(il);
}

}  // namespace

int csr_kernel_occupancy(spmv_dtype dtype, bool x_smem, bool il, size_t dyn_smem,
                         size_t budget) {
  return occupancy_within(csr_entry(dtype, x_smem, il), kThreads, dyn_smem, budget);
}

size_t csr_stage_bytes(spmv_dtype dtype) {
  return dtype == SPMV_F32 ? stage_bytes<float>() : stage_bytes<__half>();
}

int csr_set_smem_limit(size_t dyn) {
  if (dyn == 0) return 0;
  for (spmv_dtype dt : {SPMV_F32, SPMV_F16})
    for (bool xs : {false, true})
      for (bool il : {false, true})
        if (cudaFuncSetAttribute(csr_entry(dt, xs, il), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dyn) != cudaSuccess)
          return -1;
  return 0;
}

int launch_csr(const Plan& p, const void* x, float* y, void* stream, const int* skip) {
  if (p.n_tiles == 0) return 0;
  CsrArgs a;
  a.skip = skip;
  a.row_ptr = p.row_ptr;
  a.col = p.col_idx;
  a.val = p.values;
  a.x = x;
  a.y = y;
  a.tiles = reinterpret_cast<const int4*>(p.tiles);
  a.cta_first = p.cta_first;
  a.n_tiles = (int)p.n_tiles;
  a.n_cols = p.n_cols;
  a.splits = p.splits;
  a.partials = p.partials;
  a.counters = p.counters;
  a.split_chunk = p.split_chunk;
  a.status = p.status;
  void* args[] = {&a};
  return launch_pdl(csr_entry(p.dtype, p.x_smem, p.interleaved), p.grid, kThreads, p.dyn_smem,
                    stream, args);
}

}  // namespace spmv
