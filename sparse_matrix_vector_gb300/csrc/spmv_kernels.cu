// Device half of the library: the sm_103a kernels of y = A x.
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
// DELTA4 kernel ("MACKO-SpMV" 2.2): persistent like the CSR kernel; a work
// unit is a slice of one row (at most 512 packed words = 4096 entries) whose
// starting column, and each warp's starting column in it, the planner
// stored, so units and warps are independent. Lane l of warp w decodes two
// words: a per-lane sum of their 16 nibbles and a 5-step __shfl_up_sync
// inclusive scan give the column before its first entry; products are taken
// in half2 (__hmul2) and accumulated in fp32 per row across units.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// CTA-wide sum; the result is valid in thread 0. Fixed order.
__device__ __forceinline__ float cta_sum(float v, float* s_red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (warp == 0) {
    t = lane < kWarps ? s_red[lane] : 0.f;
    t = warp_sum(t);
  }
  return t;
}

// Sum over a block of NW warps; the result is valid in thread 0. Fixed order.
template <int NW>
__device__ __forceinline__ float block_sum(float v, float* s_red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (warp == 0) {
    t = lane < NW ? s_red[lane] : 0.f;
    t = warp_sum(t);
  }
  return t;
}

// Copy x (n elements) into shared memory, 16 bytes at a time when aligned.
template <typename XT>
__device__ __forceinline__ void stage_x(XT* xs, const XT* x, int n) {
  if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
    const int nv = (int)(((size_t)n * sizeof(XT)) >> 4);
    const int4* src = reinterpret_cast<const int4*>(x);
    int4* dst = reinterpret_cast<int4*>(xs);
    for (int i = threadIdx.x; i < nv; i += kThreads) dst[i] = __ldg(src + i);
    for (int i = nv * (int)(16 / sizeof(XT)) + threadIdx.x; i < n; i += kThreads)
      xs[i] = x[i];
  } else {
    for (int i = threadIdx.x; i < n; i += kThreads) xs[i] = x[i];
  }
  __syncthreads();
}

// ------------------------------------------------------------ TMA / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Every wait on a barrier gives up after this many polls (each poll may
// itself suspend the thread for a while): the kernel then records an error
// in the plan's status word instead of hanging.
constexpr uint32_t kWaitPolls = 1u << 22;

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Order this thread's earlier generic-proxy accesses to shared memory before
// later async-proxy (TMA) writes to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: let the next kernel on the stream start its
// prologue, and wait until every kernel this one depends on has finished and
// its memory is visible (a no-op when launched without the attribute).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes and both
// addresses are multiples of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
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

// Short-row tile from a stage, lanes mode (rows of similar length): every
// thread multiplies its 8 staged nonzeros by the gathered x and parks the
// products in place of the staged columns; then each row is summed by
// g = 2^lg lanes and a shuffle reduction (g = 64..256: by g / 32 warps, whose
// sums meet in shared memory).
template <typename VT, typename XT, bool XS>
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
  for (int c = tid; c < n8; c += kThreads) {
    float p[8];
    chunk_products<VT, XT, XS>(s_col, s_val, c, s_rel, e_rel, xg, xs, p);
    reinterpret_cast<float4*>(s_prod)[2 * c] = make_float4(p[0], p[1], p[2], p[3]);
    reinterpret_cast<float4*>(s_prod)[2 * c + 1] = make_float4(p[4], p[5], p[6], p[7]);
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

// Per-thread partial sum of a staged slice [b, e) of one row.
template <typename VT, typename XT, bool XS>
__device__ __forceinline__ float chunk_sum(const CsrArgs& a, const int4 d,
                                           unsigned char* stage, const XT* xs) {
  const int a0 = d.y & ~7;
  const int lo_rel = d.y - a0, hi_rel = d.z - a0;
  const int n8 = (hi_rel + 7) >> 3;
  const int* s_col = reinterpret_cast<const int*>(stage);
  const VT* s_val = reinterpret_cast<const VT*>(stage + Stage<VT>::kColBytes);
  const XT* xg = static_cast<const XT*>(a.x);
  float acc = 0.f;
  for (int c = threadIdx.x; c < n8; c += kThreads) {
    float p[8];
    chunk_products<VT, XT, XS>(s_col, s_val, c, lo_rel, hi_rel, xg, xs, p);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc += p[q];
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
template <typename VT, typename XT, bool XS>
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
    if (kind == kKindStream) {
      if (w & kStreamWalk)
        stream_tile_walk<VT, XT, XS>(a, d, stage, xs, s_carry);
      else
        stream_tile_lanes<VT, XT, XS>(a, d, stage, xs, s_red);
    } else if (kind == kKindRow) {
      const float part = cta_sum(chunk_sum<VT, XT, XS>(a, d, stage, xs), s_red);
      if (tid == 0) a.y[d.x] = part;
    } else {
      if (piece_b0 < 0) {
        piece_b0 = d.y;
        piece_first = (w & kSplitFirst) != 0;
      }
      row_acc += chunk_sum<VT, XT, XS>(a, d, stage, xs);
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

// ------------------------------------------------------------ DELTA4 kernel
struct DeltaArgs {
  const uint32_t* __restrict__ words;   // 8 nibbles per word
  const __half* __restrict__ vals;      // 8 fp16 values per word, 16 bytes
  const __half* __restrict__ x;
  float* __restrict__ y;
  const int4* __restrict__ units;       // {row | FIRST | LAST, wb, we, column base}
  const int32_t* __restrict__ warp_base;  // kDeltaWarps starting columns per unit
  const int32_t* __restrict__ cta_first;
  const int32_t* __restrict__ row_split;
  const SplitInfo* __restrict__ splits;  // {first_slot, n_units, row word, words/unit}
  float* partials;
  int32_t* counters;
  int32_t* status;
  int n_cols;
};

// Shared-memory stage of one DELTA4 unit: the warps' starting columns, the
// unit's words (aligned out to 4 words) and its values (16 bytes per word).
struct DeltaStage {
  static constexpr int kBaseBytes = kDeltaWarps * 4;
  static constexpr int kWordBytes = (kDeltaUnitWords + 8) * 4;
  static constexpr int kValBytes = kDeltaUnitWords * 16;
  static constexpr int kBytes = kBaseBytes + kWordBytes + kValBytes;
};
static_assert(DeltaStage::kBaseBytes % 16 == 0, "stage regions must stay 16-byte aligned");

// x in shared memory, skewed by one 4-byte word per 128 bytes: lanes that
// gather at a 64-byte stride (16 entries per lane at 50% density) then hit
// distinct banks. Half i lives at i + 2 * (i / 64).
// Skewed copy of x (half i at i + 2 * (i / 64)) for the CTA-barrier kernel,
// whose lanes gather 64 bytes apart at 50% density; the producer / consumer
// kernel measured best on the plain copy (SPMV_X_SKEW 0 there).
#ifndef SPMV_X_SKEW
#define SPMV_X_SKEW 0
#endif
__device__ __forceinline__ int x_skew(int i) { return SPMV_X_SKEW ? i + 2 * (i >> 6) : i; }

__device__ __forceinline__ void stage_x_skewed(__half* xs, const __half* x, int n,
                                               bool sync = true, int nthreads = kDeltaThreads) {
  uint32_t* dst = reinterpret_cast<uint32_t*>(xs);
  const int pairs = n >> 1;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
    const uint4* src = reinterpret_cast<const uint4*>(x);
    for (int v = threadIdx.x; v < (pairs >> 2); v += nthreads) {
      const uint4 q = __ldg(src + v);
      const int j = 4 * v;  // first pair of the vector; 4 pairs never cross a 32-pair row
      const int o = SPMV_X_SKEW ? j + (j >> 5) : j;
      dst[o] = q.x;
      dst[o + 1] = q.y;
      dst[o + 2] = q.z;
      dst[o + 3] = q.w;
    }
    for (int i = ((pairs >> 2) << 3) + threadIdx.x; i < n; i += nthreads) xs[x_skew(i)] = x[i];
  } else {
    for (int i = threadIdx.x; i < n; i += nthreads) xs[x_skew(i)] = x[i];
  }
  if (sync) __syncthreads();
}

// Sum of the eight 4-bit fields of w (<= 120).
__device__ __forceinline__ int nibble_sum(uint32_t w) {
  const uint32_t b = (w & 0x0F0F0F0Fu) + ((w >> 4) & 0x0F0F0F0Fu);
  return (int)((b * 0x01010101u) >> 24);
}

// acc + (float)h, one fp32 rounding (mixed-precision add, f16 operand).
__device__ __forceinline__ float add_f16(float acc, __half h) {
  asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(__half_as_ushort(h)));
  return acc;
}

template <bool XS>
__device__ __forceinline__ __half gather_h(const __half* xg, const __half* xs, int c) {
  return XS ? xs[x_skew(c)] : __ldg(xg + c);
}

// Decode one word (8 entries) starting after column `col`: add each delta,
// gather x, multiply pairs in half2, add both products to fp32 accumulators.
template <bool XS>
__device__ __forceinline__ void decode_word(uint32_t w, const uint4 v, int& col,
                                            const __half* xg, const __half* xs,
                                            float& acc0, float& acc1) {
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    col += (int)((w >> (8 * h)) & 0xFu);
    const __half x0 = gather_h<XS>(xg, xs, col);
    col += (int)((w >> (8 * h + 4)) & 0xFu);
    const __half x1 = gather_h<XS>(xg, xs, col);
    __half2 av;
    *reinterpret_cast<uint32_t*>(&av) = vw[h];
    const __half2 prod = __hmul2(av, __halves2half2(x0, x1));
    acc0 = add_f16(acc0, __low2half(prod));
    acc1 = add_f16(acc1, __high2half(prod));
  }
}

// fp32 acc + a * x for fp16 a and x: the product is exact in fp32, so one
// fp32 rounding (mixed-precision fma).
__device__ __forceinline__ float fma_f16(float acc, uint16_t a, uint16_t x) {
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(x));
  return acc;
}

// Decode one word (8 entries) whose first entry follows column `col`, with x
// read through L1. The eight columns come from byte-wise prefix sums of the
// nibbles: with lo / hi the even / odd nibbles spread into bytes, byte j of
// P = (lo + hi) * 0x01010101 is the sum of nibbles 0..2j+1 (at most 120, so
// no carries), and byte j of P - hi the sum of nibbles 0..2j; each column is
// one byte extract and one address, and each entry one mixed fma.
__device__ __forceinline__ void decode_word_l1(uint32_t w, const uint4 v, int& col,
                                               const __half* xg, float& acc0, float& acc1) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t P = (lo + hi) * 0x01010101u;
  const uint32_t Q = P - hi;
  const uint16_t* xb = reinterpret_cast<const uint16_t*>(xg) + col;
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t c0 = __byte_perm(Q, 0u, 0x4440u + (uint32_t)j);
    const uint32_t c1 = __byte_perm(P, 0u, 0x4440u + (uint32_t)j);
    const uint16_t x0 = __ldg(xb + c0);
    const uint16_t x1 = __ldg(xb + c1);
    acc0 = fma_f16(acc0, (uint16_t)(vw[j] & 0xFFFFu), x0);
    acc1 = fma_f16(acc1, (uint16_t)(vw[j] >> 16), x1);
  }
  col += (int)(P >> 24);
}

// decode_word_l1 with x from the skewed shared-memory copy.
__device__ __forceinline__ void decode_word_smem(uint32_t w, const uint4 v, int& col,
                                                 const uint16_t* xs, float& acc0,
                                                 float& acc1) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t P = (lo + hi) * 0x01010101u;
  const uint32_t Q = P - hi;
  const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c0 = col + (int)__byte_perm(Q, 0u, 0x4440u + (uint32_t)j);
    const int c1 = col + (int)__byte_perm(P, 0u, 0x4440u + (uint32_t)j);
    acc0 = fma_f16(acc0, (uint16_t)(vw[j] & 0xFFFFu), xs[x_skew(c0)]);
    acc1 = fma_f16(acc1, (uint16_t)(vw[j] >> 16), xs[x_skew(c1)]);
  }
  col += (int)(P >> 24);
}

// Thread 0: start the TMA copies of DELTA4 unit u (descriptor d) into a stage.
__device__ __forceinline__ void issue_unit(const DeltaArgs& a, unsigned char* stage,
                                           uint64_t* bar, int4* desc, int u, const int4 d,
                                           uint64_t pol) {
  if (u < 0) {
    *desc = make_int4(-1, 0, 0, 0);
    mbar_arrive(bar);
    return;
  }
  *desc = d;
  const int wb = d.y, we = d.z;
  const int wa = wb & ~3;
  const uint32_t nwb = (uint32_t)(((we + 3) & ~3) - wa) * 4u;
  const uint32_t nvb = (uint32_t)(we - wb) * 16u;
  if (nvb == 0) {
    mbar_arrive(bar);
    return;
  }
  mbar_arrive_expect_tx(bar, DeltaStage::kBaseBytes + nwb + nvb);
  bulk_g2s(stage, a.warp_base + (size_t)u * kDeltaWarps, DeltaStage::kBaseBytes, bar, pol);
  bulk_g2s(stage + DeltaStage::kBaseBytes, a.words + wa, nwb, bar, pol);
  bulk_g2s(stage + DeltaStage::kBaseBytes + DeltaStage::kWordBytes, a.vals + (size_t)wb * 8,
           nvb, bar, pol);
}

// Thread 0, at the end of this CTA's piece of a row split into units: as
// split_publish for CSR, with units in place of chunks.
__device__ __forceinline__ void delta_publish(const DeltaArgs& a, int row, bool whole,
                                              int wb0, int wb, float part) {
  if (whole) {
    a.y[row] = part;
    return;
  }
  const int sid = __ldg(a.row_split + row);
  const SplitInfo si = a.splits[sid];
  const int k0 = (wb0 - si.row_begin) / si.reserved;
  const int k = (wb - si.row_begin) / si.reserved;
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

// Persistent DELTA4 kernel ("MACKO-SpMV" 2.2): each CTA walks its block of
// units (equal weight per CTA); thread 0 keeps kDeltaStages units in flight
// with TMA bulk copies. In a unit, warp w decodes words [64w, 64w+64) and
// lane l words 64w+2l and 64w+2l+1 (16 entries; in a HALF unit, of a short
// row, words [32w, 32w+32) and word 32w+l): the column before the
// lane's first entry is the warp's starting column (from the planner) plus
// the lane's nibble sum put through a 5-step __shfl_up_sync inclusive scan.
// Products are formed in half2 and accumulated in fp32 across the units of a
// row; the row total is a CTA reduction.
// Decode of the x-through-L1 path: 2 byte-prefix columns and mixed fma
// (decode_word_l1), 1 per-entry columns and half2 products (decode_word).
#ifndef SPMV_DELTA_DECODE
#define SPMV_DELTA_DECODE 2
#endif
#ifndef SPMV_DELTA_MIN_BLOCKS
#define SPMV_DELTA_MIN_BLOCKS (kDeltaThreads == 128 ? 8 : 6)
#endif
template <bool XS>
__global__ void __launch_bounds__(kDeltaThreads, SPMV_DELTA_MIN_BLOCKS)
    delta4_kernel(const DeltaArgs a) {
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  __shared__ __align__(8) uint64_t s_bar[kDeltaStages];
  __shared__ int4 s_desc[kDeltaStages];
  __shared__ float s_red[kDeltaWarps];
  __shared__ int s_fail;
  unsigned char* stages = dyn_smem;
  __half* xs = reinterpret_cast<__half*>(dyn_smem + kDeltaStages * DeltaStage::kBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u_begin = __ldg(a.cta_first + blockIdx.x);
  const int u_end = __ldg(a.cta_first + blockIdx.x + 1);
  uint64_t pol = 0;
  int4 next_d = make_int4(0, 0, 0, 0);
  int next_u = u_begin;
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kDeltaStages; ++s) mbar_init(&s_bar[s], 1);
    fence_mbar_init();
    s_fail = 0;
  }
  __syncthreads();
  if (tid == 0) {
    pol = policy_evict_first();
    int4 d0[kDeltaStages];
#pragma unroll
    for (int s = 0; s < kDeltaStages; ++s)
      d0[s] = next_u + s < u_end ? __ldg(a.units + next_u + s) : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int s = 0; s < kDeltaStages; ++s)
      issue_unit(a, stages + s * DeltaStage::kBytes, &s_bar[s], &s_desc[s],
                 next_u + s < u_end ? next_u + s : -1, d0[s], pol);
    next_u += kDeltaStages;
    if (next_u < u_end) next_d = __ldg(a.units + next_u);
    pdl_launch_dependents();
  }
  // plan-owned data only above; x and y below
  pdl_wait();
  if (XS) stage_x_skewed(xs, a.x, a.n_cols);
  float acc0 = 0.f, acc1 = 0.f;  // this thread's share of the current row piece
  int piece_wb0 = -1;
  bool piece_first = false;
  int i = 0;
  for (;; ++i) {
    const int s = i % kDeltaStages;
    const uint32_t parity = (uint32_t)(i / kDeltaStages) & 1u;
    const bool ok = mbar_wait_bounded(&s_bar[s], parity);
    if (!ok) s_fail = 1;  // seen by all after the barrier that ends this unit
    const int4 d = s_desc[s];
    if (d.x == -1) break;  // uniform: every thread reads the same descriptor
    unsigned char* stage = stages + s * DeltaStage::kBytes;
    const uint32_t rw = (uint32_t)d.x;
    const int row = (int)(rw & kUnitRowMask);
    const int wb = d.y, n_w = d.z - d.y;
    if (piece_wb0 < 0) {
      piece_wb0 = wb;
      piece_first = (rw & kUnitFirst) != 0;
    }
    const int* s_base = reinterpret_cast<const int*>(stage);
    const uint32_t* s_words =
        reinterpret_cast<const uint32_t*>(stage + DeltaStage::kBaseBytes) + (wb & 3);
    const uint4* s_vals =
        reinterpret_cast<const uint4*>(stage + DeltaStage::kBaseBytes + DeltaStage::kWordBytes);
    const int lg = (int)((rw >> kUnitLgShift) & 3u);  // log2(words per lane)
    const int j0 = tid << lg;  // this lane's first word in the unit
    uint32_t wd[kDeltaMaxLaneWords];
    int ls = 0;
#pragma unroll
    for (int q = 0; q < kDeltaMaxLaneWords; ++q) {
      wd[q] = (q < (1 << lg) && ok && j0 + q < n_w) ? s_words[j0 + q] : 0u;
      ls += nibble_sum(wd[q]);
    }
    int incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += up;
    }
    if (ok && j0 < n_w) {
      int col = s_base[warp] + incl - ls;  // column before this lane's first entry
#pragma unroll
      for (int q = 0; q < kDeltaMaxLaneWords; ++q)
        if (q < (1 << lg) && j0 + q < n_w) {
          if (XS || SPMV_DELTA_DECODE == 1)
            decode_word<XS>(wd[q], s_vals[j0 + q], col, a.x, xs, acc0, acc1);
          else
            decode_word_l1(wd[q], s_vals[j0 + q], col, a.x, acc0, acc1);
        }
    }
    const bool last = (rw & kUnitLast) != 0;
    if (last || u_begin + i == u_end - 1) {  // row ends, or this CTA's share does
      const float part = block_sum<kDeltaWarps>(acc0 + acc1, s_red);
      if (tid == 0) delta_publish(a, row, piece_first && last, piece_wb0, wb, part);
      acc0 = acc1 = 0.f;
      piece_wb0 = -1;
    }
    __syncthreads();  // stage s is free again
    if (s_fail) break;
    if (tid == 0) {
      fence_proxy_async_smem();
      issue_unit(a, stage, &s_bar[s], &s_desc[s], next_u < u_end ? next_u : -1, next_d, pol);
      ++next_u;
      if (next_u < u_end) next_d = __ldg(a.units + next_u);
    }
  }
  if (tid == 0 && s_fail) {
    atomicExch(a.status, 1);
    // let copies still in flight land before the CTA's shared memory goes
    for (int s = 0; s < kDeltaStages; ++s) {
      const int fills = 1 + (i > s ? (i - 1 - s) / kDeltaStages + 1 : 0);
      mbar_wait_bounded(&s_bar[s], (uint32_t)(fills - 1) & 1u);
    }
  }
}

// ------------------------------------- DELTA4, producer / consumer variant
// One producer lane per group issues the TMA copies; each group's
// kDeltaWarps consumer warps decode its units. A stage is handed back by
// each consumer warp arriving on the stage's "empty" mbarrier once it has
// read it, so consumer warps never wait for one another per unit (no CTA
// barrier in the loop): a warp that is done with a unit moves on to the next
// staged one. A row's total is formed when its last unit ends: each warp
// parks its shuffle-reduced sum in a slot, and the warp whose shared-memory
// atomicAdd completes the slot's count adds the kDeltaWarps sums in warp
// order (deterministic) and publishes the row.
// A CTA holds G groups, each with its own block of units (a "virtual CTA"
// of the plan: v = blockIdx.x * G + g), stage ring and slots; with x in
// shared memory the groups share one copy of it.
#ifndef SPMV_DELTA_PC_STAGES
#define SPMV_DELTA_PC_STAGES 3
#endif
#ifndef SPMV_DELTA_PC_XS_STAGES
#define SPMV_DELTA_PC_XS_STAGES 2
#endif
#ifndef SPMV_DELTA_PC_XS_GROUPS
#define SPMV_DELTA_PC_XS_GROUPS 3
#endif
template <bool XS>
struct PcCfg {
  static constexpr int kGroups = XS ? SPMV_DELTA_PC_XS_GROUPS : 1;
  static constexpr int kStages = XS ? SPMV_DELTA_PC_XS_STAGES : SPMV_DELTA_PC_STAGES;
  // row sums in flight: a group's warps are less than kStages units apart
  static constexpr int kSlots = kStages + 2;
  static constexpr int kThreads = kGroups * kDeltaThreads + 32;
  static constexpr int kMinBlocks = XS ? 2 : 5;
};

template <bool XS>
__global__ void __launch_bounds__(PcCfg<XS>::kThreads, PcCfg<XS>::kMinBlocks)
    delta4_pc_kernel(const DeltaArgs a) {
  using C = PcCfg<XS>;
  constexpr int G = C::kGroups, S = C::kStages;
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  __shared__ __align__(8) uint64_t s_full[G][S];
  __shared__ __align__(8) uint64_t s_empty[G][S];
  __shared__ int4 s_desc[G][S];
  __shared__ float s_part[G][C::kSlots][kDeltaWarps];
  __shared__ int s_cnt[G][C::kSlots];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int g = 0; g < G; ++g) {
      for (int s = 0; s < S; ++s) {
        mbar_init(&s_full[g][s], 1);
        mbar_init(&s_empty[g][s], kDeltaWarps);
      }
      for (int k = 0; k < C::kSlots; ++k) s_cnt[g][k] = 0;
    }
    fence_mbar_init();
  }
  __syncthreads();  // the only CTA-wide barrier

  if (warp == G * kDeltaWarps) {  // producer warp: lane g feeds group g
    if (lane < G) {
      const int g = lane;
      const int v = blockIdx.x * G + g;
      const int u_begin = __ldg(a.cta_first + v);
      const int n_units = __ldg(a.cta_first + v + 1) - u_begin;
      unsigned char* stages = dyn_smem + (size_t)g * S * DeltaStage::kBytes;
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < n_units; ++i) {
        const int s = i % S;
        if (i >= S && !mbar_wait_bounded(&s_empty[g][s], (uint32_t)(i / S - 1) & 1u)) {
          ok = false;
          break;
        }
        issue_unit(a, stages + s * DeltaStage::kBytes, &s_full[g][s], &s_desc[g][s],
                   u_begin + i, __ldg(a.units + u_begin + i), pol);
        issued = i + 1;
        if (issued == S) pdl_launch_dependents();
      }
      if (issued < S) pdl_launch_dependents();
      if (!ok) {
        atomicExch(a.status, 1);
        // let copies still in flight land before the CTA's shared memory goes
        for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
          mbar_wait_bounded(&s_full[g][j % S], (uint32_t)(j / S) & 1u);
      }
    }
    return;
  }

  // consumers; plan-owned data only above, x and y below
  pdl_wait();
  const int g = warp / kDeltaWarps, lw = warp % kDeltaWarps;
  const int gt = tid - g * kDeltaThreads;  // thread index within the group
  const uint16_t* xs =
      reinterpret_cast<const uint16_t*>(dyn_smem + (size_t)G * S * DeltaStage::kBytes);
  if (XS) {
    stage_x_skewed(reinterpret_cast<__half*>(dyn_smem + (size_t)G * S * DeltaStage::kBytes),
                   a.x, a.n_cols, false, G * kDeltaThreads);
    asm volatile("bar.sync 1, %0;" ::"n"(G * kDeltaThreads) : "memory");  // consumers only
  }
  const int v = blockIdx.x * G + g;
  const int u_begin = __ldg(a.cta_first + v);
  const int n_units = __ldg(a.cta_first + v + 1) - u_begin;
  const unsigned char* stages = dyn_smem + (size_t)g * S * DeltaStage::kBytes;
  float acc0 = 0.f, acc1 = 0.f;  // this thread's share of the current row piece
  int piece_wb0 = -1;
  bool piece_first = false;
  int slot = 0;
  for (int i = 0; i < n_units; ++i) {
    const int s = i % S;
    if (!mbar_wait_bounded(&s_full[g][s], (uint32_t)(i / S) & 1u)) {
      if (lane == 0) atomicExch(a.status, 1);
      break;
    }
    const int4 d = s_desc[g][s];
    const unsigned char* stage = stages + s * DeltaStage::kBytes;
    const uint32_t rw = (uint32_t)d.x;
    const int row = (int)(rw & kUnitRowMask);
    const int wb = d.y, n_w = d.z - d.y;
    if (piece_wb0 < 0) {
      piece_wb0 = wb;
      piece_first = (rw & kUnitFirst) != 0;
    }
    const int* s_base = reinterpret_cast<const int*>(stage);
    const uint32_t* s_words =
        reinterpret_cast<const uint32_t*>(stage + DeltaStage::kBaseBytes) + (wb & 3);
    const uint4* s_vals =
        reinterpret_cast<const uint4*>(stage + DeltaStage::kBaseBytes + DeltaStage::kWordBytes);
    const int lg = (int)((rw >> kUnitLgShift) & 3u);  // log2(words per lane)
    const int j0 = gt << lg;  // this lane's first word in the unit
    uint32_t wd[kDeltaMaxLaneWords];
    uint4 vd[kDeltaMaxLaneWords];
    int ls = 0;
#pragma unroll
    for (int q = 0; q < kDeltaMaxLaneWords; ++q) {
      const bool in = q < (1 << lg) && j0 + q < n_w;
      wd[q] = in ? s_words[j0 + q] : 0u;
      vd[q] = in ? s_vals[j0 + q] : make_uint4(0, 0, 0, 0);
      ls += nibble_sum(wd[q]);
    }
    const int base = s_base[lw];
    __syncwarp();
    if (lane == 0) mbar_arrive(&s_empty[g][s]);  // this warp is done with the stage
    int incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += up;
    }
    if (j0 < n_w) {
      int col = base + incl - ls;  // column before this lane's first entry
#pragma unroll
      for (int q = 0; q < kDeltaMaxLaneWords; ++q)
        if (q < (1 << lg) && j0 + q < n_w) {
          if (XS)
            decode_word_smem(wd[q], vd[q], col, xs, acc0, acc1);
          else
            decode_word_l1(wd[q], vd[q], col, a.x, acc0, acc1);
        }
    }
    const bool last = (rw & kUnitLast) != 0;
    if (last || i == n_units - 1) {  // row ends, or this group's share does
      const float vsum = warp_sum(acc0 + acc1);
      if (lane == 0) {
        s_part[g][slot][lw] = vsum;
        __threadfence_block();
        if (atomicAdd(&s_cnt[g][slot], 1) == kDeltaWarps - 1) {
          __threadfence_block();
          const volatile float* sp = s_part[g][slot];
          float t = 0.f;
#pragma unroll
          for (int w2 = 0; w2 < kDeltaWarps; ++w2) t += sp[w2];
          s_cnt[g][slot] = 0;
          delta_publish(a, row, piece_first && last, piece_wb0, wb, t);
        }
      }
      slot = slot + 1 == C::kSlots ? 0 : slot + 1;
      acc0 = acc1 = 0.f;
      piece_wb0 = -1;
    }
  }
}

template <typename VT, typename XT, bool XS>
const void* csr_fn() {
  return reinterpret_cast<const void*>(&csr_kernel<VT, XT, XS>);
}

template <typename VT>
constexpr size_t stage_bytes() {
  return (size_t)Stage<VT>::kBytes;
}

const void* csr_entry(spmv_dtype dt, bool xs) {
  if (dt == SPMV_F32) return xs ? csr_fn<float, float, true>() : csr_fn<float, float, false>();
  return xs ? csr_fn<__half, __half, true>() : csr_fn<__half, __half, false>();
}

const void* delta_pc_entry(bool xs) {
  return xs ? reinterpret_cast<const void*>(&delta4_pc_kernel<true>)
            : reinterpret_cast<const void*>(&delta4_pc_kernel<false>);
}

const void* delta_entry(bool xs) {
  return xs ? reinterpret_cast<const void*>(&delta4_kernel<true>)
            : reinterpret_cast<const void*>(&delta4_kernel<false>);
}

// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel on the stream drains; it orders itself with
// griddepcontrol.wait before touching anything that kernel may write. Every
// CTA of these grids is resident at once (persistent grids), so CTAs that
// wait can never keep the kernel they wait on from running.
int launch_pdl(const void* fn, int grid, int block, size_t smem, void* stream, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args) == cudaSuccess ? 0 : -1;
}

}  // namespace

// CTAs per SM that fit, and at most as many as keep the shared memory they
// hold (dynamic + static + the per-CTA reservation) within `budget` bytes.
int occupancy_within(const void* fn, int block, size_t dyn_smem, size_t budget) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, block, dyn_smem) != cudaSuccess)
    return -1;
  cudaFuncAttributes fa;
  int reserved = 0, dev = 0;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
          cudaSuccess)
    return -1;
  const size_t per_cta = dyn_smem + fa.sharedSizeBytes + (size_t)reserved;
  const int cap = (int)(budget / per_cta);
  return n < cap ? n : (cap > 0 ? cap : 1);
}

int csr_kernel_occupancy(spmv_dtype dtype, bool x_smem, size_t dyn_smem, size_t budget) {
  return occupancy_within(csr_entry(dtype, x_smem), kThreads, dyn_smem, budget);
}

int delta_kernel_occupancy(bool x_smem, size_t dyn_smem, size_t budget) {
  if (delta_use_pc(x_smem))
    return occupancy_within(delta_pc_entry(x_smem), delta_block(x_smem), dyn_smem, budget);
  return occupancy_within(delta_entry(x_smem), kDeltaThreads, dyn_smem, budget);
}

size_t delta_stages_bytes(bool x_smem) {
  if (!delta_use_pc(x_smem)) return (size_t)kDeltaStages * DeltaStage::kBytes;
  return x_smem ? (size_t)PcCfg<true>::kGroups * PcCfg<true>::kStages * DeltaStage::kBytes
                : (size_t)PcCfg<false>::kGroups * PcCfg<false>::kStages * DeltaStage::kBytes;
}

int delta_groups(bool x_smem) {
  if (!delta_use_pc(x_smem)) return 1;
  return x_smem ? PcCfg<true>::kGroups : PcCfg<false>::kGroups;
}

int delta_block(bool x_smem) {
  if (!delta_use_pc(x_smem)) return kDeltaThreads;
  return x_smem ? PcCfg<true>::kThreads : PcCfg<false>::kThreads;
}

size_t delta_stage_bytes() { return (size_t)DeltaStage::kBytes; }

size_t delta_x_smem_bytes(int n_cols) {
  return ((size_t)n_cols + 2 * ((size_t)n_cols / 64) + 16) * 2;
}

size_t csr_stage_bytes(spmv_dtype dtype) {
  return dtype == SPMV_F32 ? stage_bytes<float>() : stage_bytes<__half>();
}

int set_kernel_smem_limits(size_t csr_dyn, size_t delta_dyn) {
  const void* fns[] = {csr_entry(SPMV_F32, true), csr_entry(SPMV_F16, true),
                       csr_entry(SPMV_F32, false), csr_entry(SPMV_F16, false)};
  if (csr_dyn > 0)
    for (const void* f : fns)
      if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)csr_dyn) != cudaSuccess)
        return -1;
  if (delta_dyn > 0 &&
      (cudaFuncSetAttribute(delta_entry(true), cudaFuncAttributeMaxDynamicSharedMemorySize,
                            (int)delta_dyn) != cudaSuccess ||
       cudaFuncSetAttribute(delta_pc_entry(true), cudaFuncAttributeMaxDynamicSharedMemorySize,
                            (int)delta_dyn) != cudaSuccess ||
       cudaFuncSetAttribute(delta_pc_entry(false), cudaFuncAttributeMaxDynamicSharedMemorySize,
                            (int)delta_dyn) != cudaSuccess))
    return -1;
  return 0;
}

int launch_csr(const Plan& p, const void* x, float* y, void* stream) {
  if (p.n_tiles == 0) return 0;
  CsrArgs a;
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
  return launch_pdl(csr_entry(p.dtype, p.x_smem), p.grid, kThreads, p.dyn_smem, stream, args);
}

int launch_delta(const Plan& p, const void* x, float* y, void* stream) {
  if (p.n_tiles == 0) return 0;
  DeltaArgs a;
  a.words = p.words;
  a.vals = static_cast<const __half*>(p.values);
  a.x = static_cast<const __half*>(x);
  a.y = y;
  a.units = reinterpret_cast<const int4*>(p.tiles);
  a.warp_base = p.warp_base;
  a.cta_first = p.cta_first;
  a.row_split = p.row_split;
  a.splits = p.splits;
  a.partials = p.partials;
  a.counters = p.counters;
  a.status = p.status;
  a.n_cols = p.n_cols;
  void* args[] = {&a};
  if (delta_use_pc(p.x_smem))
    return launch_pdl(delta_pc_entry(p.x_smem), p.grid, delta_block(p.x_smem), p.dyn_smem,
                      stream, args);
  return launch_pdl(delta_entry(p.x_smem), p.grid, kDeltaThreads, p.dyn_smem, stream, args);
}

}  // namespace spmv
