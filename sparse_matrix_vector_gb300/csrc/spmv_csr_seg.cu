// CSR kernel with warp-owned segments (fp32 or fp16 values, int32 columns):
// y[row] = sum over the row's nonzeros of values[k] * x[col[k]] ("CUDA CSR
// SpMV optimisation" 2.1), with the work laid out as for the column-delta
// kernel.
//
// The planner cuts the rows into segments and gives each warp of the grid a
// contiguous share of them, of equal weight. Long-row plans: every segment is
// a slice of at most 512 nonzeros of one row (full ones first). Mixed plans
// (irregular matrices): a run of consecutive whole rows of at most 256
// nonzeros in all is packed into one segment ("Hash-based multi-phase
// SpGEMM" 5.2, batching tiny rows), longer rows are cut into slices of 256.
// A segment's block (a 32-byte header, its columns, its values) is staged by
// one bulk copy into the warp's own ring of shared-memory buffers; lane s of
// the warp issues the copies into buffer s, so warps never wait for one
// another and no CTA barrier sits in the loop (the CTA-wide tiles of
// spmv_csr.cu pay one per work unit, which dominates when a row of ~1,000
// nonzeros leaves a 256-thread CTA five per thread).
// Lane l takes nonzeros l, l + 32, ... of a segment: a warp-wide step reads
// 32 consecutive columns and values (conflict-free) and gathers x at 32
// neighbouring columns of the row ("CUDA CSR SpMV optimisation" 4.1: a warp
// per row, shuffle reduction). fp16 values multiply fp16 x exactly in fp32
// (mixed-precision fma); fp32 values use fp32 fma.
// Packed rows: the products are parked in shared memory and lane l sums rows
// l, l + 32, ... of the run. Slices: lanes keep fp32 partials; at a row's
// last segment, or the end of the warp's piece of it, the warp reduces them.
// A row inside one share is written at once. A row split into two pieces
// (two warps) meets in one 64-bit exchange per piece (hand_over, settle:
// nothing waits, and the sum is the same bits in either order); a row of
// more pieces leaves one partial per warp, and the warp whose atomicAdd
// completes the row's count adds them in warp order. The planner puts the
// piece a warp shares with the next warp at the front of its share, so that
// both of the warp's hand-overs go out early.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "spmv_device.cuh"
#include "spmv_internal.h"

namespace spmv {
namespace {

#ifndef SPMV_CSR_SEG_STAGES
#define SPMV_CSR_SEG_STAGES 2
#endif
constexpr int kCS = SPMV_CSR_SEG_STAGES;
// Warps per CTA (one CTA per SM). Long-row plans: fewer warps give each
// thread more registers and keep more gathers in flight; the LLM 12288^2
// fp16 matrices at 30 / 70 / 90% sparsity (fraction of HBM peak, before
// rows of two pieces met in one exchange): 20 warps 0.99 / 0.94 / 0.74, 16
// warps 1.00 / 0.94 / 0.74, 24 warps 1.00 / 0.93 / 0.73, 28 warps 0.92 /
// 0.89 / 0.72; after it, 20 warps 1.01 / 1.01 / 0.86, 16 and 24 warps
// within 2%. Mixed plans gather x mostly at
// random: their rings stay near 125 KB so that L1 keeps about 100 KB, which
// random gathers through L1 need (with 28 KB of L1 they ran at half the
// rate). On the power-law matrix (916k rows, 5.1M nonzeros): 16, 24 or 32
// warps 27.8, 26.6, 26.6 us; packing rows of at most 64, 128 or 256
// nonzeros 27.1, 26.6, 26.0 us.
#ifndef SPMV_CSR_MIXED_WARPS
#define SPMV_CSR_MIXED_WARPS 24
#endif
#ifndef SPMV_CSR_LONG_WARPS_F16
#define SPMV_CSR_LONG_WARPS_F16 20
#endif
#ifndef SPMV_CSR_LONG_WARPS_F32
#define SPMV_CSR_LONG_WARPS_F32 24
#endif
template <typename VT, bool MIXED>
constexpr int kCW = MIXED ? SPMV_CSR_MIXED_WARPS
                          : (sizeof(VT) == 2 ? SPMV_CSR_LONG_WARPS_F16 : SPMV_CSR_LONG_WARPS_F32);

template <typename VT, bool MIXED>
struct CSeg {
  static constexpr int kCap = MIXED ? kCsrSegNnzMixed : kCsrSegNnzLong;
  static constexpr int kK = kCap / 32;  // nonzeros per lane in a full segment
  static constexpr int kBytes =
      (int)csr_seg_bytes(kCap, MIXED ? kCsrSegNnzMixed : 0, (int)sizeof(VT));
  static_assert(kBytes % 16 == 0, "segment buffers stay 16-byte aligned");
};

struct CsrSegArgs {
  const unsigned char* __restrict__ blocks;  // one block per segment
  const int32_t* __restrict__ seg_off;       // block offsets (16-byte steps), n_segs + 1
  const int32_t* __restrict__ warp_first;    // first segment per warp, n_warps + 1
  const int32_t* __restrict__ empty_rows;
  const SplitInfo* __restrict__ splits;      // {first slot, pieces, 0, 0}
  const void* __restrict__ x;
  float* __restrict__ y;
  float* partials;
  int32_t* counters;
  unsigned long long* cells;  // one per split row, zero between runs
  int32_t* status;
  const int* skip;  // when set and nonzero at launch: do nothing (a finished solve)
  int n_empty;
  int n_cols;
};

// acc + a * x: fp32 fma, or for fp16 the mixed-precision fma (exact product).
__device__ __forceinline__ float fma_v(float acc, float a, float x) { return fmaf(a, x, acc); }
__device__ __forceinline__ float fma_v(float acc, uint16_t a, uint16_t x) {
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(x));
  return acc;
}

// a * x as fp32 (exact for fp16 operands).
__device__ __forceinline__ float mul_v(float a, float x) { return a * x; }
__device__ __forceinline__ float mul_v(uint16_t a, uint16_t x) {
  return __half2float(__ushort_as_half(a)) * __half2float(__ushort_as_half(x));
}

template <typename VT> struct Bits;
template <> struct Bits<float> { using T = float; };
template <> struct Bits<__half> { using T = uint16_t; };

// x at column c: shared memory (XS) or the read-only path.
template <typename VT, bool XS>
__device__ __forceinline__ typename Bits<VT>::T load_x(const typename Bits<VT>::T* xs,
                                                       const void* x, int c) {
  using T = typename Bits<VT>::T;
  return XS ? xs[c] : __ldg(static_cast<const T*>(x) + c);
}

// Copy x (n elements) into shared memory with every thread of the CTA.
template <typename VT>
__device__ __forceinline__ void copy_x(typename Bits<VT>::T* xs, const void* x, int n, int nt) {
  using T = typename Bits<VT>::T;
  const T* src = static_cast<const T*>(x);
  constexpr int per = 16 / (int)sizeof(T);
  int done = 0;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
    const int nv = n / per;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(xs);
    // four loads a thread before their stores: one trip to memory for the x
    // that fits shared memory
    for (int v0 = 0; v0 < nv; v0 += 4 * nt) {
      uint4 r[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (v0 + k * nt + (int)threadIdx.x < nv) r[k] = __ldg(s4 + v0 + k * nt + threadIdx.x);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (v0 + k * nt + (int)threadIdx.x < nv) d4[v0 + k * nt + threadIdx.x] = r[k];
    }
    done = nv * per;
  }
  for (int i = done + threadIdx.x; i < n; i += nt) xs[i] = __ldg(src + i);
}

// Lane 0, after its share: make the parked pieces of rows shared with other
// warps visible (one fence), count each; the warp that completes a row's
// count adds its pieces in warp order, writes y and re-arms the count.
__device__ __forceinline__ void finish_pieces(const CsrSegArgs& a, const int2 (&pend)[2],
                                              int n_pend) {
  __threadfence();
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    if (p >= n_pend) break;
    const int row = pend[p].x, sid = pend[p].y;
    const SplitInfo si = a.splits[sid];
    if (atomicAdd(a.counters + sid, 1) == si.n_chunks - 1) {
      __threadfence();
      float sum = 0.f;
      for (int j = 0; j < si.n_chunks; ++j) sum += __ldcg(a.partials + si.first_slot + j);
      a.y[row] = sum;
      a.counters[sid] = 0;
    }
  }
}

// Checked builds: the staged columns of a segment are tested against n_cols
// and a packed run's row starts clamped into [0, nonzeros] (first and last
// exactly to its ends) before the segment is used (see spmv_internal.h).
template <typename VT>
__device__ __noinline__ void check_segment(const CsrSegArgs& a, unsigned char* st, int nz,
                                           int R, int lane) {
  bool bad = false;
  unsigned char* cols = st + kSegHeaderBytes;
  if (R > 0) {
    int16_t* rs = reinterpret_cast<int16_t*>(cols);
    for (int q = lane; q <= R; q += 32) {
      const int v = checked_offset(rs[q], 0, nz, &bad);
      rs[q] = (int16_t)(q == 0 ? 0 : q == R ? nz : v);
      if ((q == 0 && v != 0) || (q == R && v != nz)) bad = true;
    }
    cols += ((R + 1) * 2 + 15) & ~15;
  }
  int* s_col = reinterpret_cast<int*>(cols);
  for (int j = lane; j < nz; j += 32) s_col[j] = checked_col(s_col[j], a.n_cols, &bad);
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicExch(a.status, kStatusBadIndex);
  __syncwarp();
}

// A packed run of R whole rows: every lane forms the products of nonzeros
// lane, lane + 32, ... (a warp-wide step gathers x for 32 consecutive
// nonzeros) and parks them in place of the columns. Then, 32 rows at a time,
// lane l sums row l of the group from there in nonzero order if it holds at
// most kLaneRowMax nonzeros; the longer rows of the group are summed by the
// whole warp one after another (strided partials, shuffle tree). y is
// written once per row; the order of every sum is fixed.
constexpr int kLaneRowMax = 32;

template <typename VT, bool XS, int K>
__device__ __forceinline__ void packed_rows(const CsrSegArgs& a, unsigned char* st, int R,
                                            int nz, int row0, int lane,
                                            const typename Bits<VT>::T* xs) {
  using T = typename Bits<VT>::T;
  const int16_t* rs = reinterpret_cast<const int16_t*>(st + kSegHeaderBytes);
  unsigned char* cols = st + kSegHeaderBytes + (((R + 1) * 2 + 15) & ~15);
  const int* s_col = reinterpret_cast<const int*>(cols);
  const T* s_val = reinterpret_cast<const T*>(cols + ((nz * 4 + 15) & ~15));
  float* s_prod = reinterpret_cast<float*>(cols);
  // every column, then every x gather, before the first product is parked
  // over the columns: the K gathers of a lane are in flight together
  // (a lane overwrites only its own columns)
  int c[K];
  T xv[K];
#pragma unroll
  for (int k = 0; k < K; ++k) c[k] = 32 * k + lane < nz ? s_col[32 * k + lane] : 0;
#pragma unroll
  for (int k = 0; k < K; ++k)
    if (32 * k + lane < nz) xv[k] = load_x<VT, XS>(xs, a.x, c[k]);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int j = 32 * k + lane;
    if (j < nz) s_prod[j] = mul_v(s_val[j], xv[k]);
  }
  __syncwarp();
  for (int q0 = 0; q0 < R; q0 += 32) {
    const int q = q0 + lane;
    int b = 0, e = 0;
    if (q < R) {
      b = rs[q];
      e = rs[q + 1];
    }
    const bool wide = e - b > kLaneRowMax;
    if (q < R && !wide) {
      float sum = 0.f;
      for (int j = b; j < e; ++j) sum += s_prod[j];
      a.y[row0 + q] = sum;
    }
    for (unsigned m = __ballot_sync(0xffffffffu, wide); m != 0u; m &= m - 1u) {
      const int src = __ffs(m) - 1;
      const int bb = __shfl_sync(0xffffffffu, b, src), ee = __shfl_sync(0xffffffffu, e, src);
      float v = 0.f;
      for (int j = bb + lane; j < ee; j += 32) v += s_prod[j];
      v = warp_sum(v);
      if (lane == 0) a.y[row0 + q0 + src] = v;
    }
  }
}

template <typename VT, bool XS, bool MIXED>
__global__ void __launch_bounds__(kCW<VT, MIXED> * 32, 1) csr_seg_kernel(const CsrSegArgs a) {
  using T = typename Bits<VT>::T;
  using Sg = CSeg<VT, MIXED>;
  constexpr int W = kCW<VT, MIXED>;
  constexpr int kBytes = Sg::kBytes;
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  __shared__ __align__(8) uint64_t s_full[W][kCS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * W + warp;
  unsigned char* ring = dyn_smem + (size_t)warp * kCS * kBytes;
  T* xs = reinterpret_cast<T*>(dyn_smem + (size_t)W * kCS * kBytes);
  const int t0 = __ldg(a.warp_first + gw);
  const int n = __ldg(a.warp_first + gw + 1) - t0;
  const uint64_t pol = policy_evict_first();

  // plan-owned data only until pdl_wait: the first kCS blocks of the share;
  // lane s issues every copy into buffer s
  if (lane == 0) {
    for (int s = 0; s < kCS; ++s) mbar_init(&s_full[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane < kCS && lane < n) {
    const int o0 = __ldg(a.seg_off + t0 + lane), o1 = __ldg(a.seg_off + t0 + lane + 1);
    mbar_arrive_expect_tx(&s_full[warp][lane], (uint32_t)(o1 - o0) * 16u);
    bulk_g2s(ring + lane * kBytes, a.blocks + (size_t)o0 * 16, (uint32_t)(o1 - o0) * 16u,
             &s_full[warp][lane], pol);
  }
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();
  if (a.skip && *a.skip) {  // let the copies issued above land, then leave
    if (lane < kCS && lane < n) mbar_wait_bounded(&s_full[warp][lane], 0u);
    return;
  }
  if (XS) copy_x<VT>(xs, a.x, a.n_cols, W * 32);
  for (int i = blockIdx.x * W * 32 + threadIdx.x; i < a.n_empty; i += gridDim.x * W * 32)
    a.y[__ldg(a.empty_rows + i)] = 0.f;
  if (XS) __syncthreads();

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  // pieces of rows shared with other warps (lane 0): {row, split id}; a share
  // holds at most two, its first row's and its last row's
  int2 pend[2];
  int n_pend = 0;
  // lane 0: pieces of rows split in two, each handed over in one exchange
  // whose result is read only after the share: {row, this piece's sum} and
  // the cell's previous content (nonzero: the other piece, which was first)
  Pair pair0, pair1;
  int n_pair = 0;
  int s = 0;
  uint32_t phase = 0;
  int i = 0;
  for (; i < n; ++i) {
    // the warp decides together (its shuffles below need every lane)
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_full[warp][s], phase))) {
      if (lane == 0) atomicExch(a.status, 1);
      break;
    }
    unsigned char* st = ring + s * kBytes;
    const int4 h0 = *reinterpret_cast<const int4*>(st);       // rows, row | flags, nonzeros, split
    const int4 h1 = *reinterpret_cast<const int4*>(st + 16);  // next block's offset, bytes; slot
    const int nz = h0.z;
    const uint32_t rf = (uint32_t)h0.y;
    if (kChecked) check_segment<VT>(a, st, nz, (MIXED && (rf & kSegPacked)) ? h0.x : 0, lane);
    if (MIXED && (rf & kSegPacked)) {
      packed_rows<VT, XS, Sg::kK>(a, st, h0.x, nz, (int)(rf & kSegRowMask), lane, xs);
      // the products written into the buffer are ordered before the bulk
      // copy's writes into it
      __syncwarp();
      if (lane == s && h1.y > 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&s_full[warp][s], (uint32_t)h1.y);
        bulk_g2s(ring + s * kBytes, a.blocks + (size_t)h1.x * 16, (uint32_t)h1.y,
                 &s_full[warp][s], pol);
      }
      if (++s == kCS) {
        s = 0;
        phase ^= 1u;
      }
      continue;
    }
    const int* s_col = reinterpret_cast<const int*>(st + kSegHeaderBytes);
    const T* s_val = reinterpret_cast<const T*>(st + kSegHeaderBytes + ((nz * 4 + 15) & ~15));
    if (nz == Sg::kCap) {  // one straight-line block: all gathers can overlap
#pragma unroll
      for (int k = 0; k < Sg::kK; ++k) {
        const int j = 32 * k + lane;
        acc[k & 3] = fma_v(acc[k & 3], s_val[j], load_x<VT, XS>(xs, a.x, s_col[j]));
      }
    } else {
#pragma unroll
      for (int k = 0; k < Sg::kK; ++k) {
        const int j = 32 * k + lane;
        if (j < nz) acc[k & 3] = fma_v(acc[k & 3], s_val[j], load_x<VT, XS>(xs, a.x, s_col[j]));
      }
    }
    // every lane has used the buffer's contents: refill it
    __syncwarp();
    if (lane == s && h1.y > 0) {
      mbar_arrive_expect_tx(&s_full[warp][s], (uint32_t)h1.y);
      bulk_g2s(ring + s * kBytes, a.blocks + (size_t)h1.x * 16, (uint32_t)h1.y, &s_full[warp][s],
               pol);
    }
    // the row ends, this warp's piece of it does, or this warp's share does
    if ((rf & kSegLast) || (h1.w & kSegCtlPieceEnd) || i == n - 1) {
      const float v = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      if (lane == 0) {
        const int row = (int)(rf & kSegRowMask);
        if (h0.w < 0) {
          a.y[row] = v;
        } else if ((h1.w & kSegCtlPair) && n_pair < 2) {
          if (n_pair == 0)
            pair0 = hand_over(a.cells, h0.w, row, v);
          else
            pair1 = hand_over(a.cells, h0.w, row, v);
          ++n_pair;
        } else if (!(h1.w & kSegCtlPair) && n_pend < 2) {  // park it, count it later
          a.partials[h1.z] = v;
          if (n_pend == 0)
            pend[0] = make_int2(row, h0.w);
          else
            pend[1] = make_int2(row, h0.w);
          ++n_pend;
        } else {
          atomicExch(a.status, 2);  // the plan broke its own rule: report, never write
        }
      }
    }
    // every piece of a shared row this warp holds is parked: count them now,
    // while the warp still has rows to stream, not at the end of the launch
    if ((h1.w & kSegCtlCombine) && lane == 0 && n_pend > 0) {
      finish_pieces(a, pend, n_pend);
      n_pend = 0;
    }
    if (++s == kCS) {
      s = 0;
      phase ^= 1u;
    }
  }
  if (i == n && lane == 0 && n_pend > 0) finish_pieces(a, pend, n_pend);
  if (i == n && lane == 0) {
    if (n_pair > 0) settle(pair0, a.y, a.cells);
    if (n_pair > 1) settle(pair1, a.y, a.cells);
  }
  if (i < n && lane == 0) {
    // a wait gave up: let this warp's copies still in flight land before the
    // CTA's shared memory goes (bounded again)
    for (int j = i; j < n && j < i + kCS; ++j) {
      mbar_wait_bounded(&s_full[warp][s], phase);
      if (++s == kCS) {
        s = 0;
        phase ^= 1u;
      }
    }
  }
}

template <bool MIXED>
const void* csr_seg_entry_m(spmv_dtype dt, bool xs) {
  if (dt == SPMV_F32)
    return xs ? reinterpret_cast<const void*>(&csr_seg_kernel<float, true, MIXED>)
              : reinterpret_cast<const void*>(&csr_seg_kernel<float, false, MIXED>);
  return xs ? reinterpret_cast<const void*>(&csr_seg_kernel<__half, true, MIXED>)
            : reinterpret_cast<const void*>(&csr_seg_kernel<__half, false, MIXED>);
}

const void* csr_seg_entry(spmv_dtype dt, bool xs, bool mixed) {
  return mixed ? csr_seg_entry_m<true>(dt, xs) : csr_seg_entry_m<false>(dt, xs);
}

}  // namespace

int csr_seg_warps_per_cta(spmv_dtype dt, bool mixed) {
  if (mixed) return dt == SPMV_F32 ? kCW<float, true> : kCW<__half, true>;
  return dt == SPMV_F32 ? kCW<float, false> : kCW<__half, false>;
}

int csr_seg_stages(spmv_dtype) { return kCS; }

size_t csr_seg_rings_bytes(spmv_dtype dt, bool mixed) {
  if (mixed)
    return dt == SPMV_F32 ? (size_t)kCW<float, true> * kCS * CSeg<float, true>::kBytes
                          : (size_t)kCW<__half, true> * kCS * CSeg<__half, true>::kBytes;
  return dt == SPMV_F32 ? (size_t)kCW<float, false> * kCS * CSeg<float, false>::kBytes
                        : (size_t)kCW<__half, false> * kCS * CSeg<__half, false>::kBytes;
}

int csr_seg_set_smem_limit(size_t dyn) {
  if (dyn == 0) return 0;
  for (spmv_dtype dt : {SPMV_F32, SPMV_F16})
    for (bool xs : {false, true})
      for (bool mixed : {false, true})
        if (cudaFuncSetAttribute(csr_seg_entry(dt, xs, mixed),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)dyn) != cudaSuccess)
          return -1;
  return 0;
}

int csr_seg_occupancy(spmv_dtype dt, bool x_smem, bool mixed, size_t dyn_smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, csr_seg_entry(dt, x_smem, mixed),
                                                    csr_seg_warps_per_cta(dt, mixed) * 32,
                                                    dyn_smem) != cudaSuccess)
    return -1;
  return n;
}

int launch_csr_seg(const Plan& p, const void* x, float* y, void* stream, const int* skip) {
  if (p.grid == 0) return 0;
  CsrSegArgs a;
  a.skip = skip;
  a.blocks = p.blocks;
  a.seg_off = p.seg_off;
  a.warp_first = p.cta_first;
  a.empty_rows = p.empty_rows;
  a.splits = p.splits;
  a.x = x;
  a.y = y;
  a.partials = p.partials;
  a.counters = p.counters;
  a.cells = p.cells;
  a.status = p.status;
  a.n_empty = p.n_empty_rows;
  a.n_cols = p.n_cols;
  void* args[] = {&a};
  return launch_pdl(csr_seg_entry(p.dtype, p.x_smem, p.csr_mixed), p.grid,
                    csr_seg_warps_per_cta(p.dtype, p.csr_mixed) * 32, p.dyn_smem, stream, args);
}

}  // namespace spmv
