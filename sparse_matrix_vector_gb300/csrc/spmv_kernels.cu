// Device half of the library: the sm_103a kernels of y = A x.
//
// CSR kernel (one launch, one work unit per CTA, or a grid-stride loop when x
// is staged in shared memory). Work units come from the host planner:
//   short-row tile  -- a run of consecutive short rows whose nonzeros are
//                      streamed with 16-byte loads across the whole CTA
//                      (coalesced regardless of where rows start), multiplied
//                      by the gathered x, parked in shared memory, then
//                      reduced with 2^lg lanes per row (sub-warp / warp bins);
//   CTA-row tile    -- one long row, the CTA strides over it, CTA reduction;
//   split chunk     -- a slice of a very long row; the chunk's partial sum
//                      goes to plan-owned scratch and the last chunk to
//                      finish (atomic counter) adds the partials in chunk
//                      order and writes y.
// Sources: "CUDA CSR SpMV optimisation" (codechina.net) 2.1 (row sum), 3.1
// (read-only path and shared-memory staging of x), 3.2 (vector loads), 4.1
// (warp per row with shuffle reduction); "Hash-based multi-phase SpGEMM"
// (mlqm.cn) 2.1.1 / 2.2 (rows binned to partial-warp, warp and block-per-row
// kernels); "MACKO-SpMV" (maplevalley.com.cn) 3.3 (splitting long rows).
//
// DELTA4 kernel ("MACKO-SpMV" 2.2): one CTA per row (grid-stride over rows).
// A round covers 256 packed words (2048 entries): thread t loads word t (four
// bytes of nibbles, coalesced) and the eight fp16 values of those entries (16
// bytes, coalesced); the columns are rebuilt by a per-thread sum of 8 nibbles,
// a 5-step __shfl_up_sync inclusive scan inside each warp and a prefix over the
// CTA's warp totals; products are taken in half2 (__hmul2) and accumulated in
// fp32. The next round's loads are issued before the current round is
// decoded, across row boundaries too.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "spmv_internal.h"

namespace spmv {
namespace {

// ------------------------------------------------------------ load helpers
// Matrix data is read exactly once: read-only path, no L1 allocation.
__device__ __forceinline__ int4 ld_stream_i4(const int32_t* p) {
  int4 r;
  asm("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
  float4 r;
  asm("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
      : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
  uint2 r;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
      : "=r"(r.x), "=r"(r.y)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const uint32_t* p) {
  uint32_t r;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

template <int Q>
__device__ __forceinline__ int lane_of(const int4& c) {
  return Q == 0 ? c.x : Q == 1 ? c.y : Q == 2 ? c.z : c.w;
}

// Four consecutive matrix values, widened to fp32 on use.
template <typename VT>
struct Vals4;

template <>
struct Vals4<float> {
  float4 v;
  __device__ __forceinline__ void load(const float* p) { v = ld_stream_f4(p); }
  template <int Q>
  __device__ __forceinline__ float get() const {
    return Q == 0 ? v.x : Q == 1 ? v.y : Q == 2 ? v.z : v.w;
  }
};

template <>
struct Vals4<__half> {
  uint2 v;
  __device__ __forceinline__ void load(const __half* p) { v = ld_stream_u2(p); }
  template <int Q>
  __device__ __forceinline__ float get() const {
    const uint32_t w = Q < 2 ? v.x : v.y;
    const unsigned short h =
        (unsigned short)((Q & 1) ? (w >> 16) : (w & 0xFFFFu));
    return __half2float(__ushort_as_half(h));
  }
};

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

// ------------------------------------------------------------ CSR kernel
struct CsrArgs {
  const int32_t* __restrict__ row_ptr;
  const int32_t* __restrict__ col;
  const void* __restrict__ val;
  const void* __restrict__ x;
  float* __restrict__ y;
  const int4* __restrict__ tiles;
  int n_tiles;
  int n_cols;
  const SplitInfo* __restrict__ splits;
  float* partials;
  int32_t* counters;
  int split_chunk;
};

// Short-row tile: rows [r0, r0+R), nonzeros [s, e).
template <typename VT, typename XT, bool XS>
__device__ __forceinline__ void stream_tile(const CsrArgs& a, const int4 t,
                                            const XT* xs, float* s_prod,
                                            int* s_rp) {
  const int tid = threadIdx.x;
  const int r0 = t.x, s = t.y, e = t.z;
  const uint32_t meta = (uint32_t)t.w;
  const int R = (int)(meta & kRowsMask);
  const int lg = (int)((meta >> kLanesShift) & 7u);
  const int a0 = s & ~(kVec - 1);           // 16-byte aligned start
  const int s_rel = s - a0, e_rel = e - a0;
  const int nvec = (e_rel + kVec - 1) / kVec;
  const VT* val = static_cast<const VT*>(a.val);
  const XT* xg = static_cast<const XT*>(a.x);

  int4 c[kStreamVecs];
  Vals4<VT> v[kStreamVecs];
#pragma unroll
  for (int k = 0; k < kStreamVecs; ++k) {
    const int j = tid + k * kThreads;
    if (j < nvec) {
      c[k] = ld_stream_i4(a.col + a0 + j * kVec);
      v[k].load(val + a0 + j * kVec);
    }
  }
  for (int i = tid; i <= R; i += kThreads) s_rp[i] = __ldg(a.row_ptr + r0 + i) - a0;
#pragma unroll
  for (int k = 0; k < kStreamVecs; ++k) {
    const int j = tid + k * kThreads;
    if (j < nvec) {
      const int rel = j * kVec;
      float4 p;
      p.x = (rel + 0 >= s_rel && rel + 0 < e_rel)
                ? v[k].template get<0>() * gather<XS>(xg, xs, lane_of<0>(c[k])) : 0.f;
      p.y = (rel + 1 >= s_rel && rel + 1 < e_rel)
                ? v[k].template get<1>() * gather<XS>(xg, xs, lane_of<1>(c[k])) : 0.f;
      p.z = (rel + 2 >= s_rel && rel + 2 < e_rel)
                ? v[k].template get<2>() * gather<XS>(xg, xs, lane_of<2>(c[k])) : 0.f;
      p.w = (rel + 3 >= s_rel && rel + 3 < e_rel)
                ? v[k].template get<3>() * gather<XS>(xg, xs, lane_of<3>(c[k])) : 0.f;
      *reinterpret_cast<float4*>(s_prod + rel) = p;
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
      const int b = s_rp[r], en = s_rp[r + 1];
      for (int i = b + lig; i < en; i += g) acc += s_prod[i];
    }
    for (int o = g >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lig == 0 && r < R) a.y[r0 + r] = acc;
  }
}

// Per-thread partial sum of nonzeros [b, e) of one row.
template <typename VT, typename XT, bool XS>
__device__ __forceinline__ float range_sum(const CsrArgs& a, int b, int e,
                                           const XT* xs) {
  const int tid = threadIdx.x;
  const int a0 = b & ~(kVec - 1);
  const int b_rel = b - a0, e_rel = e - a0;
  const int nvec = (e_rel + kVec - 1) / kVec;
  const VT* val = static_cast<const VT*>(a.val) + a0;
  const int32_t* col = a.col + a0;
  const XT* xg = static_cast<const XT*>(a.x);
  float acc = 0.f;
  for (int j0 = tid; j0 < nvec; j0 += kThreads * kRowUnroll) {
    int4 c[kRowUnroll];
    Vals4<VT> v[kRowUnroll];
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
      const int j = j0 + u * kThreads;
      if (j < nvec) {
        c[u] = ld_stream_i4(col + j * kVec);
        v[u].load(val + j * kVec);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowUnroll; ++u) {
      const int j = j0 + u * kThreads;
      if (j < nvec) {
        const int rel = j * kVec;
        if (rel + 0 >= b_rel && rel + 0 < e_rel)
          acc = fmaf(v[u].template get<0>(), gather<XS>(xg, xs, lane_of<0>(c[u])), acc);
        if (rel + 1 >= b_rel && rel + 1 < e_rel)
          acc = fmaf(v[u].template get<1>(), gather<XS>(xg, xs, lane_of<1>(c[u])), acc);
        if (rel + 2 >= b_rel && rel + 2 < e_rel)
          acc = fmaf(v[u].template get<2>(), gather<XS>(xg, xs, lane_of<2>(c[u])), acc);
        if (rel + 3 >= b_rel && rel + 3 < e_rel)
          acc = fmaf(v[u].template get<3>(), gather<XS>(xg, xs, lane_of<3>(c[u])), acc);
      }
    }
  }
  return acc;
}

// Thread 0 of a split chunk: publish the partial; the last chunk of the row
// to arrive adds all partials in chunk order, writes y and re-arms the
// counter for the next run.
__device__ __forceinline__ void split_finish(const CsrArgs& a, int row, int b,
                                             int sid, float part) {
  const SplitInfo si = a.splits[sid];
  const int chunk = (b - __ldg(a.row_ptr + row)) / a.split_chunk;
  a.partials[si.first_slot + chunk] = part;
  __threadfence();
  const int arrived = atomicAdd(a.counters + sid, 1);
  if (arrived == si.n_chunks - 1) {
    __threadfence();
    float sum = 0.f;
    for (int k = 0; k < si.n_chunks; ++k) sum += __ldcg(a.partials + si.first_slot + k);
    a.y[row] = sum;
    a.counters[sid] = 0;
  }
}

template <typename VT, typename XT, bool XS>
__global__ void __launch_bounds__(kThreads) csr_kernel(const CsrArgs a) {
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  __shared__ __align__(16) float s_prod[kProdCap];
  __shared__ int s_rp[kMaxTileRows + 1];
  __shared__ float s_red[kWarps];
  XT* xs = reinterpret_cast<XT*>(dyn_smem);
  if (XS) stage_x<XT>(xs, static_cast<const XT*>(a.x), a.n_cols);
  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const int4 d = __ldg(a.tiles + t);
    const uint32_t kind = (uint32_t)d.w >> kKindShift;
    if (kind == kKindStream) {
      stream_tile<VT, XT, XS>(a, d, xs, s_prod, s_rp);
    } else {
      const float part = cta_sum(range_sum<VT, XT, XS>(a, d.y, d.z, xs), s_red);
      if (threadIdx.x == 0) {
        if (kind == kKindRow)
          a.y[d.x] = part;
        else
          split_finish(a, d.x, d.y, (int)((uint32_t)d.w & kSplitIdMask), part);
      }
    }
    __syncthreads();  // shared buffers are reused by the next tile
  }
}

// ------------------------------------------------------------ DELTA4 kernel
struct DeltaArgs {
  const int32_t* __restrict__ row_ptr;  // entry offsets, multiples of 8
  const uint32_t* __restrict__ words;   // 8 nibbles per word
  const uint4* __restrict__ vals;       // 8 fp16 values per 16 bytes
  const __half* __restrict__ x;
  float* __restrict__ y;
  int n_rows;
  int n_cols;
};

// Sum of the eight 4-bit fields of w (<= 120).
__device__ __forceinline__ int nibble_sum(uint32_t w) {
  const uint32_t b = (w & 0x0F0F0F0Fu) + ((w >> 4) & 0x0F0F0F0Fu);
  return (int)((b * 0x01010101u) >> 24);
}

template <bool XS>
__device__ __forceinline__ __half gather_h(const __half* xg, const __half* xs, int c) {
  return XS ? xs[c] : __ldg(xg + c);
}

template <bool XS>
__global__ void __launch_bounds__(kThreads) delta4_kernel(const DeltaArgs a) {
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  __shared__ int s_tot[2][kWarps];
  __shared__ float s_red[kWarps];
  __half* xs = reinterpret_cast<__half*>(dyn_smem);
  if (XS) stage_x<__half>(xs, a.x, a.n_cols);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  int r = blockIdx.x;
  if (r >= a.n_rows) return;
  int rb = __ldg(a.row_ptr + r) >> 3;         // first word of this round
  int w_end = __ldg(a.row_ptr + r + 1) >> 3;  // one past the row's last word
  int nr = r + G, nb0 = 0, nb1 = 0;           // next row and its word range
  if (nr < a.n_rows) {
    nb0 = __ldg(a.row_ptr + nr) >> 3;
    nb1 = __ldg(a.row_ptr + nr + 1) >> 3;
  }
  uint32_t cw = 0;
  uint4 cv = make_uint4(0u, 0u, 0u, 0u);
  if (rb + tid < w_end) {
    cw = ld_stream_u32(a.words + rb + tid);
    cv = ld_stream_u4(a.vals + rb + tid);
  }
  float acc = 0.f;
  int base = 0, buf = 0;
  while (true) {
    const bool row_done = rb + kDeltaWordsPerRound >= w_end;
    // issue the next round's loads before decoding this one
    const int fb = row_done ? nb0 : rb + kDeltaWordsPerRound;
    const int fe = row_done ? nb1 : w_end;
    const bool have_next = !row_done || nr < a.n_rows;
    uint32_t pw = 0;
    uint4 pv = make_uint4(0u, 0u, 0u, 0u);
    if (have_next && fb + tid < fe) {
      pw = ld_stream_u32(a.words + fb + tid);
      pv = ld_stream_u4(a.vals + fb + tid);
    }
    // columns: base + (warps before) + (lanes before) + (nibbles before)
    const int ls = nibble_sum(cw);
    int incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += up;
    }
    if (lane == 31) s_tot[buf][warp] = incl;
    __syncthreads();
    int pre = 0, tot = 0;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      const int t = s_tot[buf][w2];
      tot += t;
      pre += w2 < warp ? t : 0;
    }
    buf ^= 1;
    if (rb + tid < w_end) {
      int col = base + pre + incl - ls;
      const uint32_t vw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        col += (int)((cw >> (8 * h)) & 0xFu);
        const __half x0 = gather_h<XS>(a.x, xs, col);
        col += (int)((cw >> (8 * h + 4)) & 0xFu);
        const __half x1 = gather_h<XS>(a.x, xs, col);
        __half2 av;
        *reinterpret_cast<uint32_t*>(&av) = vw[h];
        const float2 f = __half22float2(__hmul2(av, __halves2half2(x0, x1)));
        acc += f.x;
        acc += f.y;
      }
    }
    base += tot;
    if (row_done) {
      const float sum = cta_sum(acc, s_red);
      if (tid == 0) a.y[r] = sum;
      acc = 0.f;
      base = 0;
      r = nr;
      if (r >= a.n_rows) break;
      rb = nb0;
      w_end = nb1;
      nr = r + G;
      if (nr < a.n_rows) {
        nb0 = __ldg(a.row_ptr + nr) >> 3;
        nb1 = __ldg(a.row_ptr + nr + 1) >> 3;
      }
    } else {
      rb += kDeltaWordsPerRound;
    }
    cw = pw;
    cv = pv;
  }
}

template <typename VT, typename XT, bool XS>
const void* csr_fn() {
  return reinterpret_cast<const void*>(&csr_kernel<VT, XT, XS>);
}

const void* csr_entry(spmv_dtype dt, bool xs) {
  if (dt == SPMV_F32) return xs ? csr_fn<float, float, true>() : csr_fn<float, float, false>();
  return xs ? csr_fn<__half, __half, true>() : csr_fn<__half, __half, false>();
}

const void* delta_entry(bool xs) {
  return xs ? reinterpret_cast<const void*>(&delta4_kernel<true>)
            : reinterpret_cast<const void*>(&delta4_kernel<false>);
}

}  // namespace

int csr_kernel_occupancy(spmv_dtype dtype, bool x_smem, size_t dyn_smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, csr_entry(dtype, x_smem),
                                                    kThreads, dyn_smem) != cudaSuccess)
    return -1;
  return n;
}

int delta_kernel_occupancy(bool x_smem, size_t dyn_smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, delta_entry(x_smem), kThreads,
                                                    dyn_smem) != cudaSuccess)
    return -1;
  return n;
}

int set_kernel_smem_limits(size_t csr_dyn, size_t delta_dyn) {
  const void* fns[] = {csr_entry(SPMV_F32, true), csr_entry(SPMV_F16, true)};
  if (csr_dyn > 0)
    for (const void* f : fns)
      if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)csr_dyn) != cudaSuccess)
        return -1;
  if (delta_dyn > 0 &&
      cudaFuncSetAttribute(delta_entry(true), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)delta_dyn) != cudaSuccess)
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
  a.n_tiles = (int)p.n_tiles;
  a.n_cols = p.n_cols;
  a.splits = p.splits;
  a.partials = p.partials;
  a.counters = p.counters;
  a.split_chunk = p.split_chunk;
  void* args[] = {&a};
  return cudaLaunchKernel(csr_entry(p.dtype, p.x_smem), dim3((unsigned)p.grid),
                          dim3(kThreads), args, p.dyn_smem,
                          static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? 0
             : -1;
}

int launch_delta(const Plan& p, const void* x, float* y, void* stream) {
  if (p.n_rows == 0) return 0;
  DeltaArgs a;
  a.row_ptr = p.row_ptr;
  a.words = p.words;
  a.vals = reinterpret_cast<const uint4*>(p.values);
  a.x = static_cast<const __half*>(x);
  a.y = y;
  a.n_rows = p.n_rows;
  a.n_cols = p.n_cols;
  void* args[] = {&a};
  return cudaLaunchKernel(delta_entry(p.x_smem), dim3((unsigned)p.grid), dim3(kThreads),
                          args, p.dyn_smem, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? 0
             : -1;
}

}  // namespace spmv
