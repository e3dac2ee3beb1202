// Sliced-ELL kernel of y = A x for sm_103a ("CUDA CSR SpMV optimisation"
// 2.1, ELL, cut into slices of SPMV_SELL_C = 32 rows).
//
// One warp per slice, lane = row: at step k the warp reads slot k of its 32
// rows, 32 consecutive columns and 32 consecutive values (one 128-byte line
// each for fp32), so the matrix streams fully coalesced with no row
// boundaries to find. Steps are unrolled by 8 (the last group predicated),
// so that each lane has up to 16 matrix loads and then 8 x gathers in
// flight, and the kernel is held to 32 registers for 64 warps per SM (on
// GB300, 3D FEM stiffness rows of ~78 nonzeros: 73.6 us against 77.8 us with
// 44 registers and 80.1 us unrolled by 4). x is gathered through L1; the
// matrix streams past it (evict-first loads). Padding slots (value 0 at an
// in-range column) add exactly 0 * x[c].
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "spmv_device.cuh"
#include "spmv_internal.h"

namespace spmv {
namespace {

struct SellArgs {
  const int32_t* __restrict__ slice_ptr;  // n_slices + 1 slot offsets
  const int32_t* __restrict__ perm;       // original row per slice lane, or null
  const int32_t* __restrict__ cols;
  const void* __restrict__ vals;
  const void* __restrict__ x;
  float* __restrict__ y;
  const int* skip;  // when set and nonzero at launch: do nothing (a finished solve)
  float* dot;       // when set: per-block x . y of a square matrix (conjugate gradients)
  int n_rows;
  int n_slices;
};

__device__ __forceinline__ float sell_fma(float acc, float a, float x) { return fmaf(a, x, acc); }

// fp32 acc + a * x for fp16 a and x: the product is exact in fp32, so one
// fp32 rounding (mixed-precision fma).
__device__ __forceinline__ float sell_fma(float acc, __half a, __half x) {
  asm("fma.rn.f32.f16 %0, %1, %2, %0;"
      : "+f"(acc)
      : "h"(__half_as_ushort(a)), "h"(__half_as_ushort(x)));
  return acc;
}

template <typename T>
__device__ __forceinline__ T stream_load(const T* p);
template <>
__device__ __forceinline__ int32_t stream_load(const int32_t* p) { return __ldcs(p); }
template <>
__device__ __forceinline__ float stream_load(const float* p) { return __ldcs(p); }
template <>
__device__ __forceinline__ __half stream_load(const __half* p) {
  return __ushort_as_half(__ldcs(reinterpret_cast<const unsigned short*>(p)));
}

template <typename T>
__device__ __forceinline__ T gather(const T* x, int c) {
  return __ldg(x + c);
}

#ifndef SPMV_SELL_UNROLL
#define SPMV_SELL_UNROLL 8
#endif
#ifndef SPMV_SELL_MIN_BLOCKS
#define SPMV_SELL_MIN_BLOCKS 8  // 32 registers: 64 warps per SM
#endif

template <typename VT>
__global__ void __launch_bounds__(kSellSlicesPerCta * 32, SPMV_SELL_MIN_BLOCKS)
    sell_kernel(const SellArgs a) {
  constexpr int U = SPMV_SELL_UNROLL;
  const int slice = blockIdx.x * kSellSlicesPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  const bool live = slice < a.n_slices;
  if (!live && !a.dot) return;
  const int s0 = live ? __ldg(a.slice_ptr + slice) : 0;
  const int width = live ? (__ldg(a.slice_ptr + slice + 1) - s0) >> 5 : 0;
  const int32_t* cols = a.cols + s0 + lane;
  const VT* vals = static_cast<const VT*>(a.vals) + s0 + lane;
  const int pos = slice * 32 + lane;
  const int row = !live ? -1 : a.perm ? __ldg(a.perm + pos) : (pos < a.n_rows ? pos : -1);
  // x and y belong to the stream's earlier work: read and write them only
  // after the kernels this launch depends on have completed
  pdl_wait();
  if (a.skip && *a.skip) return;
  const VT* x = static_cast<const VT*>(a.x);
  float acc[2] = {0.f, 0.f};
  // steps in groups of U, the last group predicated: a slice of width <= U
  // costs one round of matrix loads and one of gathers
  for (int k = 0; k < width; k += U) {
    int32_t c[U];
    VT v[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      if (k + j < width) {
        c[j] = stream_load(cols + (k + j) * 32);
        v[j] = stream_load(vals + (k + j) * 32);
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j)
      if (k + j < width) acc[j & 1] = sell_fma(acc[j & 1], v[j], gather(x, c[j]));
  }
  const float yv = acc[0] + acc[1];
  if (row >= 0) a.y[row] = yv;
  if (a.dot) {  // the block's x . y (square matrix: x[row] pairs with y[row]), fixed order
    __shared__ float s_red[kSellSlicesPerCta];
    const float xy = row >= 0 ? static_cast<float>(gather(x, row)) * yv : 0.f;
    const float t = block_sum<kSellSlicesPerCta>(xy, s_red);
    if (threadIdx.x == 0) a.dot[blockIdx.x] = t;
  }
}

}  // namespace

int launch_sell(const Plan& p, const void* x, float* y, void* stream, const int* skip,
                float* dot) {
  if (p.n_tiles == 0) return 0;
  SellArgs a;
  a.skip = skip;
  a.dot = dot;
  a.slice_ptr = p.row_ptr;
  a.perm = p.perm;
  a.cols = p.col_idx;
  a.vals = p.values;
  a.x = x;
  a.y = y;
  a.n_rows = p.n_rows;
  a.n_slices = (int)p.n_tiles;
  void* args[] = {&a};
  const void* fn = p.dtype == SPMV_F32 ? reinterpret_cast<const void*>(&sell_kernel<float>)
                                       : reinterpret_cast<const void*>(&sell_kernel<__half>);
  return launch_pdl(fn, p.grid, kSellSlicesPerCta * 32, 0, stream, args);
}

}  // namespace spmv
