// Device-side helpers shared by the CSR and DELTA4 kernels: warp and CTA
// reductions, the x staging copy, TMA bulk copies and mbarriers with bounded
// waits, programmatic dependent launch, and the occupancy rule.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "spmv_internal.h"

namespace spmv {
namespace {

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
  // (whole CTA of kThreads threads; ends with a CTA barrier)
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

// A warp's piece of a row split into exactly two pieces (segment kernels).
// Each piece's warp swaps {1, its fp32 sum} into the row's 64-bit cell (zero
// between runs) and goes on without waiting: the swap returns the cell's
// previous content, which is read only after the warp's share. The piece
// that finds the other's sum there came second; it writes y = its sum + the
// other (fp32 addition is commutative, so the result does not depend on
// which came first) and empties the cell. No fence is needed: the other
// piece's sum travels in the exchange itself.
struct Pair {
  int row;
  int cell;
  float mine;
  unsigned long long prev;
};

__device__ __forceinline__ Pair hand_over(unsigned long long* cells, int cell, int row, float v) {
  Pair p;
  p.row = row;
  p.cell = cell;
  p.mine = v;
  p.prev = atomicExch(cells + cell, (1ull << 32) | __float_as_uint(v));
  return p;
}

__device__ __forceinline__ void settle(const Pair& p, float* y, unsigned long long* cells) {
  if (p.prev != 0) {
    y[p.row] = p.mine + __uint_as_float((uint32_t)p.prev);
    cells[p.cell] = 0;
  }
}

// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel on the stream drains; it orders itself with
// griddepcontrol.wait before touching anything that kernel may write. The
// dependent grid is launched only once every CTA of the earlier one has
// executed griddepcontrol.launch_dependents or exited, so by then all of the
// earlier kernel's CTAs have started, and CTAs that wait can never keep it
// from running.
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
inline int occupancy_within(const void* fn, int block, size_t dyn_smem, size_t budget) {
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

}  // namespace spmv
