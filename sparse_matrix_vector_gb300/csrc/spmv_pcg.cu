// Jacobi-preconditioned conjugate gradients around spmv_run ("Fused FEM
// matvec" 6.1: CG with the diagonal preconditioner, its iterations the
// consumer of the matrix-vector products).
//
// One iteration is the plan's y = A x launch followed by three small kernels
// (step length, updates, new direction). Vectors are fp32; the scalars of
// the recurrence live in device memory in fp64, so the host never waits
// inside an iteration. Dot products are reduced in two fixed-order levels
// (per block; then the block partials by whichever block finishes last, each
// of its threads a fixed stride of them before a fixed-order block sum), so a
// solve gives the same bits every time. Once the
// residual test passes (or the iteration limit or a breakdown is hit) a
// device flag turns the remaining kernels of a batch into no-ops, and the
// host only reads the scalars between batches.
#include <cuda_runtime.h>

#include <cstdint>

#include "spmv_device.cuh"
#include "spmv_internal.h"

namespace spmv {
namespace {

struct PcgVectors {
  const float* __restrict__ b;
  float* __restrict__ x;
  float* __restrict__ r;
  float* __restrict__ z;
  float* __restrict__ p;
  float* __restrict__ q;
  const float* __restrict__ diag;
  double* partials;  // 3 * kPcgBlocks
  PcgScalars* sc;
  int n;
};

// Fixed-order sums of up to three per-thread values over the block; thread 0
// gets the totals. Called by every thread.
template <int K>
__device__ __forceinline__ void block_sums(double (&v)[K]) {
  __shared__ double s_w[K][kPcgThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_down_sync(0xffffffffu, v[k], o);
    if (lane == 0) s_w[k][w] = v[k];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      double t = 0.0;
      for (int i = 0; i < kPcgThreads / 32; ++i) t += s_w[k][i];
      v[k] = t;
    }
  }
}

// Every thread: thread 0 parks the block's sums (from block_sums); the block
// that arrives last then adds all the blocks' sums, each thread a fixed
// stride of them and then block_sums in fixed order, and returns true with
// the grid totals in thread 0's tot. Every other block returns false.
template <int K>
__device__ __forceinline__ bool grid_sums(const PcgVectors& a, const double (&v)[K],
                                          double (&tot)[K]) {
  __shared__ int s_last;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) a.partials[k * kPcgBlocks + blockIdx.x] = v[k];
    __threadfence();
    s_last = atomicAdd(&a.sc->arrived, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return false;
  __threadfence();
  double w[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    w[k] = 0.0;
    for (int i = threadIdx.x; i < (int)gridDim.x; i += kPcgThreads)
      w[k] += __ldcg(a.partials + k * kPcgBlocks + i);
  }
  block_sums<K>(w);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) tot[k] = w[k];
    a.sc->arrived = 0;
  }
  return true;
}

__device__ __forceinline__ float jacobi(const float* diag, int i, float r) {
  const float d = diag[i];
  return d != 0.f ? r / d : r;  // a row without a diagonal is left unscaled
}

// r = b - q (q = A x0), z = D^-1 r, p = z; rz, rr, bb.
__global__ void __launch_bounds__(kPcgThreads) pcg_init(const PcgVectors a) {
  double v[3] = {0.0, 0.0, 0.0};
  for (int i = blockIdx.x * kPcgThreads + threadIdx.x; i < a.n; i += gridDim.x * kPcgThreads) {
    const float bi = a.b[i];
    const float ri = bi - a.q[i];
    const float zi = jacobi(a.diag, i, ri);
    a.r[i] = ri;
    a.z[i] = zi;
    a.p[i] = zi;
    v[0] += (double)ri * zi;
    v[1] += (double)ri * ri;
    v[2] += (double)bi * bi;
  }
  block_sums<3>(v);
  double t[3];
  if (grid_sums<3>(a, v, t) && threadIdx.x == 0) {
    PcgScalars* sc = a.sc;
    sc->rz = t[0];
    sc->rr = t[1];
    sc->bb = t[2];
    sc->iter = 0;
    sc->done = t[1] <= sc->tol2 * t[2] ? kPcgConverged : (sc->max_iter <= 0 ? kPcgMaxIter : 0);
  }
}

// alpha = rz / (p . q).
__global__ void __launch_bounds__(kPcgThreads) pcg_alpha(const PcgVectors a) {
  if (a.sc->done) return;
  double v[1] = {0.0};
  for (int i = blockIdx.x * kPcgThreads + threadIdx.x; i < a.n; i += gridDim.x * kPcgThreads)
    v[0] += (double)a.p[i] * a.q[i];
  block_sums<1>(v);
  double t[1];
  if (grid_sums<1>(a, v, t) && threadIdx.x == 0) {
    PcgScalars* sc = a.sc;
    if (!(t[0] > 0.0)) {
      sc->done = kPcgBreakdown;  // p . A p <= 0: A is not positive definite
    } else {
      sc->alpha = sc->rz / t[0];
    }
  }
}

// x += alpha p, r -= alpha q, z = D^-1 r; beta = (r . z) / rz, convergence.
__global__ void __launch_bounds__(kPcgThreads) pcg_update(const PcgVectors a) {
  if (a.sc->done) return;
  const float alpha = (float)a.sc->alpha;
  double v[2] = {0.0, 0.0};
  for (int i = blockIdx.x * kPcgThreads + threadIdx.x; i < a.n; i += gridDim.x * kPcgThreads) {
    a.x[i] = fmaf(alpha, a.p[i], a.x[i]);
    const float ri = fmaf(-alpha, a.q[i], a.r[i]);
    const float zi = jacobi(a.diag, i, ri);
    a.r[i] = ri;
    a.z[i] = zi;
    v[0] += (double)ri * zi;
    v[1] += (double)ri * ri;
  }
  block_sums<2>(v);
  double t[2];
  if (grid_sums<2>(a, v, t) && threadIdx.x == 0) {
    PcgScalars* sc = a.sc;
    sc->beta = t[0] / sc->rz;
    sc->rz = t[0];
    sc->rr = t[1];
    sc->iter += 1;
    if (t[1] <= sc->tol2 * sc->bb)
      sc->done = kPcgConverged;
    else if (sc->iter >= sc->max_iter)
      sc->done = kPcgMaxIter;
  }
}

// p = z + beta p.
__global__ void __launch_bounds__(kPcgThreads) pcg_direction(const PcgVectors a) {
  if (a.sc->done) return;
  const float beta = (float)a.sc->beta;
  for (int i = blockIdx.x * kPcgThreads + threadIdx.x; i < a.n; i += gridDim.x * kPcgThreads)
    a.p[i] = fmaf(beta, a.p[i], a.z[i]);
}

}  // namespace

size_t pcg_work_bytes(int n) {
  const size_t vec = ((size_t)n * 4 + 255) / 256 * 256;
  return 4 * vec + 3 * kPcgBlocks * sizeof(double) + 256;
}

int pcg_grid(int n) {
  const int need = (n + kPcgThreads - 1) / kPcgThreads;
  return need < 1 ? 1 : (need < kPcgBlocks ? need : kPcgBlocks);
}

int launch_pcg(int stage, const Plan& p, const float* b, float* x, const float* diag,
               void* stream) {
  const int n = p.n_rows;
  const size_t vec = ((size_t)n * 4 + 255) / 256 * 256;
  unsigned char* w = p.pcg_work;
  PcgVectors a;
  a.b = b;
  a.x = x;
  a.r = reinterpret_cast<float*>(w);
  a.z = reinterpret_cast<float*>(w + vec);
  a.p = reinterpret_cast<float*>(w + 2 * vec);
  a.q = reinterpret_cast<float*>(w + 3 * vec);
  a.partials = reinterpret_cast<double*>(w + 4 * vec);
  a.sc = reinterpret_cast<PcgScalars*>(w + 4 * vec + 3 * kPcgBlocks * sizeof(double));
  a.diag = diag;
  a.n = n;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = pcg_grid(n);
  switch (stage) {
    case 0: pcg_init<<<grid, kPcgThreads, 0, st>>>(a); break;
    case 1: pcg_alpha<<<grid, kPcgThreads, 0, st>>>(a); break;
    case 2: pcg_update<<<grid, kPcgThreads, 0, st>>>(a); break;
    default: pcg_direction<<<grid, kPcgThreads, 0, st>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace spmv
