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

__device__ __forceinline__ float jacobi(float d, float r) {
  return d != 0.f ? r / d : r;  // a row without a diagonal is left unscaled
}

// Each thread takes elements i, i + S, i + 2S, i + 3S (S = the grid's
// threads) per pass, all four loads issued before any is used, so a thread
// waits on one memory round trip per pass instead of one per element. A
// thread's share of a dot product is summed in fp32 over a pass (at most 4
// terms) and then added into an fp64 total (fp64 arithmetic is scarce on
// this part).
constexpr int kPcgUnroll = 4;

// r = b - q (q = A x0), z = D^-1 r, p = z; rz, rr, bb.
__global__ void __launch_bounds__(kPcgThreads) pcg_init(const PcgVectors a) {
  const int S = gridDim.x * kPcgThreads;
  double v[3] = {0.0, 0.0, 0.0};
  for (int i0 = blockIdx.x * kPcgThreads + threadIdx.x; i0 < a.n; i0 += kPcgUnroll * S) {
    float bv[kPcgUnroll], qv[kPcgUnroll], dv[kPcgUnroll];
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) {
      const int i = i0 + u * S;
      if (i < a.n) {
        bv[u] = a.b[i];
        qv[u] = a.q[i];
        dv[u] = a.diag[i];
      }
    }
    float c[3] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) {
      const int i = i0 + u * S;
      if (i < a.n) {
        const float ri = bv[u] - qv[u];
        const float zi = jacobi(dv[u], ri);
        a.r[i] = ri;
        a.z[i] = zi;
        a.p[i] = zi;
        c[0] = fmaf(ri, zi, c[0]);
        c[1] = fmaf(ri, ri, c[1]);
        c[2] = fmaf(bv[u], bv[u], c[2]);
      }
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) v[q] += c[q];
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
  const int S = gridDim.x * kPcgThreads;
  double v[1] = {0.0};
  for (int i0 = blockIdx.x * kPcgThreads + threadIdx.x; i0 < a.n; i0 += kPcgUnroll * S) {
    float pv[kPcgUnroll], qv[kPcgUnroll];
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) {
      const int i = i0 + u * S;
      pv[u] = i < a.n ? a.p[i] : 0.f;
      qv[u] = i < a.n ? a.q[i] : 0.f;
    }
    float c = 0.f;
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) c = fmaf(pv[u], qv[u], c);
    v[0] += c;
  }
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
  const int S = gridDim.x * kPcgThreads;
  double v[2] = {0.0, 0.0};
  for (int i0 = blockIdx.x * kPcgThreads + threadIdx.x; i0 < a.n; i0 += kPcgUnroll * S) {
    float xv[kPcgUnroll], pv[kPcgUnroll], rv[kPcgUnroll], qv[kPcgUnroll], dv[kPcgUnroll];
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) {
      const int i = i0 + u * S;
      if (i < a.n) {
        xv[u] = a.x[i];
        pv[u] = a.p[i];
        rv[u] = a.r[i];
        qv[u] = a.q[i];
        dv[u] = a.diag[i];
      }
    }
    float c[2] = {0.f, 0.f};
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) {
      const int i = i0 + u * S;
      if (i < a.n) {
        a.x[i] = fmaf(alpha, pv[u], xv[u]);
        const float ri = fmaf(-alpha, qv[u], rv[u]);
        const float zi = jacobi(dv[u], ri);
        a.r[i] = ri;
        a.z[i] = zi;
        c[0] = fmaf(ri, zi, c[0]);
        c[1] = fmaf(ri, ri, c[1]);
      }
    }
    v[0] += c[0];
    v[1] += c[1];
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
  const int S = gridDim.x * kPcgThreads;
  for (int i0 = blockIdx.x * kPcgThreads + threadIdx.x; i0 < a.n; i0 += kPcgUnroll * S) {
    float zv[kPcgUnroll], pv[kPcgUnroll];
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) {
      const int i = i0 + u * S;
      if (i < a.n) {
        zv[u] = a.z[i];
        pv[u] = a.p[i];
      }
    }
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) {
      const int i = i0 + u * S;
      if (i < a.n) a.p[i] = fmaf(beta, pv[u], zv[u]);
    }
  }
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
