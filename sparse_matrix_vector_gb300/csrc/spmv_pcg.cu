// Jacobi-preconditioned conjugate gradients around spmv_run ("Fused FEM
// matvec" 6.1: CG with the diagonal preconditioner, its iterations the
// consumer of the matrix-vector products).
//
// One iteration is the plan's y = A x launch followed by small kernels: the
// step length (only for plans whose product does not hand over p . q
// itself), the updates, the new direction. Vectors are fp32; the scalars of
// the recurrence live in device memory in fp64, formed once per block (fp64
// runs at about 1/64 of the fp32 rate here), so the host never waits inside
// an iteration. Dot products are reduced in two fixed-order levels: per
// block, parked in a partials array, then summed by every block of the next
// kernel in the same fixed order (each thread a fixed stride, then a
// fixed-order block sum), so a solve gives the same bits every time and no
// kernel ends with one block reducing while the rest of the GPU idles. The
// direction kernel decides, on the device, whether the solve goes on: it
// sets the condition of the solve's device-side loop, and a done flag turns
// any kernels still queued into no-ops.
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
  float* partials;  // 3 * kPcgBlocks
  const float* pq_parts;  // per-block p . q: partials, or the product kernel's
  int pq_count;           // how many
  PcgScalars* sc;
  unsigned long long cond;  // while-node handle set by pcg_direction (0: none)
  int n;
};

// Continue (1) or stop (0) the device-side iteration loop, if there is one:
// called once per iteration by one thread of pcg_direction.
__device__ __forceinline__ void set_continue(const PcgVectors& a, bool go) {
  if (a.cond) cudaGraphSetConditional((cudaGraphConditionalHandle)a.cond, go ? 1u : 0u);
}

// Fixed-order sums of up to three per-thread values over the block (a
// shuffle tree per warp, then the warps' sums in order); thread 0 gets the
// totals. Called by every thread. fp32: fp64 arithmetic runs at about 1/64
// of the fp32 rate on this part, and a fixed-order tree over the ~7e5 terms
// of a dot product keeps a relative error near 1e-6, far below what the
// recurrence needs; the order is fixed, so the bits repeat.
template <int K>
__device__ __forceinline__ void block_sums(float (&v)[K]) {
  __shared__ float s_w[K][kPcgThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    if (lane == 0) s_w[k][w] = v[k];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      float t = 0.f;
      for (int i = 0; i < kPcgThreads / 32; ++i) t += s_w[k][i];
      v[k] = t;
    }
  }
}

// This thread's fixed-stride share of K rows of parked per-block values
// (rows kPcgBlocks apart; elements threadIdx.x, + kPcgThreads, ... below
// `blocks`), added in that order. The loads of a group of kPcgLoadGroup go
// out before the first add, so a share costs one memory round trip per group
// rather than one per element. CG: read through L2 only (values written by
// other blocks of the running grid).
constexpr int kPcgLoadGroup = 8;

template <int K, bool CG>
__device__ __forceinline__ void thread_share(const float* partials, int blocks, float (&w)[K]) {
#pragma unroll
  for (int k = 0; k < K; ++k) w[k] = 0.f;
  for (int i0 = threadIdx.x; i0 < blocks; i0 += kPcgLoadGroup * kPcgThreads) {
    float t[K][kPcgLoadGroup];
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
      for (int j = 0; j < kPcgLoadGroup; ++j) {
        const int i = i0 + j * kPcgThreads;
        const float* q = partials + k * kPcgBlocks + i;
        t[k][j] = i < blocks ? (CG ? __ldcg(q) : *q) : 0.f;
      }
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
      for (int j = 0; j < kPcgLoadGroup; ++j)
        if (i0 + j * kPcgThreads < blocks) w[k] += t[k][j];
  }
}

// Every thread: thread 0 parks the block's sums (from block_sums); the block
// that arrives last then adds all the blocks' sums, each thread a fixed
// stride of them and then block_sums in fixed order, and returns true with
// the grid totals in thread 0's tot. Every other block returns false.
template <int K>
__device__ __forceinline__ bool grid_sums(const PcgVectors& a, const float (&v)[K],
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
  float w[K];
  thread_share<K, true>(a.partials, (int)gridDim.x, w);
  block_sums<K>(w);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) tot[k] = w[k];
    a.sc->arrived = 0;
  }
  return true;
}

// num / den in fp64, formed by one thread of the block and handed to all
// as fp32 (thread 0 also gets the fp64 value in *q64). fp64 runs at about
// 1/64 of the fp32 rate on this part: the same division done by every thread
// of the grid cost about 2.5 us per kernel. Called by every thread.
__device__ __forceinline__ float block_ratio(double num, double den, double* q64) {
  __shared__ float s_q;
  if (threadIdx.x == 0) {
    *q64 = num / den;
    s_q = (float)*q64;
  }
  __syncthreads();
  return s_q;
}

__device__ __forceinline__ float jacobi(float d, float r) {
  return d != 0.f ? r / d : r;  // a row without a diagonal is left unscaled
}

// Each thread takes elements i, i + S, ..., i + 5S (S = the grid's threads)
// per pass, all loads issued before any is used, so a thread waits on one
// memory round trip per pass instead of one per element; one pass covers up
// to 608 x 256 x 6 = 933,888 unknowns (the 686k of the hex-mesh system: with
// four per pass, 41% of the threads took a second round trip). A thread's
// share of a dot product is summed in fp32.
constexpr int kPcgUnroll = 6;

// r = b - q (q = A x0), z = D^-1 r, p = z; rz, rr, bb.
__global__ void __launch_bounds__(kPcgThreads) pcg_init(const PcgVectors a) {
  const int S = gridDim.x * kPcgThreads;
  float v[3] = {0.f, 0.f, 0.f};
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

// The three per-iteration kernels are launched with programmatic dependent
// launch: each waits for the kernel before it (whose results it reads) and
// then lets the next one be scheduled, so launch latency overlaps the tail.
__device__ __forceinline__ void pcg_enter() {
  pdl_wait();
  pdl_launch_dependents();
}

// Every block: the grid total of K rows of per-block values parked at
// `partials` by the previous kernel (rows kPcgBlocks apart, `blocks` values
// each), summed in one fixed order: each thread a fixed stride, then
// block_sums. Every block gets the same bits; no block waits for another
// (the previous kernel's completion, via pdl_wait, makes them visible).
// Returned in every thread.
template <int K>
__device__ __forceinline__ void grid_totals(const float* partials, int blocks, float (&tot)[K]) {
  __shared__ float s_tot[K];
  float w[K];
  thread_share<K, false>(partials, blocks, w);
  block_sums<K>(w);
  if (threadIdx.x == 0)
#pragma unroll
    for (int k = 0; k < K; ++k) s_tot[k] = w[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) tot[k] = s_tot[k];
}

// Scalars each kernel reads were written by earlier kernels only: the step
// length kernel parks p . q; the update kernel reads rz (and records it as
// rz_prev for the direction kernel); the direction kernel reads rz_prev and
// writes the new rz, rr, iter and the done flag.

// p . q, per block.
__global__ void __launch_bounds__(kPcgThreads) pcg_alpha(const PcgVectors a) {
  pcg_enter();
  if (a.sc->done) return;
  const int S = gridDim.x * kPcgThreads;
  float v[1] = {0.f};
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
  if (threadIdx.x == 0) a.partials[blockIdx.x] = v[0];
}

// alpha = rz / (p . q); x += alpha p, r -= alpha q, z = D^-1 r; r . z and
// r . r per block. A thread's loads of its first pass are issued before the
// step length is summed, so the two latencies overlap.
struct UpdateLoads {
  float x[kPcgUnroll], p[kPcgUnroll], r[kPcgUnroll], q[kPcgUnroll], d[kPcgUnroll];
};

// x, r and diag: not written by the product before this kernel nor by the
// direction kernel before that (which may still be running under
// programmatic dependent launch), so these loads may go out before the wait.
__device__ __forceinline__ void update_load_xrd(const PcgVectors& a, int i0, int S,
                                                UpdateLoads& L) {
#pragma unroll
  for (int u = 0; u < kPcgUnroll; ++u) {
    const int i = i0 + u * S;
    if (i < a.n) {
      L.x[u] = __ldcg(a.x + i);
      L.r[u] = __ldcg(a.r + i);
      L.d[u] = a.diag[i];
    }
  }
}

// p and q: written by the two kernels before this one; after the wait only.
__device__ __forceinline__ void update_load_pq(const PcgVectors& a, int i0, int S,
                                               UpdateLoads& L) {
#pragma unroll
  for (int u = 0; u < kPcgUnroll; ++u) {
    const int i = i0 + u * S;
    if (i < a.n) {
      L.p[u] = a.p[i];
      L.q[u] = a.q[i];
    }
  }
}

__global__ void __launch_bounds__(kPcgThreads) pcg_update(const PcgVectors a) {
  const int S = gridDim.x * kPcgThreads;
  int i0 = blockIdx.x * kPcgThreads + threadIdx.x;
  UpdateLoads L;
  update_load_xrd(a, i0, S, L);
  pcg_enter();
  update_load_pq(a, i0, S, L);
  // the scalars' loads go out with the partials' (one round trip); a done
  // solve (uniform over the grid) leaves after them
  PcgScalars* sc = a.sc;
  const int done = sc->done;
  const double rz = sc->rz;
  float pq[1];
  grid_totals<1>(a.pq_parts, a.pq_count, pq);
  if (done) return;
  if (!(pq[0] > 0.0f)) {  // p . A p <= 0: A is not positive definite (every block agrees)
    if (blockIdx.x == 0 && threadIdx.x == 0) sc->done = kPcgBreakdown;
    return;
  }
  double alpha_d = 0.0;
  const float alpha = block_ratio(rz, (double)pq[0], &alpha_d);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    sc->alpha = alpha_d;
    sc->rz_prev = rz;
  }
  float v[2] = {0.f, 0.f};
  for (; i0 < a.n; i0 += kPcgUnroll * S) {
    float c[2] = {0.f, 0.f};
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) {
      const int i = i0 + u * S;
      if (i < a.n) {
        a.x[i] = fmaf(alpha, L.p[u], L.x[u]);
        const float ri = fmaf(-alpha, L.q[u], L.r[u]);
        const float zi = jacobi(L.d[u], ri);
        a.r[i] = ri;
        a.z[i] = zi;
        c[0] = fmaf(ri, zi, c[0]);
        c[1] = fmaf(ri, ri, c[1]);
      }
    }
    v[0] += c[0];
    v[1] += c[1];
    if (i0 + kPcgUnroll * S < a.n) {
      update_load_xrd(a, i0 + kPcgUnroll * S, S, L);
      update_load_pq(a, i0 + kPcgUnroll * S, S, L);
    }
  }
  block_sums<2>(v);
  if (threadIdx.x == 0) {
    a.partials[kPcgBlocks + blockIdx.x] = v[0];
    a.partials[2 * kPcgBlocks + blockIdx.x] = v[1];
  }
}

// beta = (r . z) / rz_prev; p = z + beta p; block 0 records the new rz and
// r . r and decides convergence.
__global__ void __launch_bounds__(kPcgThreads) pcg_direction(const PcgVectors a) {
  const int S = gridDim.x * kPcgThreads;
  int i0 = blockIdx.x * kPcgThreads + threadIdx.x;
  // p: last written by the direction kernel of the previous iteration, which
  // has finished once the update kernel before this one passed its wait, so
  // its loads go out before this kernel's wait; z after it
  float zv[kPcgUnroll], pv[kPcgUnroll];
#pragma unroll
  for (int u = 0; u < kPcgUnroll; ++u) {
    const int i = i0 + u * S;
    if (i < a.n) pv[u] = __ldcg(a.p + i);
  }
  pcg_enter();
#pragma unroll
  for (int u = 0; u < kPcgUnroll; ++u) {
    const int i = i0 + u * S;
    if (i < a.n) zv[u] = a.z[i];
  }
  PcgScalars* sc = a.sc;
  const int done = sc->done;
  const double rz_prev = sc->rz_prev;
  // r . z and r . r (only block 0 uses the latter), in one round trip
  float t[2];
  grid_totals<2>(a.partials + kPcgBlocks, gridDim.x, t);
  if (done) {  // solved, stopped or broken down before this iteration
    if (blockIdx.x == 0 && threadIdx.x == 0) set_continue(a, false);
    return;
  }
  double beta_d = 0.0;
  const float beta = block_ratio((double)t[0], rz_prev, &beta_d);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    sc->beta = beta_d;
    sc->rz = t[0];
    sc->rr = t[1];
    sc->iter += 1;
    int state = 0;
    if ((double)t[1] <= sc->tol2 * sc->bb)
      state = kPcgConverged;
    else if (sc->iter >= sc->max_iter)
      state = kPcgMaxIter;
    sc->done = state;
    set_continue(a, state == 0);
  }
  for (; i0 < a.n; i0 += kPcgUnroll * S) {
#pragma unroll
    for (int u = 0; u < kPcgUnroll; ++u) {
      const int i = i0 + u * S;
      if (i < a.n) a.p[i] = fmaf(beta, pv[u], zv[u]);
    }
    if (i0 + kPcgUnroll * S < a.n) {
#pragma unroll
      for (int u = 0; u < kPcgUnroll; ++u) {
        const int i = i0 + kPcgUnroll * S + u * S;
        if (i < a.n) {
          zv[u] = a.z[i];
          pv[u] = a.p[i];
        }
      }
    }
  }
}

}  // namespace

size_t pcg_work_bytes(int n, int product_grid) {
  const size_t vec = ((size_t)n * 4 + 255) / 256 * 256;
  return 4 * vec + 3 * kPcgBlocks * sizeof(float) + 256 + (size_t)product_grid * sizeof(float);
}

int pcg_grid(int n) {
  const int need = (n + kPcgThreads - 1) / kPcgThreads;
  return need < 1 ? 1 : (need < kPcgBlocks ? need : kPcgBlocks);
}

int launch_pcg(int stage, const Plan& p, const float* b, float* x, const float* diag,
               void* stream, unsigned long long cond) {
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
  a.partials = reinterpret_cast<float*>(w + 4 * vec);
  a.sc = reinterpret_cast<PcgScalars*>(w + 4 * vec + 3 * kPcgBlocks * sizeof(float));
  // SELL and FEM products hand over p . q per CTA, after the scalars
  const bool fused = pcg_fused_dot(p);
  a.pq_parts = fused ? reinterpret_cast<float*>(w + 4 * vec + 3 * kPcgBlocks * sizeof(float) + 256)
                     : a.partials;
  a.pq_count = fused ? p.grid : pcg_grid(n);
  a.diag = diag;
  a.cond = cond;
  a.n = n;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = pcg_grid(n);
  if (stage == 0) {
    pcg_init<<<grid, kPcgThreads, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
  }
  void* args[] = {&a};
  const void* fn = stage == 1   ? reinterpret_cast<const void*>(&pcg_alpha)
                   : stage == 2 ? reinterpret_cast<const void*>(&pcg_update)
                                : reinterpret_cast<const void*>(&pcg_direction);
  return launch_pdl(fn, grid, kPcgThreads, 0, stream, args);
}


}  // namespace spmv
