// Matrix-free stiffness operator y = K x on a structured hexahedral mesh for
// sm_103a ("Fused FEM matvec" 2.1, 2.2, 5.2): K = sum_e P_e^T (rho_e K0) P_e,
// never assembled.
//
// The page fuses gather, element product and scatter-add into one kernel
// with one thread per element and atomic adds into y. Here the same sum is
// taken from the output side: one thread per node adds, for each of the (up
// to) 8 elements around it, rho_e times the node's 3 rows of K0 times the
// element's 24 values, gathered through L1 element by element (48 registers:
// on GB300 the 120x60x30 mesh takes 11.1 us, against 14.4 us when the 81
// values of the 27 neighbouring nodes are held in registers at once, 85
// registers). Every y entry is written once (no atomics, results
// reproducible run to run), and the only per-element data read is rho_e. K0 travels in the kernel's parameter space: in the
// fully unrolled loops every K0 index is a compile-time constant that is
// the same for all threads, so it is read as a constant-bank operand of the
// fma. The kernel is bound by fp32 fma issue, not by memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "spmv_device.cuh"
#include "spmv_internal.h"

namespace spmv {
namespace {

struct FemArgs {
  const float* __restrict__ rho;  // n_elem densities
  const float* __restrict__ x;    // n_dofs
  float* __restrict__ y;          // n_dofs
  int nex, ney, nez;
  int n_nodes;
  float K0[24 * 24];              // row-major element matrix
};

// Element corner b sits at (hx(b), hy(b), hz(b)): (0,0,0) (1,0,0) (1,1,0)
// (0,1,0), then the same on the top face; local dof 3 b + c.
__host__ __device__ constexpr int hx(int b) { return ((b & 3) == 1 || (b & 3) == 2) ? 1 : 0; }
__host__ __device__ constexpr int hy(int b) { return (b & 3) >= 2 ? 1 : 0; }
__host__ __device__ constexpr int hz(int b) { return b >= 4 ? 1 : 0; }

// Local corner index of position (px, py, pz) in {0, 1}^3.
__host__ __device__ constexpr int corner_of(int px, int py, int pz) {
  return 4 * pz + (py ? (px ? 2 : 3) : (px ? 1 : 0));
}

__global__ void __launch_bounds__(kFemThreads) fem_kernel(const __grid_constant__ FemArgs a) {
  pdl_launch_dependents();
  const int node = blockIdx.x * kFemThreads + threadIdx.x;
  if (node >= a.n_nodes) return;
  const int nnx = a.nex + 1, nny = a.ney + 1;
  const int i = node % nnx, j = (node / nnx) % nny, k = node / (nnx * nny);
  // x and y belong to the stream's earlier work
  pdl_wait();
  float f[3] = {0.f, 0.f, 0.f};
#pragma unroll
  for (int oz = 0; oz < 2; ++oz)
#pragma unroll
    for (int oy = 0; oy < 2; ++oy)
#pragma unroll
      for (int ox = 0; ox < 2; ++ox) {
        const int ex = i - 1 + ox, ey = j - 1 + oy, ez = k - 1 + oz;
        const bool in = ex >= 0 && ex < a.nex && ey >= 0 && ey < a.ney && ez >= 0 && ez < a.nez;
        const int e = in ? ex + a.nex * (ey + a.ney * ez) : 0;
        const float rv = __ldg(a.rho + e);
        const float r = in ? rv : 0.f;
        // the element's 24 values (an element outside the mesh reads
        // element 0's, in bounds, and is weighted by 0)
        const int exx = in ? ex : 0, eyy = in ? ey : 0, ezz = in ? ez : 0;
        float u[24];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const float* p = a.x + 3 * ((exx + hx(b)) + nnx * ((eyy + hy(b)) + nny * (ezz + hz(b))));
#pragma unroll
          for (int cc = 0; cc < 3; ++cc) u[3 * b + cc] = __ldg(p + cc);
        }
        const int an = corner_of(1 - ox, 1 - oy, 1 - oz);
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const float* krow = a.K0 + (3 * an + c) * 24;
          float t = 0.f;
#pragma unroll
          for (int q = 0; q < 24; ++q) t = fmaf(krow[q], u[q], t);
          f[c] = fmaf(r, t, f[c]);
        }
      }
#pragma unroll
  for (int c = 0; c < 3; ++c) a.y[3 * node + c] = f[c];
}

static_assert(corner_of(hx(0), hy(0), hz(0)) == 0 && corner_of(hx(2), hy(2), hz(2)) == 2 &&
                  corner_of(hx(3), hy(3), hz(3)) == 3 && corner_of(hx(5), hy(5), hz(5)) == 5 &&
                  corner_of(hx(7), hy(7), hz(7)) == 7,
              "corner table and its inverse agree");

}  // namespace

int launch_fem(const Plan& p, const void* x, float* y, void* stream) {
  if (p.n_tiles == 0) return 0;
  FemArgs a;
  a.rho = static_cast<const float*>(p.values);
  a.x = static_cast<const float*>(x);
  a.y = y;
  a.nex = p.fem_dims[0];
  a.ney = p.fem_dims[1];
  a.nez = p.fem_dims[2];
  a.n_nodes = (int)p.n_tiles;
  for (int q = 0; q < 24 * 24; ++q) a.K0[q] = p.fem_k0[q];
  void* args[] = {&a};
  return launch_pdl(reinterpret_cast<const void*>(&fem_kernel), p.grid, kFemThreads, 0, stream,
                    args);
}

}  // namespace spmv
