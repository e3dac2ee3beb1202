// Matrix-free stiffness operator y = K x on a structured hexahedral mesh for
// sm_103a ("Fused FEM matvec" 2.1, 2.2, 5.2): K = sum_e P_e^T (rho_e K0) P_e,
// never assembled.
//
// The page fuses gather, element product and scatter-add into one kernel
// with one thread per element and atomic adds into y. Here the same sum is
// taken from the output side: one thread per node adds, for each of the (up
// to) 8 elements around it, rho_e times the node's 3 rows of K0 times the
// element's 24 values, gathered through L1 element by element. Neighbour
// coordinates are clamped into the mesh once (only elements outside it,
// weighted by rho = 0, ever reach a clamped node), so each gather is a base
// offset plus a constant. Every y entry is written once (no atomics, results
// reproducible run to run), and the only per-element data read is rho_e.
// K0 travels in the kernel's parameter space: in the fully unrolled loops
// every K0 index is a compile-time constant that is the same for all
// threads. The row products use the paired fp32 fma (two independent
// round-to-nearest fmas per instruction, even and odd columns summed
// separately). The kernel is bound by fp32 issue, not by memory. On GB300,
// 120x60x30 mesh: 10.1 us; 10.4 us with scalar fmas, 10.8 us loading each of
// the 27 neighbours once and accumulating per element, 11.1 us without the
// clamped bases, 14.4 us holding all 81 neighbour values in registers,
// 22.9 us staging them in shared memory.
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
  const int* skip;                // when set and nonzero at launch: do nothing
  float* dot;                     // when set: per-block x . y (conjugate gradients)
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
  const bool live = node < a.n_nodes;
  if (!live && !a.dot) return;
  const int nnx = a.nex + 1, nny = a.ney + 1;
  const int i = node % nnx, j = (node / nnx) % nny, k = node / (nnx * nny);
  // x and y belong to the stream's earlier work
  pdl_wait();
  if (a.skip && *a.skip) return;
  float xy = 0.f;  // this node's share of x . y
  if (live) {
    // neighbour coordinates clamped into the mesh: only elements outside the
    // mesh (weighted by rho = 0 below) ever reach a clamped node
    const int xo[3] = {3 * (i > 0 ? i - 1 : 0), 3 * i, 3 * (i + 1 < nnx ? i + 1 : i)};
    const int yc[3] = {j > 0 ? j - 1 : 0, j, j + 1 < nny ? j + 1 : j};
    const int zc[3] = {k > 0 ? k - 1 : 0, k, k + 1 <= a.nez ? k + 1 : k};
    int line[9];  // offset of node (0, j + dy, k + dz) in x, (dz + 1) * 3 + (dy + 1)
#pragma unroll
    for (int dz = 0; dz < 3; ++dz)
#pragma unroll
      for (int dy = 0; dy < 3; ++dy) line[dz * 3 + dy] = 3 * nnx * (yc[dy] + nny * zc[dz]);
    float f[3] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int oz = 0; oz < 2; ++oz)
#pragma unroll
      for (int oy = 0; oy < 2; ++oy)
#pragma unroll
        for (int ox = 0; ox < 2; ++ox) {
          const int ex = i - 1 + ox, ey = j - 1 + oy, ez = k - 1 + oz;
          const bool in = ex >= 0 && ex < a.nex && ey >= 0 && ey < a.ney && ez >= 0 && ez < a.nez;
          const float rv = __ldg(a.rho + (in ? ex + a.nex * (ey + a.ney * ez) : 0));
          const float r = in ? rv : 0.f;
          float u[24];
#pragma unroll
          for (int bb = 0; bb < 8; ++bb) {
            const float* p = a.x + (line[(oz + hz(bb)) * 3 + (oy + hy(bb))] + xo[ox + hx(bb)]);
#pragma unroll
            for (int cc = 0; cc < 3; ++cc) u[3 * bb + cc] = __ldg(p + cc);
          }
          const int an = corner_of(1 - ox, 1 - oy, 1 - oz);
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            const float* krow = a.K0 + (3 * an + c) * 24;
            float2 t2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 12; ++q)
              t2 = __ffma2_rn(make_float2(krow[2 * q], krow[2 * q + 1]),
                              make_float2(u[2 * q], u[2 * q + 1]), t2);
            f[c] = fmaf(r, t2.x + t2.y, f[c]);
          }
        }
#pragma unroll
    for (int c = 0; c < 3; ++c) a.y[3 * node + c] = f[c];
    if (a.dot)
#pragma unroll
      for (int c = 0; c < 3; ++c) xy = fmaf(__ldg(a.x + 3 * node + c), f[c], xy);
  }
  if (a.dot) {  // the block's x . y, summed in a fixed order
    __shared__ float s_red[kFemThreads / 32];
    const float t = block_sum<kFemThreads / 32>(xy, s_red);
    if (threadIdx.x == 0) a.dot[blockIdx.x] = t;
  }
}

static_assert(corner_of(hx(0), hy(0), hz(0)) == 0 && corner_of(hx(2), hy(2), hz(2)) == 2 &&
                  corner_of(hx(3), hy(3), hz(3)) == 3 && corner_of(hx(5), hy(5), hz(5)) == 5 &&
                  corner_of(hx(7), hy(7), hz(7)) == 7,
              "corner table and its inverse agree");

}  // namespace

int launch_fem(const Plan& p, const void* x, float* y, void* stream, const int* skip,
               float* dot) {
  if (p.n_tiles == 0) return 0;
  FemArgs a;
  a.skip = skip;
  a.dot = dot;
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
