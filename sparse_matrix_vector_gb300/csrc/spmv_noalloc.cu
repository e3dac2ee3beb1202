// y = A x for a CSR matrix that the caller already holds in device memory,
// without a plan and without allocating anything.
//
// Who needs this: code that may not allocate device memory -- a latency-
// critical loop after its set-up phase (cudaMalloc can synchronise the
// device and its cost is unbounded), a component inside a memory pool that
// owns all device memory, or a plug-in that is handed device buffers but no
// allocator. spmv_plan_create allocates (it copies the matrix and its tile
// tables into memory the plan owns), so such callers use this entry point.
//
// How: the nonzeros are cut into fixed slices of kChunk; CTA k streams slice
// k with 16-byte loads, multiplies by the gathered x, parks the products in
// shared memory and writes y for every row that starts inside the slice and
// ends inside it (empty rows included). A row that crosses slice boundaries
// leaves partial sums in a file-scope scratch array: the slice where it
// starts stores a "tail" partial, every later slice it covers stores a
// "head" partial. A second, small kernel adds tail + heads in slice order and
// writes y for those rows, so results are deterministic.
//
// Scratch: one static __device__ array of kScratchBytes (768 KiB) per device
// that loads the library, held until the process exits. All calls share it
// and it keeps the last call's contents; every slot a call reads is written
// earlier in the same call, so nothing needs clearing. Calls that overlap on
// the GPU (different streams, or different host threads) race on it.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/spmv.h"
#include "spmv_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 2048;      // nonzeros per slice (8 per thread)
constexpr int kMaxSlices = 65536; // => at most 134,217,728 nonzeros
constexpr size_t kTailOffset = 0;
constexpr size_t kHeadOffset = (size_t)kMaxSlices * 4;
constexpr size_t kRowOffset = (size_t)kMaxSlices * 8;
constexpr size_t kStatusOffset = (size_t)kMaxSlices * 12;
constexpr size_t kScratchBytes = (size_t)kMaxSlices * 12 + 256;  // 768 KiB + a status word
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct Scratch {
  float* tail;        // [slice] partial of the row that starts in the slice
                      //         and continues past it
  float* head;        // [slice] partial of the row that started before it
  int32_t* tail_row;  // [slice] that row's index, or -1
  int32_t* status;    // checked builds: set when an index was out of range
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// first i in [0, n] with row_ptr[i] >= target (row_ptr is non-decreasing)
__device__ __forceinline__ int lower_bound_rows(const int32_t* row_ptr, int n,
                                                int target) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(row_ptr + mid) < target)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

__device__ __forceinline__ float as_float(float v) { return v; }
__device__ __forceinline__ float as_float(__half v) { return __half2float(v); }

// Four values starting at p, 16-byte (fp32) or 8-byte (fp16) aligned.
__device__ __forceinline__ void load4(const float* p, float (&o)[4]) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void load4(const __half* p, float (&o)[4]) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  const __half2 a = *reinterpret_cast<const __half2*>(&v.x);
  const __half2 b = *reinterpret_cast<const __half2*>(&v.y);
  o[0] = __low2float(a); o[1] = __high2float(a);
  o[2] = __low2float(b); o[3] = __high2float(b);
}

template <typename VT>
__global__ void __launch_bounds__(kThreads)
noalloc_slices(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col,
               const VT* __restrict__ val, const VT* __restrict__ x,
               float* __restrict__ y, int n_rows, int n_cols, int nnz, int n_slices,
               Scratch s) {
  bool bad = false;  // checked builds: an index was out of range
  __shared__ __align__(16) float s_prod[kChunk];
  __shared__ int s_rows[2];
  __shared__ float s_red[kThreads / 32];
  const int tid = threadIdx.x, k = blockIdx.x;
  const int lo = k * kChunk;
  const int hi = min(lo + kChunk, nnz);
  if (tid == 0) {
    s_rows[0] = lower_bound_rows(row_ptr, n_rows, lo);
    s.tail_row[k] = -1;
  }
  if (tid == 1)
    s_rows[1] = k == n_slices - 1 ? n_rows : lower_bound_rows(row_ptr, n_rows, hi);

  // products of the slice's nonzeros; positions past hi hold 0
#pragma unroll
  for (int u = 0; u < kChunk / (4 * kThreads); ++u) {
    const int j = tid + u * kThreads;
    const int i0 = lo + 4 * j;
    float p[4] = {0.f, 0.f, 0.f, 0.f};
    if (i0 + 4 <= hi) {
      int4 c = __ldg(reinterpret_cast<const int4*>(col + i0));
      if (spmv::kChecked) {
        c.x = spmv::checked_col(c.x, n_cols, &bad);
        c.y = spmv::checked_col(c.y, n_cols, &bad);
        c.z = spmv::checked_col(c.z, n_cols, &bad);
        c.w = spmv::checked_col(c.w, n_cols, &bad);
      }
      float v[4];
      load4(val + i0, v);
      p[0] = v[0] * as_float(__ldg(x + c.x));
      p[1] = v[1] * as_float(__ldg(x + c.y));
      p[2] = v[2] * as_float(__ldg(x + c.z));
      p[3] = v[3] * as_float(__ldg(x + c.w));
    } else {
      for (int q = 0; q < 4 && i0 + q < hi; ++q) {
        int c = __ldg(col + i0 + q);
        if (spmv::kChecked) c = spmv::checked_col(c, n_cols, &bad);
        p[q] = as_float(__ldg(val + i0 + q)) * as_float(__ldg(x + c));
      }
    }
    *reinterpret_cast<float4*>(s_prod + 4 * j) = make_float4(p[0], p[1], p[2], p[3]);
  }
  __syncthreads();
  const int rb = s_rows[0], re = s_rows[1];

  // head: nonzeros [lo, min(row_ptr[rb], hi)) belong to a row that started
  // before this slice
  int h_end = min(__ldg(row_ptr + rb), hi) - lo;
  if (spmv::kChecked) h_end = spmv::checked_offset(h_end, 0, hi - lo, &bad);
  if (h_end > 0) {
    float v = 0.f;
    for (int i = tid; i < h_end; i += kThreads) v += s_prod[i];
    v = warp_sum(v);
    if ((tid & 31) == 0) s_red[tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
      float t = tid < kThreads / 32 ? s_red[tid] : 0.f;
      t = warp_sum(t);
      if (tid == 0) s.head[k] = t;
    }
  }

  // rows that start in [lo, hi) (the last slice also owns trailing empty rows)
  const int nrows = re - rb;
  const int avg = nrows > 0 ? (hi - lo) / nrows : 0;
  const int lg = avg <= 8 ? 0 : avg <= 16 ? 1 : avg <= 32 ? 2 : avg <= 64 ? 3
               : avg <= 128 ? 4 : 5;
  const int g = 1 << lg, per_pass = kThreads >> lg;
  const int grp = tid >> lg, lig = tid & (g - 1);
  for (int base = 0; base < nrows; base += per_pass) {
    const int r = rb + base + grp;
    float acc = 0.f;
    int end = 0;
    if (r < re) {
      int b = __ldg(row_ptr + r) - lo;
      end = __ldg(row_ptr + r + 1);
      int e = min(end, hi) - lo;
      if (spmv::kChecked) {
        b = spmv::checked_offset(b, 0, hi - lo, &bad);
        e = spmv::checked_offset(e, 0, hi - lo, &bad);
      }
      for (int i = b + lig; i < e; i += g) acc += s_prod[i];
    }
    for (int o = g >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lig == 0 && r < re) {
      if (end > hi) {
        s.tail[k] = acc;
        s.tail_row[k] = r;
      } else {
        y[r] = acc;
      }
    }
  }
  if (spmv::kChecked && bad) atomicExch(s.status, spmv::kStatusBadIndex);
}

// One thread per slice with a tail: y[row] = tail + heads of the slices the
// row covers, in slice order.
// Every head read here was written by this call: a row r whose tail sits in
// slice k ends in slice last = (row_ptr[r+1] - 1) / kChunk > k, and for each
// slice j in (k, last] the row is still open at its first nonzero lo_j (row r
// started before lo_j and ends after it), so lower_bound gives that slice
// rb > r, row_ptr[rb] > lo_j and h_end > 0: noalloc_slices stores head[j].
__global__ void __launch_bounds__(kThreads)
noalloc_fixup(const int32_t* __restrict__ row_ptr, float* __restrict__ y,
              int n_slices, Scratch s) {
  const int k = blockIdx.x * kThreads + threadIdx.x;
  if (k >= n_slices) return;
  const int r = s.tail_row[k];
  if (r < 0) return;
  int last = (__ldg(row_ptr + r + 1) - 1) / kChunk;
  if (spmv::kChecked) {
    bool bad = false;
    last = spmv::checked_offset(last, k, n_slices - 1, &bad);
    if (bad) atomicExch(s.status, spmv::kStatusBadIndex);
  }
  float v = s.tail[k];
  for (int j = k + 1; j <= last; ++j) v += s.head[j];
  y[r] = v;
}

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does this).
spmv_status scratch_on_current_device(Scratch* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPMV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPMV_ERR_CUDA;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return SPMV_ERR_CUDA;
      }
      g_scratch_addr[dev] = p;
    }
    base = g_scratch_addr[dev];
  }
  unsigned char* b = static_cast<unsigned char*>(base);
  out->tail = reinterpret_cast<float*>(b + kTailOffset);
  out->head = reinterpret_cast<float*>(b + kHeadOffset);
  out->tail_row = reinterpret_cast<int32_t*>(b + kRowOffset);
  out->status = reinterpret_cast<int32_t*>(b + kStatusOffset);
  return SPMV_OK;
}

// True when p points to memory of device `dev` (device or managed memory).
// cudaPointerGetAttributes allocates nothing.
bool on_device(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) &&
         a.device == dev;
}

}  // namespace

extern "C" spmv_status spmv_csr_run_noalloc(int32_t n_rows, int32_t n_cols,
                                            int64_t nnz, const int32_t* row_ptr,
                                            const int32_t* col_idx,
                                            const void* values,
                                            spmv_dtype value_dtype,
                                            const void* x, float* y,
                                            void* stream) {
  if (n_rows < 0 || n_cols < 0 || nnz < 0) return SPMV_ERR_INVALID_ARG;
  if (value_dtype != SPMV_F32 && value_dtype != SPMV_F16) return SPMV_ERR_INVALID_ARG;
  if (nnz > (int64_t)kMaxSlices * kChunk) return SPMV_ERR_TOO_LARGE;
  if (n_rows == 0) return SPMV_OK;
  if (!row_ptr || !y) return SPMV_ERR_INVALID_ARG;
  if (nnz > 0 && (!col_idx || !values || !x || n_cols == 0)) return SPMV_ERR_INVALID_ARG;
  const uintptr_t vs = value_dtype == SPMV_F32 ? 4 : 2;
  if (((uintptr_t)row_ptr & 3u) || ((uintptr_t)y & 3u) || ((uintptr_t)col_idx & 15u) ||
      ((uintptr_t)values & (4 * vs - 1)) || ((uintptr_t)x & (vs - 1)))
    return SPMV_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPMV_ERR_CUDA;
  if (!on_device(row_ptr, dev) || !on_device(y, dev) ||
      (nnz > 0 && (!on_device(col_idx, dev) || !on_device(values, dev) || !on_device(x, dev))))
    return SPMV_ERR_INVALID_ARG;
  Scratch s;
  spmv_status st = scratch_on_current_device(&s);
  if (st != SPMV_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (nnz == 0)
    return cudaMemsetAsync(y, 0, (size_t)n_rows * 4, cs) == cudaSuccess ? SPMV_OK
                                                                       : SPMV_ERR_CUDA;
  int n_slices = (int)((nnz + kChunk - 1) / kChunk);
  int n_rows_arg = n_rows;
  int nnz32 = (int)nnz;
  float* y_arg = y;
  int n_cols_arg = n_cols;
  void* slice_args[] = {&row_ptr, &col_idx, &values, &x, &y_arg, &n_rows_arg,
                        &n_cols_arg, &nnz32, &n_slices, &s};
  const void* slice_fn = value_dtype == SPMV_F32
                             ? reinterpret_cast<const void*>(&noalloc_slices<float>)
                             : reinterpret_cast<const void*>(&noalloc_slices<__half>);
  cudaError_t e = cudaLaunchKernel(slice_fn, dim3((unsigned)n_slices), dim3(kThreads),
                                   slice_args, 0, cs);
  if (e != cudaSuccess) return SPMV_ERR_CUDA;
  void* fix_args[] = {&row_ptr, &y_arg, &n_slices, &s};
  e = cudaLaunchKernel(reinterpret_cast<const void*>(&noalloc_fixup),
                       dim3((unsigned)((n_slices + kThreads - 1) / kThreads)),
                       dim3(kThreads), fix_args, 0, cs);
  return e == cudaSuccess ? SPMV_OK : SPMV_ERR_CUDA;
}

extern "C" int32_t spmv_checked_build(void) { return spmv::kChecked ? 1 : 0; }

extern "C" spmv_status spmv_noalloc_check(void) {
  if (!spmv::kChecked) return SPMV_OK;
  Scratch s;
  spmv_status st = scratch_on_current_device(&s);
  if (st != SPMV_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPMV_ERR_CUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, s.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return SPMV_ERR_CUDA;
  if (word == 0) return SPMV_OK;
  const int32_t zero = 0;
  if (cudaMemcpy(s.status, &zero, 4, cudaMemcpyHostToDevice) != cudaSuccess) return SPMV_ERR_CUDA;
  return SPMV_ERR_DEVICE_STATUS;
}
