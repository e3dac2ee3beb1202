// Column-delta kernel of y = A x for sm_103a ("MACKO-SpMV" 2.2): deltas of
// B = 2, 4 or 8 bits, 32 / B to a 32-bit word, fp16 values, fp32
// accumulation.
//
// A work unit is a slice of one row (at most 512 packed words; 256 when
// B = 2) whose starting column, and each warp's starting column in it, the
// planner stored, so units and warps are independent. The plan keeps each
// unit's starting columns, words and values together in one device block,
// which one bulk copy stages. Lane l of warp w decodes LW words (LW = 1 or
// 2): a per-lane sum of their fields and a 5-step __shfl_up_sync inclusive
// scan give the column before its first entry; a word's columns come from
// prefix sums of its fields computed inside the register, and each entry is
// accumulated with one mixed-precision fma.
// Producer / consumer scheduling: no CTA barrier per unit (see below).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "spmv_device.cuh"
#include "spmv_internal.h"

namespace spmv {
namespace {

struct DeltaArgs {
  // one block per unit: kDeltaWarps starting columns, the unit's words
  // (32 / B deltas of B bits each; padded to 4 words) and their values
  // (32 / B fp16 per word; padded to 16 bytes)
  const unsigned char* __restrict__ blocks;
  const __half* __restrict__ x;
  float* __restrict__ y;
  const int4* __restrict__ units;       // {row | FIRST | LAST, wb, we, block offset / 16}
  const int32_t* __restrict__ cta_first;
  const int32_t* __restrict__ row_split;
  const SplitInfo* __restrict__ splits;  // {first_slot, n_units, row word, words/unit}
  float* partials;
  int32_t* counters;
  int32_t* status;
  int n_cols;
};

// Shared-memory stage of one unit of deltas of B bits: a copy of the unit's
// device block (the warps' starting columns, the words padded to 4, the
// values; 32 / B halves per word).
template <int B>
struct DeltaStage {
  static constexpr int kUnitWords = delta_unit_words(B);
  static constexpr int kBaseBytes = kDeltaWarps * 4;
  static constexpr int kBytes = (int)delta_block_bytes(B, kUnitWords);
  static_assert(kBaseBytes % 16 == 0 && kBytes % 16 == 0 && kUnitWords % 4 == 0,
                "stage regions must stay 16-byte aligned");
};

// A word's values: 32 / B halves.
template <int B> struct WordVals;
template <> struct WordVals<4> { uint4 v; };
template <> struct WordVals<8> { uint2 v; };
template <> struct WordVals<2> { uint4 v0, v1; };

// Copy x (n halves) into shared memory with `nthreads` threads, 16 bytes at a
// time when x is 16-byte aligned (no barrier: the caller synchronises).
__device__ __forceinline__ void copy_x_half(uint16_t* xs, const __half* x, int n, int nthreads) {
  const uint16_t* src = reinterpret_cast<const uint16_t*>(x);
  int done = 0;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
    const int nv = n >> 3;
    for (int v = threadIdx.x; v < nv; v += nthreads)
      reinterpret_cast<uint4*>(xs)[v] = __ldg(reinterpret_cast<const uint4*>(src) + v);
    done = nv << 3;
  }
  for (int i = done + threadIdx.x; i < n; i += nthreads) xs[i] = __ldg(src + i);
}

// Sum of the 32 / B fields of w (at most 48, 120 or 1020).
template <int B>
__device__ __forceinline__ int field_sum(uint32_t w) {
  if (B == 4) {
    const uint32_t b = (w & 0x0F0F0F0Fu) + ((w >> 4) & 0x0F0F0F0Fu);
    return (int)((b * 0x01010101u) >> 24);
  } else if (B == 8) {
    const uint32_t h = (w & 0x00FF00FFu) + ((w >> 8) & 0x00FF00FFu);
    return (int)((h & 0xFFFFu) + (h >> 16));
  } else {
    const uint32_t g = (w & 0x33333333u) + ((w >> 2) & 0x33333333u);
    const uint32_t b = (g & 0x0F0F0F0Fu) + ((g >> 4) & 0x0F0F0F0Fu);
    return (int)((b * 0x01010101u) >> 24);
  }
}

// fp32 acc + a * x for fp16 a and x: the product is exact in fp32, so one
// fp32 rounding (mixed-precision fma).
__device__ __forceinline__ float fma_f16(float acc, uint16_t a, uint16_t x) {
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(x));
  return acc;
}

// x at column col + off, from shared memory (XS) or through L1 (xb = x + col).
template <bool XS>
__device__ __forceinline__ uint16_t gx(const uint16_t* xs, const uint16_t* xb, int col,
                                       uint32_t off) {
  return XS ? xs[col + (int)off] : __ldg(xb + off);
}

// Decode one word whose first entry follows column `col`: the columns come
// from prefix sums of the fields computed several fields at a time inside
// the register (SWAR), and each entry is one gather and one mixed fma.
//  B = 4: with lo / hi the even / odd nibbles spread into bytes, byte j of
//         P = (lo + hi) * 0x01010101 is the sum of nibbles 0..2j+1 (at most
//         120, no carries) and byte j of P - hi the sum of nibbles 0..2j.
//  B = 8: the same with bytes spread into 16-bit halves (at most 1020).
//  B = 2: adjacent fields are first added into nibbles (g); the nibble
//         prefix as for B = 4 gives the sums through fields 4i+1 and 4i+3,
//         and fields 4i and 4i+2 take their upper neighbour back off.
template <int B, bool XS>
__device__ __forceinline__ void decode_word(uint32_t w, const WordVals<B>& v, int& col,
                                            const uint16_t* xs, const __half* x,
                                            float& acc0, float& acc1) {
  const uint16_t* xb = reinterpret_cast<const uint16_t*>(x) + (XS ? 0 : col);
  if constexpr (B == 4) {
    const uint32_t lo = w & 0x0F0F0F0Fu;
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
    const uint32_t P = (lo + hi) * 0x01010101u;
    const uint32_t Q = P - hi;
    const uint32_t vw[4] = {v.v.x, v.v.y, v.v.z, v.v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t o0 = __byte_perm(Q, 0u, 0x4440u + (uint32_t)j);
      const uint32_t o1 = __byte_perm(P, 0u, 0x4440u + (uint32_t)j);
      acc0 = fma_f16(acc0, (uint16_t)(vw[j] & 0xFFFFu), gx<XS>(xs, xb, col, o0));
      acc1 = fma_f16(acc1, (uint16_t)(vw[j] >> 16), gx<XS>(xs, xb, col, o1));
    }
    col += (int)(P >> 24);
  } else if constexpr (B == 8) {
    const uint32_t lo = w & 0x00FF00FFu;
    const uint32_t hi = (w >> 8) & 0x00FF00FFu;
    const uint32_t P = (lo + hi) * 0x00010001u;
    const uint32_t Q = P - hi;
    acc0 = fma_f16(acc0, (uint16_t)(v.v.x & 0xFFFFu), gx<XS>(xs, xb, col, Q & 0xFFFFu));
    acc1 = fma_f16(acc1, (uint16_t)(v.v.x >> 16), gx<XS>(xs, xb, col, P & 0xFFFFu));
    acc0 = fma_f16(acc0, (uint16_t)(v.v.y & 0xFFFFu), gx<XS>(xs, xb, col, Q >> 16));
    acc1 = fma_f16(acc1, (uint16_t)(v.v.y >> 16), gx<XS>(xs, xb, col, P >> 16));
    col += (int)(P >> 16);
  } else {
    const uint32_t g = (w & 0x33333333u) + ((w >> 2) & 0x33333333u);
    const uint32_t lo = g & 0x0F0F0F0Fu;
    const uint32_t hi = (g >> 4) & 0x0F0F0F0Fu;
    const uint32_t P = (lo + hi) * 0x01010101u;  // byte i: fields 0..4i+3
    const uint32_t Q = P - hi;                   // byte i: fields 0..4i+1
    const uint32_t vw[8] = {v.v0.x, v.v0.y, v.v0.z, v.v0.w, v.v1.x, v.v1.y, v.v1.z, v.v1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t o1 = __byte_perm(Q, 0u, 0x4440u + (uint32_t)i);
      const uint32_t o3 = __byte_perm(P, 0u, 0x4440u + (uint32_t)i);
      const uint32_t o0 = o1 - ((w >> (8 * i + 2)) & 3u);
      const uint32_t o2 = o3 - ((w >> (8 * i + 6)) & 3u);
      acc0 = fma_f16(acc0, (uint16_t)(vw[2 * i] & 0xFFFFu), gx<XS>(xs, xb, col, o0));
      acc1 = fma_f16(acc1, (uint16_t)(vw[2 * i] >> 16), gx<XS>(xs, xb, col, o1));
      acc0 = fma_f16(acc0, (uint16_t)(vw[2 * i + 1] & 0xFFFFu), gx<XS>(xs, xb, col, o2));
      acc1 = fma_f16(acc1, (uint16_t)(vw[2 * i + 1] >> 16), gx<XS>(xs, xb, col, o3));
    }
    col += (int)(P >> 24);
  }
}

// Values of word j of a stage.
template <int B>
__device__ __forceinline__ WordVals<B> load_vals(const unsigned char* s_vals, int j) {
  return reinterpret_cast<const WordVals<B>*>(s_vals)[j];
}

// Producer lane: stage unit d (its whole device block, one bulk copy; copies
// issued by one thread complete roughly one after another, so a unit costs one
// of them).
template <int B>
__device__ __forceinline__ void issue_unit(const DeltaArgs& a, unsigned char* stage,
                                           uint64_t* bar, int4* desc, const int4 d,
                                           uint64_t pol) {
  *desc = d;
  const uint32_t bytes = (uint32_t)delta_block_bytes(B, d.z - d.y);
  mbar_arrive_expect_tx(bar, bytes);
  bulk_g2s(stage, a.blocks + (size_t)d.w * 16, bytes, bar, pol);
}

// Thread 0, at the end of this CTA's piece of a row split into units: as
// split_publish for CSR, with units in place of chunks.
__device__ __forceinline__ void delta_publish(const DeltaArgs& a, int row, bool whole,
                                              int wb0, int wb, float part) {
  if (whole) {
    a.y[row] = part;
    return;
  }
  const int sid = __ldg(a.row_split + row);
  const SplitInfo si = a.splits[sid];
  const int k0 = (wb0 - si.row_begin) / si.reserved;
  const int k = (wb - si.row_begin) / si.reserved;
  a.partials[si.first_slot + k0] = part;
  __threadfence();
  const int add = k - k0 + 1;
  const int before = atomicAdd(a.counters + sid, add);
  if (before + add == si.n_chunks) {
    __threadfence();
    float sum = 0.f;
    for (int j = 0; j < si.n_chunks; ++j) {
      sum += __ldcg(a.partials + si.first_slot + j);
      a.partials[si.first_slot + j] = 0.f;
    }
    a.y[row] = sum;
    a.counters[sid] = 0;
  }
}

// One producer lane per group issues the TMA copies; each group's
// kDeltaWarps consumer warps decode its units. A stage is handed back by
// each consumer warp arriving on the stage's "empty" mbarrier once it has
// read it, so consumer warps never wait for one another per unit (no CTA
// barrier in the loop): a warp that is done with a unit moves on to the next
// staged one. A row's total is formed when its last unit ends: each warp
// parks its shuffle-reduced sum in a slot, and the warp whose shared-memory
// atomicAdd completes the slot's count adds the kDeltaWarps sums in warp
// order (deterministic) and publishes the row.
// A CTA holds G groups, each with its own block of units (a "virtual CTA"
// of the plan: v = blockIdx.x * G + g), stage ring and slots; with x in
// shared memory the groups share one copy of it.
#ifndef SPMV_DELTA_PC_STAGES
#define SPMV_DELTA_PC_STAGES 3
#endif
#ifndef SPMV_DELTA_PC_XS_STAGES
#define SPMV_DELTA_PC_XS_STAGES 2
#endif
#ifndef SPMV_DELTA_PC_XS_GROUPS
#define SPMV_DELTA_PC_XS_GROUPS 3
#endif
static_assert(kDeltaMaxLaneWords == 2, "the decode packs at most two words per lane");

template <bool XS>
struct PcCfg {
  static constexpr int kGroups = XS ? SPMV_DELTA_PC_XS_GROUPS : 1;
  static constexpr int kStages = XS ? SPMV_DELTA_PC_XS_STAGES : SPMV_DELTA_PC_STAGES;
  // row sums in flight: a group's warps are less than kStages units apart
  static constexpr int kSlots = kStages + 2;
  static constexpr int kThreads = kGroups * kDeltaThreads + 32;
  static constexpr int kMinBlocks = XS ? 2 : 5;
};

template <int B, bool XS>
__global__ void __launch_bounds__(PcCfg<XS>::kThreads, PcCfg<XS>::kMinBlocks)
    delta_pc_kernel(const DeltaArgs a) {
  using C = PcCfg<XS>;
  using St = DeltaStage<B>;
  constexpr int G = C::kGroups, S = C::kStages;
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  __shared__ __align__(8) uint64_t s_full[G][S];
  __shared__ __align__(8) uint64_t s_empty[G][S];
  __shared__ int4 s_desc[G][S];
  __shared__ float s_part[G][C::kSlots][kDeltaWarps];
  __shared__ int s_cnt[G][C::kSlots];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int g = 0; g < G; ++g) {
      for (int s = 0; s < S; ++s) {
        mbar_init(&s_full[g][s], 1);
        mbar_init(&s_empty[g][s], kDeltaWarps);
      }
      for (int k = 0; k < C::kSlots; ++k) s_cnt[g][k] = 0;
    }
    fence_mbar_init();
  }
  __syncthreads();  // the only CTA-wide barrier

  if (warp == G * kDeltaWarps) {  // producer warp: lane g feeds group g
    if (lane < G) {
      const int g = lane;
      const int v = blockIdx.x * G + g;
      const int u_begin = __ldg(a.cta_first + v);
      const int n_units = __ldg(a.cta_first + v + 1) - u_begin;
      unsigned char* stages = dyn_smem + (size_t)g * S * St::kBytes;
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < n_units; ++i) {
        const int s = i % S;
        if (i >= S && !mbar_wait_bounded(&s_empty[g][s], (uint32_t)(i / S - 1) & 1u)) {
          ok = false;
          break;
        }
        issue_unit<B>(a, stages + s * St::kBytes, &s_full[g][s], &s_desc[g][s],
                      __ldg(a.units + u_begin + i), pol);
        issued = i + 1;
        if (issued == S) pdl_launch_dependents();
      }
      if (issued < S) pdl_launch_dependents();
      if (!ok) {
        atomicExch(a.status, 1);
        // let copies still in flight land before the CTA's shared memory goes
        for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
          mbar_wait_bounded(&s_full[g][j % S], (uint32_t)(j / S) & 1u);
      }
    }
    return;
  }

  // consumers; plan-owned data only above, x and y below
  pdl_wait();
  const int g = warp / kDeltaWarps, lw = warp % kDeltaWarps;
  const uint16_t* xs =
      reinterpret_cast<const uint16_t*>(dyn_smem + (size_t)G * S * St::kBytes);
  if (XS) {
    copy_x_half(const_cast<uint16_t*>(xs), a.x, a.n_cols, G * kDeltaThreads);
    asm volatile("bar.sync 1, %0;" ::"n"(G * kDeltaThreads) : "memory");  // consumers only
  }
  const int v = blockIdx.x * G + g;
  const int u_begin = __ldg(a.cta_first + v);
  const int n_units = __ldg(a.cta_first + v + 1) - u_begin;
  const unsigned char* stages = dyn_smem + (size_t)g * S * St::kBytes;
  float acc0 = 0.f, acc1 = 0.f;  // this thread's share of the current row piece
  int piece_wb0 = -1;
  bool piece_first = false;
  int slot = 0;
  for (int i = 0; i < n_units; ++i) {
    const int s = i % S;
    if (!mbar_wait_bounded(&s_full[g][s], (uint32_t)(i / S) & 1u)) {
      if (lane == 0) atomicExch(a.status, 1);
      break;
    }
    const int4 d = s_desc[g][s];
    const unsigned char* stage = stages + s * St::kBytes;
    const uint32_t rw = (uint32_t)d.x;
    const int row = (int)(rw & kUnitRowMask);
    const int wb = d.y, n_w = d.z - d.y;
    if (piece_wb0 < 0) {
      piece_wb0 = wb;
      piece_first = (rw & kUnitFirst) != 0;
    }
    const int* s_base = reinterpret_cast<const int*>(stage);
    const uint32_t* s_words = reinterpret_cast<const uint32_t*>(stage + St::kBaseBytes);
    const unsigned char* s_vals = stage + St::kBaseBytes + ((n_w + 3) & ~3) * 4;
    // Lane l of warp w takes words 32 LW w + 32 q + l, q < LW: consecutive
    // lanes read consecutive words and values (conflict-free shared-memory
    // loads). The column before word q of a lane is the warp's starting column
    // plus the fields of every earlier word of the warp's segment: one 5-step
    // scan of both words' field sums packed in 16-bit halves (each at most
    // 32 * 1020) gives both. A unit of 2-bit deltas has one word per lane.
    const int lg = St::kUnitWords > kDeltaThreads ? (int)((rw >> kUnitLgShift) & 1u) : 0;
    const int wseg = lw << (5 + lg);                  // first word of the warp's segment
    const int j0 = wseg + lane, j1 = j0 + 32;
    const bool in0 = j0 < n_w, in1 = lg && j1 < n_w;
    const uint32_t w0 = in0 ? s_words[j0] : 0u;
    const uint32_t w1 = in1 ? s_words[j1] : 0u;
    const WordVals<B> v0 = in0 ? load_vals<B>(s_vals, j0) : WordVals<B>{};
    const WordVals<B> v1 = in1 ? load_vals<B>(s_vals, j1) : WordVals<B>{};
    const int ns0 = field_sum<B>(w0), ns1 = field_sum<B>(w1);
    const int base = s_base[lw];
    __syncwarp();
    if (lane == 0) mbar_arrive(&s_empty[g][s]);  // this warp is done with the stage
    int incl = ns0 | (ns1 << 16);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += up;
    }
    const int incl0 = incl & 0xFFFF, incl1 = incl >> 16;
    const int total0 = __shfl_sync(0xffffffffu, incl0, 31);
    if (in0) {
      int col = base + incl0 - ns0;  // column before word j0's first entry
      decode_word<B, XS>(w0, v0, col, xs, a.x, acc0, acc1);
    }
    if (in1) {
      int col = base + total0 + incl1 - ns1;  // column before word j1's first entry
      decode_word<B, XS>(w1, v1, col, xs, a.x, acc0, acc1);
    }
    const bool last = (rw & kUnitLast) != 0;
    if (last || i == n_units - 1) {  // row ends, or this group's share does
      const float vsum = warp_sum(acc0 + acc1);
      if (lane == 0) {
        s_part[g][slot][lw] = vsum;
        __threadfence_block();
        if (atomicAdd(&s_cnt[g][slot], 1) == kDeltaWarps - 1) {
          __threadfence_block();
          const volatile float* sp = s_part[g][slot];
          float t = 0.f;
#pragma unroll
          for (int w2 = 0; w2 < kDeltaWarps; ++w2) t += sp[w2];
          s_cnt[g][slot] = 0;
          delta_publish(a, row, piece_first && last, piece_wb0, wb, t);
        }
      }
      slot = slot + 1 == C::kSlots ? 0 : slot + 1;
      acc0 = acc1 = 0.f;
      piece_wb0 = -1;
    }
  }
}

template <int B>
const void* delta_entry_b(bool xs) {
  return xs ? reinterpret_cast<const void*>(&delta_pc_kernel<B, true>)
            : reinterpret_cast<const void*>(&delta_pc_kernel<B, false>);
}

const void* delta_entry(int bits, bool xs) {
  return bits == 2 ? delta_entry_b<2>(xs) : bits == 8 ? delta_entry_b<8>(xs) : delta_entry_b<4>(xs);
}

template <int B>
size_t stages_bytes_b(bool x_smem) {
  return x_smem ? (size_t)PcCfg<true>::kGroups * PcCfg<true>::kStages * DeltaStage<B>::kBytes
                : (size_t)PcCfg<false>::kGroups * PcCfg<false>::kStages * DeltaStage<B>::kBytes;
}

}  // namespace

int delta_kernel_occupancy(int bits, bool x_smem, size_t dyn_smem, size_t budget) {
  return occupancy_within(delta_entry(bits, x_smem), delta_block(x_smem), dyn_smem, budget);
}

size_t delta_stages_bytes(int bits, bool x_smem) {
  return bits == 2 ? stages_bytes_b<2>(x_smem)
                   : bits == 8 ? stages_bytes_b<8>(x_smem) : stages_bytes_b<4>(x_smem);
}

int delta_groups(bool x_smem) { return x_smem ? PcCfg<true>::kGroups : PcCfg<false>::kGroups; }

int delta_block(bool x_smem) { return x_smem ? PcCfg<true>::kThreads : PcCfg<false>::kThreads; }

size_t delta_x_smem_bytes(int n_cols) { return ((size_t)n_cols + 8) / 8 * 16; }

int delta_set_smem_limit(int bits, size_t dyn) {
  if (dyn == 0) return 0;
  for (bool xs : {false, true})
    if (cudaFuncSetAttribute(delta_entry(bits, xs), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dyn) != cudaSuccess)
      return -1;
  return 0;
}

int launch_delta(const Plan& p, const void* x, float* y, void* stream) {
  if (p.n_tiles == 0) return 0;
  DeltaArgs a;
  a.blocks = p.blocks;
  a.x = static_cast<const __half*>(x);
  a.y = y;
  a.units = reinterpret_cast<const int4*>(p.tiles);
  a.cta_first = p.cta_first;
  a.row_split = p.row_split;
  a.splits = p.splits;
  a.partials = p.partials;
  a.counters = p.counters;
  a.status = p.status;
  a.n_cols = p.n_cols;
  void* args[] = {&a};
  return launch_pdl(delta_entry(p.delta_bits, p.x_smem), p.grid, delta_block(p.x_smem),
                    p.dyn_smem, stream, args);
}

}  // namespace spmv
