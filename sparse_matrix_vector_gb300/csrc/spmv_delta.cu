// Column-delta kernel of y = A x for sm_103a ("MACKO-SpMV" 2.2): deltas of
// B = 2, 4 or 8 bits, 32 / B to a 32-bit word, fp16 values, fp32
// accumulation.
//
// Work: the planner cuts every row into segments of at most 32 * LW packed
// words (LW = 2 for B = 2, else 4) and gives each warp of the grid a
// contiguous share of the segments, of equal weight. A segment's device block
// (a 32-byte header, its words, its values) is staged by one bulk copy into
// the warp's own ring of kDS shared-memory buffers; lane s of the warp
// issues the copies into buffer s, so warps never wait for one another.
//
// Decode, several lanes per word (4-bit deltas, and 2-bit deltas with
// little padding): L lanes share a word and each takes two of its entries,
// so one warp-wide gather reads x for 32 entries of a few neighbouring words.
// The planner stores each word's column offset, so no scan is needed (see
// wide_pair).
// Decode, a lane per word (8-bit deltas, and 2-bit deltas that are mostly
// padding): lane l takes words l, l + 32, ... of a segment. The column
// before a word is the segment's starting column (stored by the planner)
// plus the fields of every earlier word: the per-word field sums of two
// words' rows are packed in 16-bit halves and prefix-summed over the warp by
// one 5-step __shfl_up_sync scan ("MACKO-SpMV" 2.2.2).
// Either way a word's own columns come from prefix sums of its fields
// computed inside the register (SWAR), and each entry is one shared-memory
// (or L1) gather of x and one mixed-precision fma (the fp16 x fp16 product is
// exact in fp32; the page's half2 product, 2.2.3, would round it).
//
// Rows: each lane keeps fp32 partial sums of the current row piece; at the
// row's last segment, or at the end of the warp's piece of it, the warp
// reduces them. A row inside one share is written at once. A row split into
// two pieces (two warps) meets in one 64-bit exchange per piece (hand_over,
// settle: nothing waits, and the sum is the same bits in either order); a
// row of more pieces leaves one partial per warp, and the warp whose
// atomicAdd completes the row's count adds them in warp order. The planner
// puts the piece of the row a warp shares with the next warp at the front of
// its share, so that both of the warp's hand-overs go out early.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "spmv_device.cuh"
#include "spmv_internal.h"

namespace spmv {
namespace {

#ifndef SPMV_DELTA_WARPS
#define SPMV_DELTA_WARPS 20
#endif
#ifndef SPMV_DELTA_WARPS_B8
#define SPMV_DELTA_WARPS_B8 28
#endif
#ifndef SPMV_DELTA_STAGES
#define SPMV_DELTA_STAGES 2
#endif
#ifndef SPMV_DELTA_GRID_PER_SM
#define SPMV_DELTA_GRID_PER_SM 1
#endif
#ifndef SPMV_DELTA_MIN_BLOCKS
#define SPMV_DELTA_MIN_BLOCKS 1
#endif

// Warps per CTA for B-bit deltas; each has a ring of kDS segment buffers.
// One CTA per SM. Fewer warps leave each thread more registers (the
// several-lanes decode of 4-bit deltas uses 96 at 20 warps, 72 at 28),
// which keeps more of a block's loads and gathers in flight. Measured on the
// 12288^2 LLM matrices (fraction of HBM peak at 30 / 50 / 70 / 90%
// sparsity, before rows of two pieces met in one exchange; after it, 20
// warps x 2 stages 0.88 / 0.84 / 0.70 / 0.51 and 20 x 3 0.85 / 0.83 / 0.67
// / 0.47), 4-bit deltas: 20 warps x 2 stages 0.84 / 0.79 / 0.66 / 0.45;
// 16 x 2 0.83 / 0.79 / 0.66 / 0.45; 24 x 2 0.84 / 0.79 / 0.64 / 0.45; 28 x 2
// 0.80 / 0.79 / 0.63 / 0.43; 16 x 3, 12 x 3, 12 x 4 and 8 x 4 slower; two
// CTAs of 14 x 2 per SM no better, one CTA of 14 x 2 leaving room for the
// next launch's CTA slower. 2-bit deltas at 30 / 70 / 90%: 20 warps 0.71 /
// 0.66 / 0.67, 28 warps 0.71 / 0.63 / 0.65. 8-bit deltas at 50 / 90%: 20
// warps 0.67 / 0.41, 28 warps 0.70 / 0.41.
template <int B>
constexpr int kDW = B == 8 ? SPMV_DELTA_WARPS_B8 : SPMV_DELTA_WARPS;
constexpr int kDS = SPMV_DELTA_STAGES;

struct DeltaArgs {
  const unsigned char* __restrict__ blocks;  // one block per segment
  const int32_t* __restrict__ seg_off;       // block offsets (16-byte steps), n_segs + 1
  const int32_t* __restrict__ warp_first;    // first segment per warp, n_warps + 1
  const int32_t* __restrict__ empty_rows;
  const SplitInfo* __restrict__ splits;      // {first slot, pieces, 0, 0}
  const __half* __restrict__ x;
  float* __restrict__ y;
  float* partials;
  int32_t* counters;
  unsigned long long* cells;  // one per split row, zero between runs
  int32_t* status;
  int n_empty;
  int n_cols;
};

template <int B, bool WIDE = false>
struct Seg {
  static constexpr int kLaneWords = delta_lane_words(B);
  static constexpr int kWords = 32 * kLaneWords;
  static constexpr int kBytes =
      (int)(WIDE ? delta_wide_seg_bytes_max(B) : delta_seg_bytes(B, kWords));
  static_assert(kBytes % 16 == 0, "segment buffers stay 16-byte aligned");
};

// Copy x (n halves) into shared memory with every thread of the CTA, 16
// bytes at a time when x is 16-byte aligned (no barrier: the caller
// synchronises).
__device__ __forceinline__ void copy_x_half(uint16_t* xs, const __half* x, int n) {
  const uint16_t* src = reinterpret_cast<const uint16_t*>(x);
  const int nt = blockDim.x;
  int done = 0;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
    const int nv = n >> 3;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(xs);
    // four loads a thread before their stores: x of up to 32 KB takes one
    // trip to memory
    for (int v0 = 0; v0 < nv; v0 += 4 * nt) {
      uint4 r[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (v0 + k * nt + (int)threadIdx.x < nv) r[k] = __ldg(s4 + v0 + k * nt + threadIdx.x);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (v0 + k * nt + (int)threadIdx.x < nv) d4[v0 + k * nt + threadIdx.x] = r[k];
    }
    done = nv << 3;
  }
  for (int i = done + threadIdx.x; i < n; i += nt) xs[i] = __ldg(src + i);
}

// acc + a * x for the fp16 half `H` of the 32-bit word v and an fp16 x
// (bits): one fp32 rounding, the product being exact in fp32.
template <int H>
__device__ __forceinline__ float fma_half(float acc, uint32_t v, uint16_t xb) {
  if (H == 0)
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "fma.rn.f32.f16 %0, lo, %2, %0;\n\t}"
        : "+f"(acc) : "r"(v), "h"(xb));
  else
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "fma.rn.f32.f16 %0, hi, %2, %0;\n\t}"
        : "+f"(acc) : "r"(v), "h"(xb));
  return acc;
}

// Where x[col] is: its shared-memory byte address (XS), else its global
// address; gathers add a byte offset to it.
template <bool XS>
struct XPtr {
  uint32_t s;        // XS: shared address of x[col]
  const char* g;     // otherwise: global address of x[col]
};

template <bool XS>
__device__ __forceinline__ uint16_t gather(const XPtr<XS>& p, uint32_t off) {
  if (XS) {
    uint16_t v;
    asm("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(p.s + off));
    return v;
  } else {
    return __ldg(reinterpret_cast<const unsigned short*>(p.g + off));
  }
}

// SKZ: the entry's value (fp16 bits `vb`) may be +0.0 -- a padding entry, or
// an explicit zero -- and then x is not read at all (the product is 0 either
// way for finite x): a lane whose entry is padding takes no shared-memory
// bank in that gather.
template <bool XS, bool SKZ>
__device__ __forceinline__ uint16_t gather_v(const XPtr<XS>& p, uint32_t off, uint32_t vb) {
  if (!SKZ) return gather<XS>(p, off);
  if (XS) {
    uint16_t v = 0;
    asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q ld.shared.u16 %0, [%1];\n\t}"
        : "+h"(v) : "r"(p.s + off), "r"(vb));
    return v;
  } else {
    return vb ? __ldg(reinterpret_cast<const unsigned short*>(p.g + off)) : (uint16_t)0;
  }
}

template <bool XS>
__device__ __forceinline__ XPtr<XS> xptr(uint32_t xs_addr, const __half* x, int col) {
  XPtr<XS> p;
  if (XS)
    p.s = xs_addr + 2u * (uint32_t)col;
  else
    p.g = reinterpret_cast<const char*>(x) + 2 * (size_t)col;
  return p;
}

// Per-word decode state: the field sum (S), and doubled prefix sums of the
// fields packed by bytes (B = 2, 4) or 16-bit halves (B = 8):
//  B = 4: with lo / hi the even / odd nibbles spread into bytes, byte j of
//         P = (lo + hi) * 0x01010101 is the sum of nibbles 0..2j+1 (at most
//         120, so no carries) and byte j of Q = P - hi the sum of 0..2j;
//  B = 8: the same with bytes spread into 16-bit halves (at most 1020);
//  B = 2: adjacent fields are first added into nibbles (g); the nibble
//         prefix as for B = 4 gives the sums through fields 4i+1 and 4i+3,
//         and fields 4i and 4i+2 take their upper neighbour back off.
// Offsets are doubled (fp16 x is 2 bytes a column), which still fits a byte
// (at most 240) for B = 2 and 4 and a half (at most 2040) for B = 8.
template <int B>
struct WordPrefix {
  uint32_t P2, Q2;
  int S;
};

template <int B>
__device__ __forceinline__ WordPrefix<B> word_prefix(uint32_t w) {
  WordPrefix<B> r;
  if constexpr (B == 4) {
    const uint32_t lo = (w << 1) & 0x1E1E1E1Eu;
    const uint32_t hi = (w >> 3) & 0x1E1E1E1Eu;
    r.P2 = (lo + hi) * 0x01010101u;
    r.Q2 = r.P2 - hi;
    r.S = (int)(r.P2 >> 25);
  } else if constexpr (B == 8) {
    const uint32_t lo = w & 0x00FF00FFu;
    const uint32_t hi = (w >> 8) & 0x00FF00FFu;
    const uint32_t P = (lo + hi) * 0x00010001u;
    r.P2 = P << 1;
    r.Q2 = (P - hi) << 1;
    r.S = (int)(P >> 16);
  } else {
    const uint32_t g = (w & 0x33333333u) + ((w >> 2) & 0x33333333u);
    const uint32_t lo = (g << 1) & 0x1E1E1E1Eu;
    const uint32_t hi = (g >> 3) & 0x1E1E1E1Eu;
    r.P2 = (lo + hi) * 0x01010101u;  // byte i: 2 x fields 0..4i+3
    r.Q2 = r.P2 - hi;                // byte i: 2 x fields 0..4i+1
    r.S = (int)(r.P2 >> 25);
  }
  return r;
}

// A word's values: 32 / B halves.
template <int B> struct WordVals;
template <> struct WordVals<4> { uint4 v; };
template <> struct WordVals<8> { uint2 v; };
template <> struct WordVals<2> { uint4 v0, v1; };

// Values of word j of a segment of n_w words (B = 2 keeps each word's two
// 16-byte halves in separate planes, so that both loads are conflict-free).
template <int B>
__device__ __forceinline__ WordVals<B> load_vals(const unsigned char* vals, int j, int n_w) {
  WordVals<B> r;
  if constexpr (B == 4) {
    r.v = reinterpret_cast<const uint4*>(vals)[j];
  } else if constexpr (B == 8) {
    r.v = reinterpret_cast<const uint2*>(vals)[j];
  } else {
    r.v0 = reinterpret_cast<const uint4*>(vals)[j];
    r.v1 = reinterpret_cast<const uint4*>(vals)[n_w + j];
  }
  return r;
}

// The two entries held in one 32-bit word of values (halves lo, hi), with
// their gathered x (bits): acc_lo += lo * x_lo, acc_hi += hi * x_hi, each one
// mixed-precision fma (exact product, one fp32 rounding). Measured against
// converting both operands and an fp32 fma, and against a half2 product
// widened and added: the same time, 19% more instructions for either.
__device__ __forceinline__ void fma_pair(float& acc_lo, float& acc_hi, uint32_t v, uint16_t x_lo,
                                         uint16_t x_hi) {
  acc_lo = fma_half<0>(acc_lo, v, x_lo);
  acc_hi = fma_half<1>(acc_hi, v, x_hi);
}

// Accumulate one word whose first entry follows column `col` (p: x at col).
// Four accumulators, entry e of the word into acc[e % 4].
template <int B, bool XS, bool SKZ>
__device__ __forceinline__ void decode_word(uint32_t w, const WordPrefix<B>& pf,
                                            const WordVals<B>& v, const XPtr<XS>& p,
                                            float (&acc)[4]) {
  if constexpr (B == 4) {
    const uint32_t vw[4] = {v.v.x, v.v.y, v.v.z, v.v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t o0 = __byte_perm(pf.Q2, 0u, 0x4440u + (uint32_t)j);
      const uint32_t o1 = __byte_perm(pf.P2, 0u, 0x4440u + (uint32_t)j);
      fma_pair(acc[(2 * j) & 3], acc[(2 * j + 1) & 3], vw[j],
               gather_v<XS, SKZ>(p, o0, vw[j] & 0xFFFFu), gather_v<XS, SKZ>(p, o1, vw[j] >> 16));
    }
  } else if constexpr (B == 8) {
    fma_pair(acc[0], acc[1], v.v.x, gather_v<XS, SKZ>(p, pf.Q2 & 0xFFFFu, v.v.x & 0xFFFFu),
             gather_v<XS, SKZ>(p, pf.P2 & 0xFFFFu, v.v.x >> 16));
    fma_pair(acc[2], acc[3], v.v.y, gather_v<XS, SKZ>(p, pf.Q2 >> 16, v.v.y & 0xFFFFu),
             gather_v<XS, SKZ>(p, pf.P2 >> 16, v.v.y >> 16));
  } else {
    const uint32_t vw[8] = {v.v0.x, v.v0.y, v.v0.z, v.v0.w, v.v1.x, v.v1.y, v.v1.z, v.v1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t o1 = __byte_perm(pf.Q2, 0u, 0x4440u + (uint32_t)i);
      const uint32_t o3 = __byte_perm(pf.P2, 0u, 0x4440u + (uint32_t)i);
      const uint32_t o0 = o1 - ((w >> (8 * i + 1)) & 6u);   // 2 x field 4i+1
      const uint32_t o2 = o3 - ((w >> (8 * i + 5)) & 6u);   // 2 x field 4i+3
      const uint32_t va = vw[2 * i], vb = vw[2 * i + 1];
      fma_pair(acc[0], acc[1], va, gather_v<XS, SKZ>(p, o0, va & 0xFFFFu),
               gather_v<XS, SKZ>(p, o1, va >> 16));
      fma_pair(acc[2], acc[3], vb, gather_v<XS, SKZ>(p, o2, vb & 0xFFFFu),
               gather_v<XS, SKZ>(p, o3, vb >> 16));
    }
  }
}

// Lane 0: stage a segment's block (one bulk copy) into buffer `buf`.
__device__ __forceinline__ void issue_block(unsigned char* buf, uint64_t* bar,
                                           const unsigned char* src, uint32_t bytes,
                                           uint64_t pol) {
  mbar_arrive_expect_tx(bar, bytes);
  bulk_g2s(buf, src, bytes, bar, pol);
}

// Lane 0, after its share: the pieces this warp parked for rows shared with
// other warps are made visible (one fence for all), then each is counted;
// the warp that completes a row's count adds its pieces in warp order, writes
// y and re-arms the count.
__device__ __forceinline__ void finish_pieces(const DeltaArgs& a, const int2 (&pend)[2],
                                              int n_pend) {
  __threadfence();
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    if (p >= n_pend) break;
    const int row = pend[p].x, sid = pend[p].y;
    const SplitInfo si = a.splits[sid];
    if (atomicAdd(a.counters + sid, 1) == si.n_chunks - 1) {
      __threadfence();
      float sum = 0.f;
      for (int j = 0; j < si.n_chunks; ++j) sum += __ldcg(a.partials + si.first_slot + j);
      a.y[row] = sum;
      a.counters[sid] = 0;
    }
  }
}

// Lane l takes words l, l + 32, ... of the segment (LW of them). The column before word 32 k + l is the segment's base plus
// the field sums of rows 0..k-1 and the exclusive prefix of row k; the field
// sums of two rows share one 5-step scan.
template <int B, bool XS, bool SKZ>
__device__ __forceinline__ void decode_segment_lanes(const unsigned char* st, int n_w, int base,
                                                     int lane, uint32_t xs_addr,
                                                     const __half* x, float (&acc)[4]) {
  constexpr int LW = Seg<B>::kLaneWords;
  const uint32_t* s_words = reinterpret_cast<const uint32_t*>(st + kSegHeaderBytes);
  const unsigned char* s_vals = st + kSegHeaderBytes + ((n_w * 4 + 15) & ~15);
  const bool full = n_w == Seg<B>::kWords;  // the common case: no lane idles
  uint32_t w[LW];
  WordPrefix<B> pf[LW];
#pragma unroll
  for (int k = 0; k < LW; ++k) {
    const int j = 32 * k + lane;
    w[k] = (full || j < n_w) ? s_words[j] : 0u;
    pf[k] = word_prefix<B>(w[k]);
  }
  int incl[LW / 2];
#pragma unroll
  for (int q = 0; q < LW / 2; ++q) incl[q] = pf[2 * q].S | (pf[2 * q + 1].S << 16);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int q = 0; q < LW / 2; ++q) {
      const int up = __shfl_up_sync(0xffffffffu, incl[q], o);
      if (lane >= o) incl[q] += up;
    }
  }
  XPtr<XS> xp[LW];
  int col = base;
#pragma unroll
  for (int q = 0; q < LW / 2; ++q) {
    const int tot = __shfl_sync(0xffffffffu, incl[q], 31);
    xp[2 * q] = xptr<XS>(xs_addr, x, col + (incl[q] & 0xFFFF) - pf[2 * q].S);
    col += tot & 0xFFFF;
    xp[2 * q + 1] = xptr<XS>(xs_addr, x, col + (incl[q] >> 16) - pf[2 * q + 1].S);
    col += tot >> 16;
  }
  if (full) {  // one straight-line block: the gathers of all words can overlap
#pragma unroll
    for (int k = 0; k < LW; ++k)
      decode_word<B, XS, SKZ>(w[k], pf[k], load_vals<B>(s_vals, 32 * k + lane, n_w), xp[k], acc);
  } else {
#pragma unroll
    for (int k = 0; k < LW; ++k)
      if (32 * k + lane < n_w)
        decode_word<B, XS, SKZ>(w[k], pf[k], load_vals<B>(s_vals, 32 * k + lane, n_w), xp[k], acc);
  }
}

// Several lanes per word (4 lanes for 4-bit deltas, 8 for 2-bit): lane l
// takes entries 2q and 2q+1 (q = l % L) of word W s + l / L at step s, so
// one warp-wide gather covers 32 entries of a few consecutive words -- a
// narrow window of x whose shared-memory reads spread over the banks (4-bit
// deltas at 50% sparsity: about 2.2 wavefronts per 32 gathers, against 3.2
// when the lanes hold 32 different words). Each word's starting offset
// (doubled, from the segment's base) is stored by the planner, so no scan
// is needed; the lane's two columns come from the word's doubled prefix
// sums (as in word_prefix). Words, offsets and values are stored in blocks
// of four steps, so that a lane loads a block's with three vector loads
// (five shared-memory loads a step, two of them gathers, would otherwise
// fill the load queue).
template <int B, bool XS, bool SKZ>
__device__ __forceinline__ void wide_pair(uint32_t w, uint32_t off, uint32_t v, int q,
                                          const XPtr<XS>& p0, float& acc_lo, float& acc_hi) {
  static_assert(B == 4 || B == 2, "several lanes per word: 2- and 4-bit deltas");
  uint32_t o0, o1;
  if constexpr (B == 4) {
    const uint32_t lo = (w << 1) & 0x1E1E1E1Eu;
    const uint32_t hi = (w >> 3) & 0x1E1E1E1Eu;
    const uint32_t P2 = (lo + hi) * 0x01010101u;  // byte i: 2 x fields 0..2i+1
    const uint32_t sel = 0x4440u + (uint32_t)q;
    o0 = __byte_perm(P2 - hi, 0u, sel);            // 2 x fields 0..2q
    o1 = __byte_perm(P2, 0u, sel);                 // 2 x fields 0..2q+1
  } else {
    const uint32_t g = (w & 0x33333333u) + ((w >> 2) & 0x33333333u);
    const uint32_t lo = (g << 1) & 0x1E1E1E1Eu;
    const uint32_t hi = (g >> 3) & 0x1E1E1E1Eu;
    const uint32_t P2 = (lo + hi) * 0x01010101u;  // byte i: 2 x fields 0..4i+3
    const uint32_t t = (q & 1) ? P2 : P2 - hi;     // byte i: 2 x fields 0..2q+1
    o1 = __byte_perm(t, 0u, 0x4440u + (uint32_t)(q >> 1));
    o0 = o1 - ((w >> (4 * q + 1)) & 6u);           // less 2 x field 2q+1
  }
  fma_pair(acc_lo, acc_hi, v, gather_v<XS, SKZ>(p0, off + o0, v & 0xFFFFu),
           gather_v<XS, SKZ>(p0, off + o1, v >> 16));
}

// The several-lanes layout's constants for B-bit deltas.
template <int B>
struct Wide {
  static constexpr int kL = delta_wide_lanes(B);         // lanes per word
  static constexpr int kW = delta_wide_step_words(B);    // words per step
  static constexpr int kBW = delta_wide_block_words(B);  // words per block of four steps
  static constexpr int kOB = delta_wide_off_bytes(B);    // bytes per word offset
};
template <int B>
using WideOff = std::conditional_t<Wide<B>::kOB == 2, uint16_t, uint32_t>;

// One block of four steps: the lane's four words, offsets and values.
template <int B, bool XS, bool SKZ>
__device__ __forceinline__ void wide_block(const unsigned char* bw, const unsigned char* bo,
                                           const unsigned char* bv, int h, int g, int lane,
                                           int q, const XPtr<XS>& p0, float (&acc)[4]) {
  constexpr int W = Wide<B>::kW;
  const uint4 w = reinterpret_cast<const uint4*>(bw)[h * W + g];
  const uint4 v = reinterpret_cast<const uint4*>(bv)[h * 32 + lane];
  uint32_t o[4];
  if constexpr (Wide<B>::kOB == 2) {
    const uint2 t = reinterpret_cast<const uint2*>(bo)[h * W + g];
    o[0] = t.x & 0xFFFFu;
    o[1] = t.x >> 16;
    o[2] = t.y & 0xFFFFu;
    o[3] = t.y >> 16;
  } else {
    const uint4 t = reinterpret_cast<const uint4*>(bo)[h * W + g];
    o[0] = t.x;
    o[1] = t.y;
    o[2] = t.z;
    o[3] = t.w;
  }
  wide_pair<B, XS, SKZ>(w.x, o[0], v.x, q, p0, acc[0], acc[1]);
  wide_pair<B, XS, SKZ>(w.y, o[1], v.y, q, p0, acc[2], acc[3]);
  wide_pair<B, XS, SKZ>(w.z, o[2], v.z, q, p0, acc[0], acc[1]);
  wide_pair<B, XS, SKZ>(w.w, o[3], v.w, q, p0, acc[2], acc[3]);
}

template <int B, bool XS, bool SKZ>
__device__ __forceinline__ void decode_segment_wide(const unsigned char* st, int n_w, int base,
                                                    int lane, uint32_t xs_addr,
                                                    const __half* x, float (&acc)[4]) {
  constexpr int L = Wide<B>::kL, W = Wide<B>::kW, BW = Wide<B>::kBW, OB = Wide<B>::kOB;
  constexpr int kBlocks = Seg<B, true>::kWords / BW;
  const int g = lane / L, q = lane % L;
  const XPtr<XS> p0 = xptr<XS>(xs_addr, x, base);
  const unsigned char* bw = st + kSegHeaderBytes;
  if (n_w == Seg<B, true>::kWords) {  // the common case: straight-line blocks
    const unsigned char* bo = bw + kBlocks * W * 16;
    const unsigned char* bv = bo + kBlocks * W * 4 * OB;
#pragma unroll
    for (int h = 0; h < kBlocks; ++h) wide_block<B, XS, SKZ>(bw, bo, bv, h, g, lane, q, p0, acc);
    return;
  }
  const int nb = n_w / BW, nt = n_w - nb * BW;
  const unsigned char* bo = bw + nb * W * 16;
  const unsigned char* bv = bo + nb * W * 4 * OB;
  for (int h = 0; h < nb; ++h) wide_block<B, XS, SKZ>(bw, bo, bv, h, g, lane, q, p0, acc);
  // the words after the last whole block, in plain order
  const uint32_t* tw = reinterpret_cast<const uint32_t*>(bv + nb * 512);
  const WideOff<B>* to = reinterpret_cast<const WideOff<B>*>(
      reinterpret_cast<const unsigned char*>(tw) + ((nt * 4 + 15) & ~15));
  const uint32_t* tv = reinterpret_cast<const uint32_t*>(
      reinterpret_cast<const unsigned char*>(to) + ((nt * OB + 15) & ~15));
  for (int t = g; t < nt; t += W)
    wide_pair<B, XS, SKZ>(tw[t], to[t], tv[t * L + q], q, p0, acc[0], acc[1]);
}

template <int B, bool XS, bool SKZ, bool WIDE>
__global__ void __launch_bounds__(kDW<B> * 32, SPMV_DELTA_MIN_BLOCKS)
    delta_seg_kernel(const DeltaArgs a) {
  using Sg = Seg<B, WIDE>;
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  __shared__ __align__(8) uint64_t s_full[kDW<B>][kDS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kDW<B> + warp;
  unsigned char* ring = dyn_smem + (size_t)warp * kDS * Sg::kBytes;
  uint16_t* xs = reinterpret_cast<uint16_t*>(dyn_smem + (size_t)kDW<B> * kDS * Sg::kBytes);
  const int t0 = __ldg(a.warp_first + gw);
  const int n = __ldg(a.warp_first + gw + 1) - t0;
  const uint64_t pol = policy_evict_first();

  // plan-owned data only until pdl_wait: the first kDS blocks of the share.
  // Lane s issues every copy into buffer s (copies issued by one thread
  // complete roughly one after another).
  if (lane == 0) {
    for (int s = 0; s < kDS; ++s) mbar_init(&s_full[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane < kDS && lane < n) {
    const int o0 = __ldg(a.seg_off + t0 + lane), o1 = __ldg(a.seg_off + t0 + lane + 1);
    issue_block(ring + lane * Sg::kBytes, &s_full[warp][lane], a.blocks + (size_t)o0 * 16,
                (uint32_t)(o1 - o0) * 16u, pol);
  }
  if (threadIdx.x == 0) pdl_launch_dependents();
  pdl_wait();
  if (XS) copy_x_half(xs, a.x, a.n_cols);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.n_empty; i += gridDim.x * blockDim.x)
    a.y[__ldg(a.empty_rows + i)] = 0.f;
  if (XS) __syncthreads();
  const uint32_t xs_addr = smem_u32(xs);

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  // pieces of rows shared with other warps (lane 0): {row, split id}; a share
  // holds at most two, its first row's and its last row's
  int2 pend[2];
  int n_pend = 0;
  // lane 0: pieces of rows split in two, each handed over in one exchange
  // whose result is read only after the share: {row, this piece's sum} and
  // the cell's previous content (nonzero: the other piece, which was first)
  Pair pair0, pair1;
  int n_pair = 0;
  int s = 0;
  uint32_t phase = 0;
  int i = 0;
  for (; i < n; ++i) {
    // the warp decides together (its shuffles below need every lane)
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s_full[warp][s], phase))) {
      if (lane == 0) atomicExch(a.status, 1);
      break;
    }
    const unsigned char* st = ring + s * Sg::kBytes;
    const int4 h0 = *reinterpret_cast<const int4*>(st);       // base, row | flags, words, split
    const int4 h1 = *reinterpret_cast<const int4*>(st + 16);  // next block's offset, bytes; slot
    const int n_w = h0.z;
    if constexpr (WIDE)
      decode_segment_wide<B, XS, SKZ>(st, n_w, h0.x, lane, xs_addr, a.x, acc);
    else
      decode_segment_lanes<B, XS, SKZ>(st, n_w, h0.x, lane, xs_addr, a.x, acc);
    // every lane has used the buffer's contents: refill it
    __syncwarp();
    if (lane == s && h1.y > 0)
      issue_block(ring + s * Sg::kBytes, &s_full[warp][s], a.blocks + (size_t)h1.x * 16,
                  (uint32_t)h1.y, pol);
    const uint32_t rf = (uint32_t)h0.y;
    // the row ends, this warp's piece of it does, or this warp's share does
    if ((rf & kSegLast) || (h1.w & kSegCtlPieceEnd) || i == n - 1) {
      const float v = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      if (lane == 0) {
        const int row = (int)(rf & kSegRowMask);
        if (h0.w < 0) {
          a.y[row] = v;
        } else if ((h1.w & kSegCtlPair) && n_pair < 2) {
          if (n_pair == 0)
            pair0 = hand_over(a.cells, h0.w, row, v);
          else
            pair1 = hand_over(a.cells, h0.w, row, v);
          ++n_pair;
        } else if (!(h1.w & kSegCtlPair) && n_pend < 2) {  // park it, count it later
          a.partials[h1.z] = v;
          if (n_pend == 0)
            pend[0] = make_int2(row, h0.w);
          else
            pend[1] = make_int2(row, h0.w);
          ++n_pend;
        } else {
          atomicExch(a.status, 2);  // the plan broke its own rule: report, never write
        }
      }
    }
    // every piece of a shared row this warp holds is parked: count them now,
    // while the warp still has rows to stream, not at the end of the launch
    if ((h1.w & kSegCtlCombine) && lane == 0 && n_pend > 0) {
      finish_pieces(a, pend, n_pend);
      n_pend = 0;
    }
    if (++s == kDS) {
      s = 0;
      phase ^= 1u;
    }
  }
  if (i == n && lane == 0 && n_pend > 0) finish_pieces(a, pend, n_pend);
  if (i == n && lane == 0) {
    if (n_pair > 0) settle(pair0, a.y, a.cells);
    if (n_pair > 1) settle(pair1, a.y, a.cells);
  }
  if (i < n && lane == 0) {
    // a wait gave up: let this warp's copies still in flight land before the
    // CTA's shared memory goes (bounded again)
    for (int j = i; j < n && j < i + kDS; ++j) {
      mbar_wait_bounded(&s_full[warp][s], phase);
      if (++s == kDS) {
        s = 0;
        phase ^= 1u;
      }
    }
  }
}

template <int B, bool SKZ, bool WIDE>
const void* delta_entry_bzw(bool xs) {
  return xs ? reinterpret_cast<const void*>(&delta_seg_kernel<B, true, SKZ, WIDE>)
            : reinterpret_cast<const void*>(&delta_seg_kernel<B, false, SKZ, WIDE>);
}

template <int B, bool WIDE>
const void* delta_entry_bw(bool xs, bool skz) {
  return skz ? delta_entry_bzw<B, true, WIDE>(xs) : delta_entry_bzw<B, false, WIDE>(xs);
}

// wide: several lanes per word, built for 2- and 4-bit deltas
const void* delta_entry(int bits, bool wide, bool xs, bool skz) {
  if (bits == 8) return delta_entry_bw<8, false>(xs, skz);
  if (bits == 2) return wide ? delta_entry_bw<2, true>(xs, skz) : delta_entry_bw<2, false>(xs, skz);
  return wide ? delta_entry_bw<4, true>(xs, skz) : delta_entry_bw<4, false>(xs, skz);
}

}  // namespace

int delta_warps_per_cta(int bits) { return bits == 8 ? kDW<8> : kDW<4>; }

int delta_grid_per_sm(int) { return SPMV_DELTA_GRID_PER_SM; }

int delta_stages(int) { return kDS; }

size_t delta_rings_bytes(int bits, bool wide) {
  const int seg = bits == 8   ? Seg<8>::kBytes
                  : bits == 2 ? (wide ? Seg<2, true>::kBytes : Seg<2>::kBytes)
                              : (wide ? Seg<4, true>::kBytes : Seg<4>::kBytes);
  return (size_t)delta_warps_per_cta(bits) * kDS * seg;
}

size_t delta_x_smem_bytes(int n_cols) { return ((size_t)n_cols * 2 + 15) / 16 * 16; }

int delta_set_smem_limit(int bits, bool wide, size_t dyn) {
  if (dyn == 0) return 0;
  for (bool xs : {false, true})
    for (bool skz : {false, true})
      if (cudaFuncSetAttribute(delta_entry(bits, wide, xs, skz),
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) != cudaSuccess)
        return -1;
  return 0;
}

int delta_kernel_occupancy(int bits, bool wide, bool x_smem, size_t dyn_smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, delta_entry(bits, wide, x_smem, false),
                                                    delta_warps_per_cta(bits) * 32,
                                                    dyn_smem) != cudaSuccess)
    return -1;
  return n;
}

int launch_delta(const Plan& p, const void* x, float* y, void* stream) {
  if (p.grid == 0) return 0;
  DeltaArgs a;
  a.blocks = p.blocks;
  a.seg_off = p.seg_off;
  a.warp_first = p.cta_first;
  a.empty_rows = p.empty_rows;
  a.splits = p.splits;
  a.x = static_cast<const __half*>(x);
  a.y = y;
  a.partials = p.partials;
  a.counters = p.counters;
  a.cells = p.cells;
  a.status = p.status;
  a.n_empty = p.n_empty_rows;
  a.n_cols = p.n_cols;
  void* args[] = {&a};
  return launch_pdl(delta_entry(p.delta_bits, p.delta_wide, p.x_smem, p.delta_skip_zero), p.grid,
                    delta_warps_per_cta(p.delta_bits) * 32, p.dyn_smem, stream, args);
}

}  // namespace spmv
