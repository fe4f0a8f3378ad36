// decode_impl.cuh -- the decode kernel template (instantiated per activation
// and scale dtype by decode_x<x>_s<s>.cu).
//
// Logits of a weight-only quantised lm_head for small token counts (m <= 16),
// the bandwidth-bound decode case ("Fused WNA16 GEMM for tied quantized
// lm_head logits", Perf evals rows at M = 1; reviewer comment item 1: at
// M = 1 only the bytes moved matter).
//
// Design (sm_103a, one CTA per SM -- 16 warps, 8 when the MMAs take more than
// one 8-column n-tile -- and no cross-warp handshakes on the streaming path):
//  * The vocab is cut into 16-row tiles, split evenly over the CTAs (whole
//    tiles).  Inside a CTA the tiles' "steps" -- 64 packed bytes of every row
//    of a tile, i.e. 128 int4 or 64 int8 columns -- are split evenly over the
//    warps in runs of kPD steps, so warps finish together even when a CTA
//    holds only a few tiles per warp; a tile cut between two warps is summed
//    through shared memory at the end.
//  * Every warp streams its own rows: lane (g, t) copies 16 bytes of row g
//    and of row g + 8 per step with cp.async (eight rows x 64 contiguous
//    bytes per warp instruction) into its own slots of a per-warp ring of
//    kPD steps, and later reads back exactly what it copied -- no handshake
//    with any other lane or warp, no register ring.  Each step's copies go
//    out as soon as the step kPD earlier has been consumed.
//  * Codes become exact 16-bit values offset + u with one LOP3/PRMT
//    (OffsetCodes), multiplied on the tensor cores by mma.sync m16n8k16
//    (vocab rows = M, token columns = N, fp32 accumulation).  The offset
//    times sum(x) over each step's columns is precomputed once per launch
//    and enters the step's first MMA as its accumulator input (negated), so
//    the chain sums exactly x*q; the scale of the step's group (every step
//    lies in one group, or in one per 64-column half) then multiplies it in
//    fp32.
//  * The order of the hidden columns inside one MMA is free (x is permuted
//    the same way), so a lane's 16 copied bytes feed its MMA fragments
//    directly.  For int4 with 64-column groups a step spans two groups:
//    lanes t = 0, 1 hold the first, t = 2, 3 the second.  Each group then
//    gets its own MMA output column (column = 2 * token + group half, the B
//    operand zero where the half does not match), which for m <= 4 costs no
//    extra MMA.
//  * x lives in shared memory for the whole launch (16-byte pieces XOR-
//    swizzled by token), staged while the first weight copies are in flight;
//    for fp16 int4 the columns read from the high nibble of each byte (the
//    code times 16) are pre-scaled by 1/16, saving a shift per word.
//  * Top-K: each warp keeps, per token, a short candidate buffer in shared
//    memory and a threshold (the K-th largest value it has kept so far, a
//    lower bound of the final K-th value).  A finished tile's values are
//    compared against the threshold; the few that reach it are appended.  A
//    buffer about to overflow is compacted to its K best, which raises the
//    threshold.  At the end the CTA takes, per token, the K best of its
//    warps' buffers (K rounds of a warp maximum over all buffers at once)
//    and writes them, sorted, to its slot of the workspace.  The last CTA to take the ticket (acquire-release atomic)
//    reads every slot's first entry; only the slots holding the K largest
//    first entries can hold any of the final K, so it merges those K sorted
//    slots.
//  * Programmatic dependent launch: the kernel lets the next kernel on the
//    stream launch early and reads x, the workspace and the outputs only
//    after griddepcontrol.wait.  With static weights (LogitsArgs::
//    weights_static) the first run's weight copies go out before the wait.
#pragma once

#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm100.cuh"
#include "wql_common.cuh"

namespace wql {
namespace decode_detail {

constexpr int kMaxWarps = 16;
constexpr int kPD = 4;             // steps per run = ring stages per warp
constexpr int kMaxTok = 16;
constexpr int kZeroBytes = 1024;   // zero x region: a run of kPD steps of 16-byte pieces
constexpr int kRingBytes = kPD * 2 * 32 * 16;   // per warp: kPD steps x rows g, g+8 x lanes

// Warps per CTA of a variant: 16 for one n-tile, 8 for more (the wider
// accumulators need more registers and x for 16 tokens more shared memory).
__host__ __device__ constexpr int warps_of(int nt) { return nt == 1 ? 16 : 8; }

struct DecodeParams {
  LogitsArgs a;
  int tiles;         // ceil(n / 16)
  int tpc, tex;      // tiles per CTA: tpc, one more for the first tex CTAs
  int rpt;           // runs (of kPD steps) per tile
  int S;             // steps per tile, padded to a multiple of kPD
  int S_real;        // steps holding packed columns: ceil(row_bytes / 64)
  int group;         // columns per scale group
  int ngroups;       // scale groups per row
  int nunits;        // 64-column units of a (step-padded) row: 2 * S_real (int4) or S_real
  int row_bytes;     // packed bytes per row
  int corr_pitch;    // floats per corr line
  int cap;           // candidate buffer entries per (warp, token): K + 16 to 32
  uint32_t xpitch;   // bytes per token row of x in shared memory
  uint32_t off_x, off_zero, off_corr, off_ring, off_list, off_cnt, off_misc, off_ugrp;
  int early_weights;  // 1: weights may be read before the preceding kernel ends
  int xsum_off;       // floats from the offset sums to the plain sums of x (asym)
  int corr_floats;    // floats of both (cleared at launch)
};

__host__ __device__ constexpr uint32_t round_up_u32(uint32_t v, uint32_t a) {
  return (v + a - 1) / a * a;
}

// 16-byte async copy global -> shared, bypassing L1; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Scale entries are read through L1 (a row's scales serve several steps).
__device__ __forceinline__ uint32_t ldg_scale(const uint16_t* p) {
  uint16_t v;
  asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return (uint32_t)v;
}
__device__ __forceinline__ uint32_t ldg_u8(const uint8_t* p) {
  uint16_t v;
  asm("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return (uint32_t)v;
}
__device__ __forceinline__ uint32_t ldg_scale2(const uint16_t* p) {
  uint32_t v;
  asm("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}


// Code conversion per variant: fp16 int4 reads the high nibble of each byte
// in place (x pre-scaled by 1/16 there); everything else uses OffsetCodes.
template <int BITS, typename XT, bool F8>
struct CodesOf {
  using type = OffsetCodes<BITS, XT>;
  static constexpr bool kScaledX = false;
};
template <>
struct CodesOf<4, __half, false> {
  using type = Int4F16Scaled;
  static constexpr bool kScaledX = true;
};
template <typename XT>
struct CodesOf<8, XT, true> {   // fp8 e4m3 codes: exact values, no offset
  using type = E4M3Codes<XT>;
  static constexpr bool kScaledX = false;
};

// The value the MMA adds per code on top of x*q, per activation element:
// the offset sum of one 16-byte piece of x as stored in shared memory.
template <int BITS, typename XT>
__device__ __forceinline__ float offset_sum(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float lo = 0.f, hi = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float e0 = scale_bits_to_f32<XT>((uint16_t)(w[q] & 0xFFFFu));
    const float e1 = scale_bits_to_f32<XT>((uint16_t)(w[q] >> 16));
    if (CodesOf<BITS, XT, false>::kScaledX && (q & 1)) hi += e0 + e1;
    else lo += e0 + e1;
  }
  if constexpr (CodesOf<BITS, XT, false>::kScaledX) return 1032.0f * lo + 1152.0f * hi;
  else return OffsetCodes<BITS, XT>::kOffset * lo;
}

// The plain sum of one 16-byte piece of x (eight elements).
template <typename XT>
__device__ __forceinline__ float piece_sum(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float r = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    r += scale_bits_to_f32<XT>((uint16_t)(w[q] & 0xFFFFu)) +
         scale_bits_to_f32<XT>((uint16_t)(w[q] >> 16));
  return r;
}

// Swizzle of x's 16-byte pieces inside each aligned run of 8 (by token).
template <bool GW2>
__device__ __forceinline__ uint32_t x_swz(int tok) {
  return GW2 ? (uint32_t)(tok & 3) : (uint32_t)(tok & 7);
}

// m16n8k16 MMAs: accumulating in place (read-write accumulator operands, so
// no copies surround a chain), and the chain's first one with a separate
// accumulator input.
template <typename XT> struct MmaOp;
template <> struct MmaOp<__half> {
  static __device__ __forceinline__ void acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ void first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1, float c0, float c1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%10,%11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
  }
};
template <> struct MmaOp<__nv_bfloat16> {
  static __device__ __forceinline__ void acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ void first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1, float c0, float c1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%10,%11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
  }
};

// Order-preserving 32-bit key of a value (the high half of topk_key).
__device__ __forceinline__ uint32_t value_key(float v) {
  if (v != v) return 0u;
  const uint32_t b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The K best of `count` keys load(i), by one warp (each lane a register
// list, then the lanes merged); returned on every lane in `out`.
template <int KT, typename Load>
__device__ __forceinline__ void warp_topk_of(int count, int K, Load load,
                                             unsigned long long (&out)[KT]) {
  const int lane = threadIdx.x & 31;
  unsigned long long list[KT];
#pragma unroll
  for (int i = 0; i < KT; ++i) list[i] = kEmptyKey;
  for (int i0 = lane; i0 < count; i0 += 4 * 32) {
    unsigned long long v[4];   // four loads in flight per lane
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int i = i0 + b * 32;
      v[b] = i < count ? load(i) : kEmptyKey;
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) list_insert<KT>(list, v[b]);
  }
  warp_merge_topk_redux<KT>(list, K, out);
}

// The largest of a lane's E keys (E a power of two) and its position, by a
// tree of comparisons: log2(E) levels of independent compare-selects instead
// of one chain of E.
template <int E>
__device__ __forceinline__ void lane_max(const unsigned long long (&e)[E], unsigned long long& best,
                                         int& at) {
  unsigned long long v[E];
  int ix[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    v[i] = e[i];
    ix[i] = i;
  }
#pragma unroll
  for (int w = E / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const bool gt = v[i + w] > v[i];
      v[i] = gt ? v[i + w] : v[i];
      ix[i] = gt ? ix[i + w] : ix[i];
    }
  best = v[0];
  at = ix[0];
}

// The K best of keys spread over a warp, E per lane (E a power of two; keys
// unique but for kEmptyKey), by K rounds of a warp-wide maximum (two
// hardware reductions: value half, then index half among the lanes holding
// that value).  Every lane runs every round's update, predicated on holding
// the winner (no divergent branch: a lone winner lane would expose the whole
// update's latency): it clears the winner and finds its next largest -- by a
// tree for E <= 8, by one pass for E = 16 (fewer instructions there).  The
// r-th best ends on lane r.
template <int E>
__device__ __forceinline__ unsigned long long warp_tournament(unsigned long long (&e)[E], int K) {
  static_assert((E & (E - 1)) == 0, "E is a power of two");
  const int lane = threadIdx.x & 31;
  unsigned long long best;
  int at = 0;
  if constexpr (E >= 16) {
    best = e[0];
#pragma unroll
    for (int i = 1; i < E; ++i) best = e[i] > best ? e[i] : best;
  } else {
    lane_max<E>(e, best, at);
  }
  unsigned long long mine = kEmptyKey;
  for (int r = 0; r < K; ++r) {
    const uint32_t hi = (uint32_t)(best >> 32);
    const uint32_t mh = redux_max_u32(hi);
    const uint32_t ml = redux_max_u32(hi == mh ? (uint32_t)best : 0u);
    const unsigned long long top = ((unsigned long long)mh << 32) | ml;
    mine = lane == r ? top : mine;
    const bool win = best == top;   // (with top empty: clears only empties)
    if constexpr (E >= 16) {
      unsigned long long nb = kEmptyKey;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        e[i] = win && e[i] == top ? kEmptyKey : e[i];
        nb = e[i] > nb ? e[i] : nb;
      }
      best = nb;
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) e[i] = win && i == at ? kEmptyKey : e[i];
      lane_max<E>(e, best, at);
    }
  }
  return mine;
}

// The K best of up to 32 sorted lists (descending, kEmptyKey-padded), lane
// l holding list l in registers: K rounds of a warp maximum over the lists'
// heads; the winning lane shifts its list (a predicated shift, no branch).
// The r-th best ends on lane r.
template <int KT>
__device__ __forceinline__ unsigned long long warp_merge_lists(unsigned long long (&lst)[KT],
                                                               int K) {
  const int lane = threadIdx.x & 31;
  unsigned long long mine = kEmptyKey;
  for (int r = 0; r < K; ++r) {
    const unsigned long long head = lst[0];
    const uint32_t hi = (uint32_t)(head >> 32);
    const uint32_t mh = redux_max_u32(hi);
    const uint32_t ml = redux_max_u32(hi == mh ? (uint32_t)head : 0u);
    const unsigned long long top = ((unsigned long long)mh << 32) | ml;
    mine = lane == r ? top : mine;
    const bool win = head == top && top != kEmptyKey;   // the list to shift (branch-free)
#pragma unroll
    for (int i = 0; i < KT - 1; ++i) lst[i] = win ? lst[i + 1] : lst[i];
    lst[KT - 1] = win ? kEmptyKey : lst[KT - 1];
  }
  return mine;
}

// Merge of two sorted lists of K <= 16 keys (best first, kEmptyKey padded,
// keys unique but for kEmptyKey; shared memory) into their K best, best
// first, returned on lanes 0..K-1 and left at out (which may be A): lanes
// 0..15 hold A, lanes 16..31 hold B, each key's rank is its index plus the
// keys of the other list above it (16 shuffles, no rounds), and each key
// below rank K is written at its rank.
__device__ __forceinline__ unsigned long long warp_merge2(const unsigned long long* A,
                                                          const unsigned long long* B, int K,
                                                          unsigned long long* out) {
  const int lane = threadIdx.x & 31;
  const int i = lane & 15;
  const unsigned long long x = i < K ? (lane < 16 ? A[i] : B[i]) : kEmptyKey;
  int r = i;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int src = lane < 16 ? 16 + j : j;
    const uint32_t lo = __shfl_sync(0xFFFFFFFFu, (uint32_t)x, src);
    const uint32_t hi = __shfl_sync(0xFFFFFFFFu, (uint32_t)(x >> 32), src);
    r += (((unsigned long long)hi << 32) | lo) > x ? 1 : 0;
  }
  __syncwarp();
  if (lane < K) out[lane] = kEmptyKey;
  __syncwarp();
  if (x != kEmptyKey && r < K) out[r] = x;
  __syncwarp();
  return lane < K ? out[lane] : kEmptyKey;
}

// Ticket of the last-CTA merge: an atomic add whose release makes this CTA's
// slot writes and threshold update (ordered before it by the preceding block
// barrier) visible before the ticket, and whose acquire, for the last CTA,
// makes the other CTAs' writes visible after it.
__device__ __forceinline__ unsigned int ticket_add(unsigned int* t) {
  unsigned int old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
  return old;
}

// One warp's candidate buffers (shared memory): per token `cap` keys, their
// count, and the threshold -- the value key of the K-th best kept so far
// (0 until a compaction), below which no value can be among the final K.
struct Cands {
  unsigned long long* buf;   // [m][cap]
  unsigned int* cnt;         // [m]
  unsigned int* thr;         // [m]
  int cap;
};

// Reduce a buffer (one of a warp's, or any run of at most 32 keys in shared
// memory) to its K best, sorted best first (kEmptyKey past the count): K
// rounds of a warp maximum over one key per lane.  Sets the count to
// min(count, K) and, with K keys, the threshold to the K-th best's value
// key.  One copy of the code for every call site.  (Arguments by value: a
// reference would put them in local memory.)
static __device__ __noinline__ void compact_buf(unsigned long long* b, unsigned int* cnt,
                                                unsigned int* thr, int cap, int K) {
  const int lane = threadIdx.x & 31;
  const int c = (int)min(*cnt, (unsigned int)cap);
  unsigned long long e[1] = {lane < c ? b[lane] : kEmptyKey};
  const unsigned long long mine = warp_tournament<1>(e, K);
  __syncwarp();
  if (lane < K) b[lane] = mine;
  if (lane == 0) *cnt = (unsigned int)min(c, K);
  if (lane == K - 1 && c >= K) *thr = (uint32_t)(mine >> 32);
  __syncwarp();
}

// The K best of up to 32 sorted lists (descending), lane l passing its own
// list and length (0: none; shared or global memory): K rounds of a warp
// maximum over the lists' heads, the lists held in registers.  The r-th
// best ends on lane r.  One copy of the code for every call site.
static __device__ __noinline__ unsigned long long merge_lists(const unsigned long long* lst_p,
                                                              int len, int K) {
  unsigned long long lst[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) lst[j] = j < len ? lst_p[j] : kEmptyKey;
  return warp_merge_lists<16>(lst, K);
}
__device__ __forceinline__ void compact(const Cands& C, int tk, int K) {
  compact_buf(C.buf + tk * C.cap, C.cnt + tk, C.thr + tk, C.cap, K);
}

// LIN: a step's scale entries are linear in the step -- with two group
// halves, groups of 64 columns with the two halves' entries adjacent and
// 4-byte aligned (one 32-bit load); otherwise one group per step.  Without
// LIN they are looked up per step in a unit -> group table.
template <int BITS, bool GW2, bool LIN, typename XT, typename ST, int NT, int FMT>
__global__ void __launch_bounds__(warps_of(NT) * 32, 1)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr bool F8 = FMT == WQL_FMT_E4M3;
  using Codes = typename CodesOf<BITS, XT, F8>::type;
  constexpr int W = warps_of(NT);
  constexpr int kThr = W * 32;
  constexpr bool kScaledX = CodesOf<BITS, XT, F8>::kScaledX;
  constexpr int kStepCols = BITS == 4 ? 128 : 64;       // columns per step
  constexpr int kLanePieces = kStepCols / 32;           // 16-byte x pieces per lane per step
  constexpr uint32_t kXStepBytes = kStepCols * 2;       // x bytes per step
  constexpr bool kHasOffset = !F8 && !(BITS == 8 && std::is_same<XT, __nv_bfloat16>::value);
  // zero points: int4 with one group per step only (the host enforces it)
  constexpr bool kAsym = FMT == WQL_FMT_ASYM;
  static_assert(!kAsym || (BITS == 4 && !GW2), "zero points: int4, one group per step");

  extern __shared__ __align__(128) uint8_t sm[];
  const LogitsArgs& a = p.a;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int m = a.m, n = a.n, k = a.k;
  const int K = a.topk;

  // ---- this CTA's tiles, this warp's runs of kPD steps ----
  const int bid = (int)blockIdx.x;
  const int T0 = bid * p.tpc + min(bid, p.tex);
  const int T1 = T0 + p.tpc + (bid < p.tex ? 1 : 0);
  const int rpt = p.rpt;                                    // runs per tile
  const int nruns = (T1 - T0) * rpt;
  const int rb = (int)((long long)nruns * warp / W);
  const int re = (int)((long long)nruns * (warp + 1) / W);

  const uint8_t* qw = reinterpret_cast<const uint8_t*>(a.qweight);
  const uint16_t* scales = a.scales;
  const int row_bytes = p.row_bytes;
  const int ng = p.ngroups;
  const uint32_t sm_base = smem_u32(sm);

  // Scale group of each 64-column unit of a row (0xFFFF past k), for the
  // layouts where a step's group is not a shift of its index.
  uint16_t* ugrp = reinterpret_cast<uint16_t*>(sm + p.off_ugrp);
  if (!LIN) {
    for (int u = threadIdx.x; u < p.nunits; u += kThr)
      ugrp[u] = u * 64 < k ? (uint16_t)((u * 64) / p.group) : (uint16_t)0xFFFF;
    __syncthreads();
  }

  // ---- the weight ring: this warp's kPD stages, this lane's two 16-byte
  //      slots per stage (rows g and g + 8) ----
  const uint32_t ring = sm_base + p.off_ring + (uint32_t)warp * kRingBytes + (uint32_t)lane * 16u;
  // stage j, row half h: ring + (2 * j + h) * 512

  // A run's reading position: rows g and g + 8 of its tile (clamped to the
  // last row; rows past n are never stored), its first step, how many of
  // its steps hold columns.
  struct RunPtr {
    const uint8_t* pa;      // rows g / g + 8 at the run's first step and lane t's 16 bytes
    const uint8_t* pb;
    const uint16_t* spa;    // the rows' scale entries (at the run's first group when linear)
    const uint16_t* spb;
    int s0, nsteps;
  };
  auto run_ptr = [&](int tile, int r, bool live) {
    RunPtr rp;
    rp.s0 = r * kPD;
    rp.nsteps = live ? min(kPD, p.S_real - rp.s0) : 0;
    const int ra = min(tile * 16 + g, n - 1), rb8 = min(tile * 16 + g + 8, n - 1);
    rp.pa = qw + (size_t)ra * row_bytes + rp.s0 * 64 + t * 16;
    rp.pb = qw + (size_t)rb8 * row_bytes + rp.s0 * 64 + t * 16;
    // scale entries: linear in the step (at the run's first one), or the
    // rows' first entries for the table lookup
    const int lin0 = LIN ? (GW2 ? 2 * rp.s0 : rp.s0) : 0;
    rp.spa = scales + (size_t)ra * ng + lin0;
    rp.spb = scales + (size_t)rb8 * ng + lin0;
    return rp;
  };
  // The next run of the same tile: everything moves by one run.
  auto run_next = [&](const RunPtr& c, bool live) {
    RunPtr rp = c;
    rp.s0 = c.s0 + kPD;
    rp.nsteps = live ? min(kPD, p.S_real - rp.s0) : 0;
    rp.pa = c.pa + kPD * 64;
    rp.pb = c.pb + kPD * 64;
    if (LIN) {
      rp.spa = c.spa + (GW2 ? 2 * kPD : kPD);
      rp.spb = c.spb + (GW2 ? 2 * kPD : kPD);
    }
    return rp;
  };
  // Step j of a run: its weight copies into stage j (zeros past the row;
  // nothing past the run's steps), as one commit group either way.
  auto copy_step = [&](const RunPtr& rp, int j) {
    if (j < rp.nsteps) {
      const uint32_t src = (rp.s0 + j) * 64 + t * 16 < row_bytes ? 16u : 0u;
      cp_async16(ring + (uint32_t)(2 * j) * 512u, rp.pa + j * 64, src);
      cp_async16(ring + (uint32_t)(2 * j + 1) * 512u, rp.pb + j * 64, src);
    }
    cp_async_commit();
  };
  // The scales of step j of a run (rows g and g + 8).
  auto load_scales = [&](const RunPtr& rp, int j, uint32_t& SA, uint32_t& SB) {
    SA = 0u;
    SB = 0u;
    if (j < rp.nsteps) {
      const int s = rp.s0 + j;
      if constexpr (GW2 && LIN) {   // groups of 64: halves 2s and 2s + 1, adjacent
        SA = ldg_scale2(rp.spa + 2 * j);
        SB = ldg_scale2(rp.spb + 2 * j);
      } else if constexpr (GW2) {
        const int h0 = ugrp[2 * s], h1 = ugrp[2 * s + 1];
        SA = ldg_scale(rp.spa + h0);
        SB = ldg_scale(rp.spb + h0);
        if (h1 != 0xFFFF) {
          SA |= ldg_scale(rp.spa + h1) << 16;
          SB |= ldg_scale(rp.spb + h1) << 16;
        }
      } else {                      // one group per step
        const int gi = LIN ? j : ugrp[BITS == 4 ? 2 * s : s];
        SA = ldg_scale(rp.spa + gi);
        SB = ldg_scale(rp.spb + gi);
        if constexpr (kAsym) {      // the zero points ride in the upper halves
          SA |= ldg_u8(a.zeros + (rp.spa - scales) + gi) << 16;
          SB |= ldg_u8(a.zeros + (rp.spb - scales) + gi) << 16;
        }
      }
    }
  };

  // ---- shared memory ----
  uint8_t* xs = sm + p.off_x;
  float* corr = reinterpret_cast<float*>(sm + p.off_corr);
  int* slot_tile = reinterpret_cast<int*>(sm + p.off_misc);                 // [W]
  unsigned int* flag = reinterpret_cast<unsigned int*>(sm + p.off_misc + kMaxWarps * 4);
  unsigned long long* cbuf = reinterpret_cast<unsigned long long*>(sm + p.off_list);
  unsigned int* ccnt = reinterpret_cast<unsigned int*>(sm + p.off_cnt);      // [2][W][m]

  // This CTA's own shared memory is cleared before the wait for the
  // preceding kernel: the offset sums (entries of tokens past m stay 0), the
  // zero region, the candidate counts and thresholds.
  for (int i = threadIdx.x; i < p.corr_floats; i += kThr) corr[i] = 0.f;
  for (int i = threadIdx.x; i < kZeroBytes / 16; i += kThr)
    *reinterpret_cast<uint4*>(sm + p.off_zero + i * 16) = make_uint4(0u, 0u, 0u, 0u);
  if (K > 0)
    for (int i = threadIdx.x; i < 2 * W * m; i += kThr) ccnt[i] = 0u;

  // With static weights the first run's copies go out before the wait for
  // the preceding kernel on the stream (which then does not write them);
  // otherwise after it.
  const int tile_b = T0 + (rb < re ? rb / rpt : 0);
  const int r_b = rb < re ? rb % rpt : 0;
  const RunPtr run0 = run_ptr(tile_b, r_b, rb < re);
  uint32_t sa[kPD], sb[kPD];
  if (p.early_weights) {
#pragma unroll
    for (int j = 0; j < kPD; ++j) copy_step(run0, j);
  }
  griddep_launch_dependents();
  griddep_wait();
  if (!p.early_weights) {
#pragma unroll
    for (int j = 0; j < kPD; ++j) copy_step(run0, j);
  }
  __syncthreads();   // the cleared offset sums before the atomics below

  // ---- stage x: token rows of xpitch bytes, 16-byte pieces swizzled by
  //      token, columns k .. xpitch/2 zero; each piece's offset sum goes to
  //      its unit (a 64-column half with two group halves, else a step),
  //      negated ----
  {
    const XT* xg = reinterpret_cast<const XT*>(a.x);
    const int pieces = (int)(p.xpitch / 16);
    const int kp = k / 8;
    const int total = m * pieces;
    constexpr int kB = 8;   // pieces in flight per thread
    for (int i0 = threadIdx.x; i0 < total; i0 += kB * kThr) {
      uint4 v[kB];
      int tk[kB], pc[kB];
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int i = i0 + b * kThr;
        tk[b] = i / pieces;   // one division per piece (a handful per thread)
        pc[b] = i - tk[b] * pieces;
        v[b] = make_uint4(0u, 0u, 0u, 0u);
        if (i < total && pc[b] < kp)
          v[b] = *reinterpret_cast<const uint4*>(xg + (size_t)tk[b] * k + pc[b] * 8);
      }
      float xplain[kB];   // plain sums of the pieces (zero points)
#pragma unroll
      for (int b = 0; b < kB; ++b) xplain[b] = kAsym ? piece_sum<XT>(v[b]) : 0.f;
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        if (i0 + b * kThr >= total) continue;
        if constexpr (kScaledX) {   // elements 2, 3, 6, 7 of each 8 -> x / 16
          v[b].y = hmul2_u32(v[b].y, 0x2C002C00u);
          v[b].w = hmul2_u32(v[b].w, 0x2C002C00u);
        }
        const uint32_t q = (uint32_t)pc[b];
        const uint32_t phys = (q & ~7u) | ((q ^ x_swz<GW2>(tk[b])) & 7u);
        *reinterpret_cast<uint4*>(xs + (size_t)tk[b] * p.xpitch + phys * 16) = v[b];
        if (kAsym && pc[b] < kp)
          atomicAdd(&corr[p.xsum_off + (pc[b] / (kStepCols / 8)) * kMaxTok + tk[b]], xplain[b]);
        if (kHasOffset && pc[b] < kp) {
          const float o = offset_sum<BITS, XT>(v[b]);
          if constexpr (GW2) atomicAdd(&corr[tk[b] * p.corr_pitch + (pc[b] >> 3)], -o);
          else atomicAdd(&corr[(pc[b] / (kStepCols / 8)) * kMaxTok + tk[b]], -o);
        }
      }
    }
  }
  __syncthreads();

  // ---- per-lane x addresses (B operand) ----
  //   column of n-tile nt: GW2: 2 * token + half; else: token.  A lane whose
  //   column is a token past m reads what a live lane with the same t reads
  //   (a broadcast; the column is never used).  With GW2, a live column's
  //   lanes of the other group half must give zeros: they read the zero
  //   region, at pieces whose banks the live lanes do not use.
  uint32_t xaddr[NT][kLanePieces];   // step 0's pieces
  bool xzero[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int c = 8 * nt + g;
    int tok = GW2 ? (c >> 1) : c;
    const bool live = tok < m;
    if (!live) tok = m - 1;
    xzero[nt] = GW2 && live && (c & 1) != (t >> 1);
    const uint32_t sw = x_swz<GW2>(tok);
    const uint32_t base = sm_base + p.off_x + (uint32_t)tok * p.xpitch;
#pragma unroll
    for (int i = 0; i < kLanePieces; ++i) {
      const uint32_t pc = (uint32_t)(kLanePieces * t + i);
      // zero lanes: every step of a run reads within the first kPD * 256 bytes
      xaddr[nt][i] = xzero[nt] ? sm_base + p.off_zero + ((pc + 2u) & 7u) * 16u
                               : base + ((pc & ~7u) | ((pc ^ sw) & 7u)) * 16u;
    }
  }
  // the corr entries of this lane's output columns, for step 0
  const float* corr_lane[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
    corr_lane[nt] = GW2 ? corr + (t + 4 * nt) * p.corr_pitch : corr + 8 * nt + 2 * t;

  // ---- candidate buffers and thresholds of this warp ----
  Cands CC{cbuf + (size_t)warp * m * p.cap, ccnt + warp * m, ccnt + W * m + warp * m, p.cap};
  // thresholds of this lane's tokens (GW2: token t + 4 nt; else 8 nt + 2 t + {0, 1})
  uint32_t thr[NT][2];
  auto load_thr = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int t0 = GW2 ? (t + 4 * nt) : (8 * nt + 2 * t);
      thr[nt][0] = t0 < m ? CC.thr[t0] : 0xFFFFFFFFu;
      thr[nt][1] = GW2 ? thr[nt][0] : (t0 + 1 < m ? CC.thr[t0 + 1] : 0xFFFFFFFFu);
    }
  };
  if (K > 0) load_thr();

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;

  const bool head_partial = rb < re && (rb % rpt) != 0 && (rb / rpt + 1) * rpt <= re;
  const int head_tile = T0 + rb / rpt;
  const XT* bias = reinterpret_cast<const XT*>(a.bias);
  XT* logits = reinterpret_cast<XT*>(a.logits);
  // the head tile's partial sums wait in this lane's stash (shared memory)
  float* stash = reinterpret_cast<float*>(sm + p.off_misc + 256) +
                 (size_t)(warp * 32 + lane) * (NT * 4);

  // Store a finished tile's logits; values that reach their token's
  // threshold go to the warp's candidate buffers.
  auto finish_tile = [&](int tile, float (&v)[NT][4]) {
    const int r0 = tile * 16;
    bool pass[NT][4];
    unsigned long long key[NT][4];
    bool any = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        pass[nt][c] = false;
        key[nt][c] = kEmptyKey;
        if (GW2 && (c & 1)) continue;
        const int row = r0 + g + 8 * (c >> 1);
        const int tok = GW2 ? (t + 4 * nt) : (8 * nt + 2 * t + (c & 1));
        if (row < n && tok < m) {
          float val = v[nt][c];
          if (bias) val += to_f32(bias[row]);
          if (logits) logits[(size_t)tok * n + row] = from_f32<XT>(val);
          if (K > 0) {
            key[nt][c] = topk_key(val, (uint32_t)row);
            pass[nt][c] = (uint32_t)(key[nt][c] >> 32) >= thr[nt][c & 1];
            any |= pass[nt][c];
          }
        }
      }
    }
    if (K <= 0 || !__any_sync(0xFFFFFFFFu, any)) return;
    // make room: a token whose buffer would overflow with this tile's
    // passing values is compacted first (raising its threshold), then the
    // values are re-checked (passes only become fewer)
    unsigned int need = 0u;   // tokens to compact (warp-uniform)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < (GW2 ? 1 : 2); ++h) {
        // this tile's passing values of the tokens of (nt, h): lanes of one
        // token share t
        const unsigned int pa = __ballot_sync(0xFFFFFFFFu, pass[nt][h]);
        const unsigned int pb = __ballot_sync(0xFFFFFFFFu, pass[nt][h + 2]);
        if ((pa | pb) == 0u) continue;
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) {
          const int tok = GW2 ? (tq + 4 * nt) : (8 * nt + 2 * tq + h);
          const unsigned int grp = 0x11111111u << tq;
          const unsigned int np = __popc(pa & grp) + __popc(pb & grp);
          if (tok < m && np != 0u && CC.cnt[tok] + np > (unsigned int)CC.cap) need |= 1u << tok;
        }
      }
    const bool compacted = need != 0u;
    while (need) {
      const int tk = __ffs(need) - 1;
      need &= need - 1u;
      compact(CC, tk, K);
    }
    if (compacted) {
      load_thr();
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          pass[nt][c] = pass[nt][c] && (uint32_t)(key[nt][c] >> 32) >= thr[nt][c & 1];
    }
    // appends: the two value slots of a token (rows g and g + 8: c = h and
    // h + 2) go to its buffer with one count read (a broadcast) and one count
    // write by the group's first lane; no atomics -- only this warp touches
    // its buffers and counts until the end of its runs
    const unsigned int lt = (1u << lane) - 1u;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h = 0; h < (GW2 ? 1 : 2); ++h) {
        const unsigned int pa = __ballot_sync(0xFFFFFFFFu, pass[nt][h]);
        const unsigned int pb = __ballot_sync(0xFFFFFFFFu, pass[nt][h + 2]);
        if ((pa | pb) == 0u) continue;                       // (warp-uniform)
        const int tok = GW2 ? (t + 4 * nt) : (8 * nt + 2 * t + h);
        const unsigned int grp = 0x11111111u << t;           // lanes of this token (same t)
        const unsigned int na = __popc(pa & grp), nb = __popc(pb & grp);
        const bool any_t = tok < m && na + nb != 0u;
        const unsigned int base = any_t ? CC.cnt[tok] : 0u;
        __syncwarp();                                        // every read before the write
        if (any_t) {
          unsigned long long* dst = CC.buf + tok * CC.cap + base;
          if (pass[nt][h]) dst[__popc(pa & grp & lt)] = key[nt][h];
          if (pass[nt][h + 2]) dst[na + __popc(pb & grp & lt)] = key[nt][h + 2];
          if (lane == t) CC.cnt[tok] = base + na + nb;
        }
      }
    __syncwarp();
  };

  // One step: the stage's weights (copied by this lane), the x pieces, the
  // MMAs, the scale.
  auto do_step = [&](int j, const uint32_t (&xq)[NT][kLanePieces], const float* const (&cq)[NT],
                     uint32_t scA, uint32_t scB) {
    const uint4 A = lds128(ring + (uint32_t)(2 * j) * 512u);
    const uint4 B = lds128(ring + (uint32_t)(2 * j + 1) * 512u);
    float p0[NT][4], p1[NT][4];
    float c0[NT], c1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 cc = *reinterpret_cast<const float2*>(cq[nt] + (GW2 ? 2 * j : j * kMaxTok));
      c0[nt] = cc.x;
      c1[nt] = cc.y;
    }
    const uint32_t wA[4] = {A.x, A.y, A.z, A.w};
    const uint32_t wB[4] = {B.x, B.y, B.z, B.w};
    if constexpr (BITS == 4) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t qa[4], qb[4];
        Codes::run(wA[i], qa);
        Codes::run(wB[i], qb);
        const uint32_t af0[4] = {qa[0], qb[0], qa[1], qb[1]};
        const uint32_t af1[4] = {qa[2], qb[2], qa[3], qb[3]};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 xv = lds128(xq[nt][i] + (uint32_t)j * (xzero[nt] ? 0u : kXStepBytes));
          float (&pp)[4] = (i & 1) ? p1[nt] : p0[nt];
          if (i < 2) MmaOp<XT>::first(pp, af0, xv.x, xv.y, i == 0 ? c0[nt] : 0.f, i == 0 ? c1[nt] : 0.f);
          else MmaOp<XT>::acc(pp, af0, xv.x, xv.y);
          MmaOp<XT>::acc(pp, af1, xv.z, xv.w);
        }
      }
    } else {
#pragma unroll
      for (int i2 = 0; i2 < 2; ++i2) {
        uint4 xv[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          xv[nt] = lds128(xq[nt][i2] + (uint32_t)j * (xzero[nt] ? 0u : kXStepBytes));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t qa[2], qb[2];
          Codes::run(wA[2 * i2 + h], qa);
          Codes::run(wB[2 * i2 + h], qb);
          const uint32_t af[4] = {qa[0], qb[0], qa[1], qb[1]};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float (&pp)[4] = h ? p1[nt] : p0[nt];
            const uint32_t b0 = h ? xv[nt].z : xv[nt].x, b1 = h ? xv[nt].w : xv[nt].y;
            if (i2 == 0) MmaOp<XT>::first(pp, af, b0, b1, h ? 0.f : c0[nt], h ? 0.f : c1[nt]);
            else MmaOp<XT>::acc(pp, af, b0, b1);
          }
        }
      }
    }
    // the exact scale times the step's sum, in fp32
    if constexpr (GW2) {
      const float fa0 = scale_bits_to_f32<ST>((uint16_t)(scA & 0xFFFFu));
      const float fa1 = scale_bits_to_f32<ST>((uint16_t)(scA >> 16));
      const float fb0 = scale_bits_to_f32<ST>((uint16_t)(scB & 0xFFFFu));
      const float fb1 = scale_bits_to_f32<ST>((uint16_t)(scB >> 16));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        acc[nt][0] = fmaf(fa0, p0[nt][0] + p1[nt][0], fmaf(fa1, p0[nt][1] + p1[nt][1], acc[nt][0]));
        acc[nt][2] = fmaf(fb0, p0[nt][2] + p1[nt][2], fmaf(fb1, p0[nt][3] + p1[nt][3], acc[nt][2]));
      }
    } else {
      const float fa = scale_bits_to_f32<ST>((uint16_t)scA);
      const float fb = scale_bits_to_f32<ST>((uint16_t)scB);
      if constexpr (kAsym) {
        // zero points: sum x*(u - z) = sum x*(u - 8) + (8 - z) * sum x
        const float da = 8.0f - (float)(scA >> 16), db = 8.0f - (float)(scB >> 16);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float2 sx = *reinterpret_cast<const float2*>(cq[nt] + p.xsum_off + j * kMaxTok);
          p0[nt][0] = fmaf(da, sx.x, p0[nt][0]);
          p0[nt][1] = fmaf(da, sx.y, p0[nt][1]);
          p0[nt][2] = fmaf(db, sx.x, p0[nt][2]);
          p0[nt][3] = fmaf(db, sx.y, p0[nt][3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        acc[nt][0] = fmaf(fa, p0[nt][0] + p1[nt][0], acc[nt][0]);
        acc[nt][1] = fmaf(fa, p0[nt][1] + p1[nt][1], acc[nt][1]);
        acc[nt][2] = fmaf(fb, p0[nt][2] + p1[nt][2], acc[nt][2]);
        acc[nt][3] = fmaf(fb, p0[nt][3] + p1[nt][3], acc[nt][3]);
      }
    }
  };

  // ---- main loop over this warp's runs ----
  int cur_tile = tile_b, cur_r = r_b;
  RunPtr cur = run0;
#pragma unroll
  for (int j = 0; j < kPD; ++j) load_scales(cur, j, sa[j], sb[j]);
  for (int q = rb; q < re; ++q) {
    // the next run's position (this warp's runs only) and its scales
    int nx_tile = cur_tile, nx_r = cur_r + 1;
    if (nx_r == rpt) { nx_r = 0; ++nx_tile; }
    const RunPtr nxt = nx_r == 0 ? run_ptr(nx_tile, 0, q + 1 < re) : run_next(cur, q + 1 < re);
    uint32_t sa_n[kPD], sb_n[kPD];
#pragma unroll
    for (int j = 0; j < kPD; ++j) load_scales(nxt, j, sa_n[j], sb_n[j]);
    // this run's x pieces and corr entries
    uint32_t xq[NT][kLanePieces];
    const float* cq[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int i = 0; i < kLanePieces; ++i)
        xq[nt][i] = xzero[nt] ? xaddr[nt][i] : xaddr[nt][i] + (uint32_t)cur.s0 * kXStepBytes;
      cq[nt] = corr_lane[nt] + (GW2 ? 2 * cur.s0 : cur.s0 * kMaxTok);
    }
    if (cur.nsteps == kPD) {
      // a full run: no per-step checks
#pragma unroll
      for (int j = 0; j < kPD; ++j) {
        cp_async_wait<kPD - 1>();   // this step's copies (kPD - 1 later groups may fly)
        do_step(j, xq, cq, sa[j], sb[j]);
        copy_step(nxt, j);          // the stage is free: the next run's step j
      }
    } else {
#pragma unroll
      for (int j = 0; j < kPD; ++j) {
        cp_async_wait<kPD - 1>();
        if (j < cur.nsteps) do_step(j, xq, cq, sa[j], sb[j]);
        copy_step(nxt, j);
      }
    }
#pragma unroll
    for (int j = 0; j < kPD; ++j) {
      sa[j] = sa_n[j];
      sb[j] = sb_n[j];
    }
    // tile end: finish it, or keep it for the merge when it began in a lower warp
    if (cur_r == rpt - 1) {
      if (head_partial && cur_tile == head_tile) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 4; ++c) stash[nt * 4 + c] = acc[nt][c];
      } else {
        finish_tile(cur_tile, acc);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;
    }
    cur = nxt;
    cur_tile = nx_tile;
    cur_r = nx_r;
  }
  cp_async_wait<0>();

  // ---- tiles cut between warps: the unfinished one goes to this warp's
  //      slot (in its own ring, free now) ----
  // slot of warp w: its own ring region (other warps may still be copying
  // into theirs), [32 lanes][NT * 4] floats
  auto slot_of = [&](int w) {
    return reinterpret_cast<float*>(sm + p.off_ring + (size_t)w * kRingBytes) + lane * (NT * 4);
  };
  const bool tail_partial = rb < re && (re % rpt) != 0;
  // -1: no unfinished tile; -2: no steps at all (skipped by the merge)
  if (lane == 0) slot_tile[warp] = rb >= re ? -2 : tail_partial ? T0 + (re - 1) / rpt : -1;
  if (tail_partial) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) slot_of(warp)[nt * 4 + c] = acc[nt][c];
  }
  __syncthreads();
  if (head_partial) {
    float head[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) head[nt][c] = stash[nt * 4 + c];
    for (int w = warp - 1; w >= 0 && (slot_tile[w] == head_tile || slot_tile[w] == -2); --w) {
      if (slot_tile[w] == -2) continue;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) head[nt][c] += slot_of(w)[nt * 4 + c];
    }
    finish_tile(head_tile, head);
  }
  if (K <= 0) return;

  // ---- top-K of this CTA ----
  // Every warp's buffer holds, per token, all of its values that can be
  // among its K best.  The K best of the W buffers of a token (lane l holds
  // entry l of every buffer: K rounds of a warp maximum) -- with enough
  // warps, two warps take half of the buffers each and one merges their two
  // sorted lists -- go, best first, to the CTA's slot.
  __syncthreads();   // every warp's buffers are final
  if (2 * m <= W) {
    // two warps per token, each over half of the buffers, then one merge
    constexpr int H = W / 2;
    unsigned long long* half_best = reinterpret_cast<unsigned long long*>(sm + p.off_ring);  // [m][2][16]
    if (warp < 2 * m) {
      const int tk = warp >> 1, part = warp & 1;
      unsigned long long e[H];
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const int b = part * H + i;
        const int c = (int)min(ccnt[b * m + tk], (unsigned int)p.cap);
        e[i] = lane < c ? cbuf[((size_t)b * m + tk) * p.cap + lane] : kEmptyKey;
      }
      const unsigned long long mine = warp_tournament<H>(e, K);
      if (lane < 16) half_best[(tk * 2 + part) * 16 + lane] = lane < K ? mine : kEmptyKey;
    }
    __syncthreads();
    for (int tk = warp; tk < m; tk += W) {
      const unsigned long long mine =
          warp_merge2(half_best + tk * 32, half_best + tk * 32 + 16, K, half_best + tk * 32);
      if (lane < K) a.cand[((size_t)tk * WQL_MAX_CTAS + blockIdx.x) * K + lane] = mine;
    }
  } else {
    for (int tk = warp; tk < m; tk += W) {
      unsigned long long e[W];
#pragma unroll
      for (int i = 0; i < W; ++i) {
        const int c = (int)min(ccnt[i * m + tk], (unsigned int)p.cap);
        e[i] = lane < c ? cbuf[((size_t)i * m + tk) * p.cap + lane] : kEmptyKey;
      }
      const unsigned long long mine = warp_tournament<W>(e, K);
      if (lane < K) a.cand[((size_t)tk * WQL_MAX_CTAS + blockIdx.x) * K + lane] = mine;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *flag = (ticket_add(a.counter) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (*flag == 0u) return;

  // ---- last CTA ----
  // The slots are sorted and hold disjoint rows, so every slot whose first
  // entry is below the K-th largest first entry holds nothing of the final
  // K (K larger keys exist).  Per token: every slot's first entry (one round
  // trip, staged in the free ring), the K best of them (K rounds of a warp
  // maximum), and the merge of those K slots.
  const int nsrc = (int)gridDim.x;
  unsigned long long* heads = reinterpret_cast<unsigned long long*>(sm + p.off_ring);  // [m][nsrc]
  const bool staged = nsrc <= 256 && (size_t)m * nsrc * 8u <= (size_t)W * kRingBytes;
  if (staged) {
    const int total = m * nsrc;
    constexpr int kB = 8;   // loads per thread in flight
    for (int i0 = threadIdx.x; i0 < total; i0 += kB * kThr) {
      unsigned long long v[kB];
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int i = i0 + b * kThr;
        const int tk = i / nsrc;
        v[b] = i < total ? __ldcg(a.cand + ((size_t)tk * WQL_MAX_CTAS + (i - tk * nsrc)) * K)
                         : kEmptyKey;
      }
#pragma unroll
      for (int b = 0; b < kB; ++b)
        if (i0 + b * kThr < total) heads[i0 + b * kThr] = v[b];
    }
    __syncthreads();
  }
  const int big = p.tex * (p.tpc + 1);   // tiles of the CTAs holding tpc + 1
  for (int tk = warp; tk < m; tk += W) {
    const unsigned long long* slots = a.cand + (size_t)tk * WQL_MAX_CTAS * K;
    unsigned long long mine;
    if (staged) {
      unsigned long long e[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        e[q] = lane + 32 * q < nsrc ? heads[tk * nsrc + lane + 32 * q] : kEmptyKey;
      const unsigned long long hk = warp_tournament<8>(e, K);
      int sid = -1;            // lane r: the CTA of the r-th best first entry
      if (hk != kEmptyKey) {
        const int tile = key_index(hk) >> 4;
        sid = tile < big ? tile / (p.tpc + 1) : p.tex + (tile - big) / p.tpc;
      }
      mine = merge_lists(slots + (size_t)(sid >= 0 ? sid : 0) * K, sid >= 0 ? K : 0, K);
    } else {
      // more slots than staged: every slot, straight from the workspace
      unsigned long long best[16];
      warp_topk_of<16>(nsrc * K, K, [&](int i) { return __ldcg(slots + i); }, best);
      mine = pick(best, lane);
    }
    if (__ldcg(a.counter + 1) != 0u) mine = kEmptyKey;   // a recorded timeout voids results
    if (lane < K) {
      a.topk_idx[(size_t)tk * K + lane] = mine != kEmptyKey ? key_index(mine) : -1;
      a.topk_val[(size_t)tk * K + lane] = mine != kEmptyKey ? key_value(mine) : __int_as_float(0x7FC00000);
    }
  }
  // ready for the next call
  if (threadIdx.x == 0) *a.counter = 0u;
}

template <int BITS, bool GW2, bool LIN, typename XT, typename ST, int NT, int FMT = WQL_FMT_SYM>
cudaError_t launch_t(const DecodeParams& p, size_t smem, int ctas, cudaStream_t s) {
  auto kern = decode_kernel<BITS, GW2, LIN, XT, ST, NT, FMT>;
  // per instantiation: raise the dynamic smem limit when a launch needs more,
  // and ask for the smallest shared-memory carveout that holds it, leaving
  // the rest of the SM's 256 KB to L1 (scale rows are read through L1)
  static size_t configured = 0;
  static int carveout = -1;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const int pct = (int)(((smem + 1024) * 100 + 228 * 1024 - 1) / (228 * 1024));
  if (pct != carveout) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         pct > 100 ? 100 : pct);
    if (e != cudaSuccess) return e;
    carveout = pct;
  }
  const cudaError_t e = launch_pdl(kern, dim3((unsigned)ctas), dim3(warps_of(NT) * 32), smem, s, p);
  note_launch();
  return e;
}

template <bool LIN, typename XT, typename ST>
cudaError_t dispatch_lin(const DecodeParams& p, bool gw2, int nt, size_t smem, int ctas,
                         cudaStream_t s) {
  if (p.a.bits == 4 && gw2) {
    if (nt == 1) return launch_t<4, true, LIN, XT, ST, 1>(p, smem, ctas, s);
    if (nt == 2) return launch_t<4, true, LIN, XT, ST, 2>(p, smem, ctas, s);
    return launch_t<4, true, LIN, XT, ST, 4>(p, smem, ctas, s);
  }
  if (p.a.bits == 4 && p.a.format == WQL_FMT_ASYM) {
    if (nt == 1) return launch_t<4, false, LIN, XT, ST, 1, WQL_FMT_ASYM>(p, smem, ctas, s);
    return launch_t<4, false, LIN, XT, ST, 2, WQL_FMT_ASYM>(p, smem, ctas, s);
  }
  if (p.a.bits == 4) {
    if (nt == 1) return launch_t<4, false, LIN, XT, ST, 1>(p, smem, ctas, s);
    return launch_t<4, false, LIN, XT, ST, 2>(p, smem, ctas, s);
  }
  if (p.a.format == WQL_FMT_E4M3) {
    if (nt == 1) return launch_t<8, false, LIN, XT, ST, 1, WQL_FMT_E4M3>(p, smem, ctas, s);
    return launch_t<8, false, LIN, XT, ST, 2, WQL_FMT_E4M3>(p, smem, ctas, s);
  }
  if (nt == 1) return launch_t<8, false, LIN, XT, ST, 1>(p, smem, ctas, s);
  return launch_t<8, false, LIN, XT, ST, 2>(p, smem, ctas, s);
}

// Every variant for one activation and scale dtype.
template <typename XT, typename ST>
cudaError_t dispatch_xs(const DecodeParams& p, bool gw2, bool lin, int nt, size_t smem, int ctas,
                        cudaStream_t s) {
  return lin ? dispatch_lin<true, XT, ST>(p, gw2, nt, smem, ctas, s)
             : dispatch_lin<false, XT, ST>(p, gw2, nt, smem, ctas, s);
}

}  // namespace decode_detail
}  // namespace wql
