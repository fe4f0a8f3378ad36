// decode_impl.cuh -- the decode kernel template (included by decode_f16.cu and
// decode_bf16.cu, which instantiate it per activation dtype).
//
// Logits of a weight-only quantised lm_head for small token
// counts (m <= 16), the bandwidth-bound decode case ("Fused WNA16 GEMM for
// tied quantized lm_head logits", Perf evals rows at M = 1; reviewer comment
// item 1: at M = 1 only the bytes moved matter).
//
// Design (sm_103a, one persistent CTA per SM):
//  * Work comes in units of up to 16 16-row vocab tiles (256 rows).  A CTA
//    starts with the unit of its own index and takes further ones from a
//    counter in the workspace, so CTAs whose copies stream faster take more
//    (static strided units when there is no workspace).  Each unit streams
//    along the hidden dimension in chunks of 128 packed bytes per row (256
//    int4 or 128 int8 codes).
//  * Warp 16 is the producer: one lane issues TMA tensor copies of every
//    chunk (16-row boxes, 128B-swizzled) and, once per unit, a bulk copy of
//    the unit's scale rows, into a 4-stage ring; each stage carries its unit
//    id, and a last stage with id -1 tells the consumers to stop.  Activations are either
//    resident in shared memory for the whole launch or, when m*k is too
//    large for that, copied per chunk with the weights.
//  * Warps 0..15 are consumers, one 16-row tile each.  ldmatrix moves packed
//    words straight into the A-fragment layout of a warp MMA (m16n8k16, swap
//    AB: vocab rows = M, tokens = N).  A code becomes the exact 16-bit value
//    magic + u with one LOP3 (OffsetCodes); the MMA sums x*(q + offset) with
//    exact products and fp32 accumulation, and offset * sum(x) -- computed
//    once per launch for every (token, group) -- is subtracted per scale
//    group before the exact fp32 scale multiply.
//  * Top-K: the fp32 logits of the CTA's rows go to shared memory (or, when
//    they do not fit, a global scratch row).  Each CTA takes a threshold per
//    token -- the K-th largest of each warp's lane maxima, a lower bound of
//    the K-th largest value -- keeps the rows at or above it and selects its
//    top-K from those; it raises a per-token global bound with its K-th
//    value and appends those of its K that reach the bound (as it stands
//    after its own raise) to a per-token list in the workspace.  The last
//    CTA to finish (atomic ticket, no waiting) ranks that short list: every
//    entry of the final top-K reaches the final bound, hence the bound at
//    its CTA's append, so it is on the list.
//  * All mbarrier waits are bounded; a timeout sets the workspace error word
//    and the CTA finishes without issuing further copies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm100.cuh"
#include "wql_common.cuh"

namespace wql {
namespace decode_detail {

constexpr int kConsumers = 16;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kWarpsAll = kThreads / 32;
constexpr int kBlockTiles = kConsumers;          // 16-row tiles per block
constexpr int kChunkRowBytes = 128;              // packed bytes per row per chunk
constexpr int kTileBytes = 16 * kChunkRowBytes;  // one TMA box
constexpr int kStageWBytes = kBlockTiles * kTileBytes;
constexpr int kStages = 4;
constexpr int kMaxTok = 16;
constexpr int kConsumerBarrier = 1;              // named barrier for the consumer warps
constexpr int kSelCap = 256;                     // candidate slots per token in the selection
constexpr int kTauWord = 16;                     // workspace word of token 0's global bound
constexpr int kNCandWord = 32;                   // workspace word of token 0's candidate count

struct DecodeParams {
  LogitsArgs a;
  int tiles_total;      // ceil(n / 16)
  int unit_tiles;       // 16-row tiles per work unit (a power of two <= kBlockTiles)
  int unit_rows_log2;   // log2(16 * unit_tiles)
  int units_total;      // ceil(tiles_total / unit_tiles)
  int cap_units;        // most units one CTA takes (cap_units * grid >= units_total)
  unsigned int* sched;  // [0] next unit - grid, [1] CTAs done; null: static units
  uint32_t off_blk;     // int unit id per ring stage, then the CTA's unit ids in order
  int chunks;           // chunks per row
  int gunits;           // 64-column units per scale group
  int ngroups;          // scale groups per row
  int x_resident;       // 1: activations staged once; 0: per chunk by TMA
  int xbox_bytes;       // per-chunk mode: bytes between activation boxes
  uint32_t off_x, off_s, off_corr, off_bar, off_red;
  int sbuf_bytes, nsb;  // scale buffer size and count
  int scales_aligned;   // scale table 16-byte aligned (bulk copies allowed)
  uint32_t off_vals;    // fp32 logits of the CTA's rows for the top-K, [token][vals_stride]
  int vals_stride;      // 0: no room in shared memory, the global scratch row is used
  unsigned int* err;    // sticky error word in the workspace (null: none)
};

// Working area of the top-K selection.  It lives in the weight ring, which is
// free once the main loop has consumed every stage.
struct SelWork {
  unsigned int thr[kMaxTok];                   // value-key threshold per token
  unsigned int cnt[kMaxTok];                   // entries kept per token
  unsigned long long cand[kMaxTok][kSelCap];   // the kept keys
};
static_assert(sizeof(SelWork) <= (size_t)kStages * kStageWBytes, "selection area > ring");

__host__ __device__ constexpr uint32_t round_up_u32(uint32_t v, uint32_t a) {
  return (v + a - 1) / a * a;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(kConsumerBarrier), "n"(kConsumers * 32) : "memory");
}

// Top-K keys of entries [0, count) per token, by all warps of the CTA: warp w
// takes token w % m and every S-th stretch of 32 entries (S = warps / m);
// loads go out in batches of 8 so L2 latency is paid once per batch.  Warps
// w < m return their token's merged list in `out` (out_tok = w), others -1.
template <int KT, typename Load>
__device__ __forceinline__ void select_topk(int m, int K, int count, unsigned long long* red,
                                            Load load, unsigned long long (&out)[KT],
                                            int& out_tok) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slices = max(1, kWarpsAll / m);
  unsigned long long list[KT];
#pragma unroll
  for (int i = 0; i < KT; ++i) list[i] = kEmptyKey;
  if (warp < slices * m) {
    const int tok = warp % m, sl = warp / m;
    const int step = slices * 32;
    for (int i0 = sl * 32 + lane; i0 < count; i0 += 8 * step) {
      unsigned long long v[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int i = i0 + b * step;
        v[b] = i < count ? load(tok, i) : kEmptyKey;
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) list_insert<KT>(list, v[b]);
    }
  }
  unsigned long long best[KT];
  warp_merge_topk_redux<KT>(list, K, best);
  if (warp < slices * m && lane < KT) red[warp * KT + lane] = pick(best, lane);
  __syncthreads();
  out_tok = -1;
  if (warp < m) {
    unsigned long long l2[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i)
      l2[i] = lane < slices ? red[(lane * m + warp) * KT + i] : kEmptyKey;
    warp_merge_topk_redux<KT>(l2, K, out);
    out_tok = warp;
  }
}

__device__ __forceinline__ unsigned long long shfl_u64(unsigned long long v, int src) {
  const uint32_t lo = __shfl_sync(0xFFFFFFFFu, (uint32_t)v, src);
  const uint32_t hi = __shfl_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), src);
  return ((unsigned long long)hi << 32) | lo;
}

// Order-preserving 32-bit key of a value (the high half of topk_key): NaN 0.
__device__ __forceinline__ uint32_t value_key(float v) {
  if (v != v) return 0u;
  const uint32_t b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The K-th largest of the 32 lanes' values (K <= 32), on every lane: each
// lane ranks its value against all others (ties by lane), 32 independent
// shuffles, and the lane of rank K-1 broadcasts it.
__device__ __forceinline__ uint32_t warp_kth_rank(uint32_t v, int K) {
  const int lane = threadIdx.x & 31;
  int rank = 0;
#pragma unroll
  for (int j0 = 0; j0 < 32; j0 += 8) {
    uint32_t o[8];   // eight shuffles in flight before any is used
#pragma unroll
    for (int b = 0; b < 8; ++b) o[b] = __shfl_sync(0xFFFFFFFFu, v, j0 + b);
#pragma unroll
    for (int b = 0; b < 8; ++b) rank += (o[b] > v || (o[b] == v && j0 + b < lane)) ? 1 : 0;
  }
  const unsigned int sel = __ballot_sync(0xFFFFFFFFu, rank == K - 1);
  return __shfl_sync(0xFFFFFFFFu, v, __ffs(sel) - 1);
}

// Output of a warp's selection, per lane: the key for slot `slot` of the
// descending top-K list (slot -1: this lane writes nothing).  Every slot
// 0..K-1 is written by exactly one lane; kEmptyKey where there are fewer
// than K entries.
struct LaneSlot {
  unsigned long long key;
  int slot;
};

// Top K of c <= 32 unique keys held one per lane (lanes >= c: kEmptyKey):
// each lane ranks its key by 32 shuffles and keeps slot = rank if rank < K.
__device__ __forceinline__ LaneSlot warp_rank_of_32(unsigned long long key, int c, int K) {
  const int lane = threadIdx.x & 31;
  int rank = 0;
#pragma unroll
  for (int j0 = 0; j0 < 32; j0 += 8) {
    unsigned long long o[8];   // eight shuffles in flight before any is used
#pragma unroll
    for (int b = 0; b < 8; ++b) o[b] = __shfl_sync(0xFFFFFFFFu, key, j0 + b);
#pragma unroll
    for (int b = 0; b < 8; ++b) rank += o[b] > key ? 1 : 0;
  }
  LaneSlot r{kEmptyKey, -1};
  if (lane < c) {
    if (rank < K) r = {key, rank};
  } else if (lane < K) {
    r = {kEmptyKey, lane};   // fewer than K entries: the empty tail slots
  }
  return r;
}

// The same output from a descending list held identically by every lane.
template <int KT>
__device__ __forceinline__ LaneSlot lane_slot_of_list(const unsigned long long (&out)[KT], int K) {
  const int lane = threadIdx.x & 31;
  return lane < K ? LaneSlot{pick(out, lane), lane} : LaneSlot{kEmptyKey, -1};
}

// Threshold selection of the top-K keys of entries [0, count) per token, by
// all threads of the CTA.  vkey(t, i) reads entry i's value key (a 32-bit
// key that orders values; 0 for NaN), fkey(t, i) its full 64-bit key (value
// key high, index low).  W.thr[t] must hold a lower bound of token t's K-th
// largest value key (0 if none) and W.cnt[t] zero, visible to all threads.
// Each token's entries are spread over up to kSelWarps warps; every warp
// raises the bound to the K-th largest of its lanes' maxima (K lanes hold
// disjoint entries at or above it, so it does not exceed the token's K-th
// largest value).  The entries whose value key reaches the bound are kept
// (all of the top K are among them) and warp w < m selects token w's top K
// from those (out_tok = w, slots in `res`; others -1).  Returns false, with
// nothing selected, if a token kept more than kSelCap entries (many equal
// values); the caller then selects exhaustively.
constexpr int kSelWarps = 4;
template <int KT, typename VKey, typename FKey>
__device__ __forceinline__ bool cta_topk(int m, int K, int count, VKey vkey, FKey fkey,
                                         SelWork& W, LaneSlot& res, int& out_tok) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slices = max(1, min(kSelWarps, kWarpsAll / m));
  const bool worker = warp < slices * m;
  const int tok = warp % m, sl = warp / m;
  const int step = slices * 32;
  if (worker) {
    uint32_t mx = 0u;
    for (int i0 = sl * 32 + lane; i0 < count; i0 += 8 * step) {
      uint32_t v[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int i = i0 + b * step;
        v[b] = vkey(tok, min(i, count - 1));
        if (i >= count) v[b] = 0u;
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) mx = max(mx, v[b]);
    }
    const uint32_t kth = warp_kth_rank(mx, K);
    if (lane == 0 && kth > 0u) atomicMax(&W.thr[tok], kth);
  }
  __syncthreads();
  if (worker) {
    const uint32_t th = W.thr[tok];
    // warp-uniform trip count (the ballots below need every lane)
    for (int w0 = sl * 32; w0 < count; w0 += 8 * step) {
      const int i0 = w0 + lane;
      uint32_t v[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int i = i0 + b * step;
        v[b] = vkey(tok, min(i, count - 1));
      }
      // one shared atomic per warp for the batch's passing entries
      unsigned int mask[8];
      int total = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        mask[b] = __ballot_sync(0xFFFFFFFFu, i0 + b * step < count && v[b] >= th);
        total += __popc(mask[b]);
      }
      if (total > 0) {
        unsigned int at = 0u;
        if (lane == 0) at = atomicAdd(&W.cnt[tok], (unsigned int)total);
        at = __shfl_sync(0xFFFFFFFFu, at, 0);
        const unsigned int lt = (1u << lane) - 1u;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (mask[b] >> lane & 1u) {
            const unsigned int pos = at + __popc(mask[b] & lt);
            if (pos < (unsigned int)kSelCap) W.cand[tok][pos] = fkey(tok, i0 + b * step);
          }
          at += __popc(mask[b]);
        }
      }
    }
  }
  __syncthreads();
  bool overflow = false;
  for (int t = 0; t < m; ++t) overflow |= W.cnt[t] > (unsigned int)kSelCap;
  out_tok = -1;
  if (overflow) return false;
  if (warp < m) {
    const int c = (int)W.cnt[warp];
    if (c <= 32) {
      res = warp_rank_of_32(lane < c ? W.cand[warp][lane] : kEmptyKey, c, K);
    } else {
      unsigned long long list[KT], out[KT];
#pragma unroll
      for (int i = 0; i < KT; ++i) list[i] = kEmptyKey;
      for (int i = lane; i < c; i += 32) list_insert<KT>(list, W.cand[warp][i]);
      warp_merge_topk_redux<KT>(list, K, out);
      res = lane_slot_of_list<KT>(out, K);
    }
    out_tok = warp;
  }
  return true;
}

// Ticket of the last-CTA merge: an atomic add whose release makes this CTA's
// candidate writes (ordered before it by the preceding block barrier)
// visible before the ticket, and whose acquire, for the last CTA, makes the
// other CTAs' candidates visible after it.
__device__ __forceinline__ unsigned int ticket_add(unsigned int* t) {
  unsigned int old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
  return old;
}

// This CTA's candidates, the ticket, and (last CTA only) the final merge.
// The CTA's rows are its nunits work units in the order it took them (unit
// ids in blk_list, 2^rlog rows each; the grid's last unit, cut at n, is
// always a CTA's last).  svals: their fp32 logits in shared memory
// ([token][vals_stride], entry li * R + r), or null for the global scratch
// row.
template <int KT, typename XT, bool kSmemVals>
__device__ __noinline__ void topk_tail(const DecodeParams& p, SelWork& W,
                                          unsigned long long* red, unsigned int* flags,
                                          int nunits, const int* blk_list, bool cta_bad,
                                          const float* svals) {
  const LogitsArgs& a = p.a;
  unsigned int* err = p.err;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int m = a.m, n = a.n, K = a.topk;
  unsigned int* tau = a.counter + kTauWord;   // per-token bound on the K-th value key
  if (!cta_bad) {
    const int rlog = p.unit_rows_log2, R = 1 << rlog;
    const int count = nunits > 0 ? (nunits - 1) * R + min(R, n - blk_list[nunits - 1] * R) : 0;
    const int vs = p.vals_stride;
    auto rowof = [&](int i) { return blk_list[i >> rlog] * R + (i & (R - 1)); };
    auto value = [&](int tk, int i) -> float {
      if constexpr (kSmemVals) return svals[tk * vs + i];
      else return __ldcg(a.scratch + (size_t)tk * n + rowof(i));
    };
    auto vkey = [&](int tk, int i) { return value_key(value(tk, i)); };
    auto key = [&](int tk, int i) { return topk_key(value(tk, i), (uint32_t)rowof(i)); };
    if (threadIdx.x < m) {
      W.thr[threadIdx.x] = 0u;
      W.cnt[threadIdx.x] = 0u;
    }
    __syncthreads();
    LaneSlot res{kEmptyKey, -1};
    int tok;
    if (!cta_topk<KT>(m, K, count, vkey, key, W, res, tok)) {
      unsigned long long best[KT];
      select_topk<KT>(m, K, count, red, key, best, tok);
      res = lane_slot_of_list<KT>(best, K);
    }
    if (tok >= 0) {
      // every CTA's K-th value bounds the final K-th value from below: raise
      // the token's bound, then append this CTA's entries that reach it as
      // it stands after the raise (the reply of the atomic) -- an entry of
      // the final top K reaches the final bound, hence this one, and the
      // list stays short because later CTAs see an ever higher bound
      const unsigned int kth_lane = __ballot_sync(0xFFFFFFFFu, res.slot == K - 1);
      unsigned long long kth_key = shfl_u64(res.key, kth_lane ? __ffs(kth_lane) - 1 : 0);
      if (kth_lane == 0u) kth_key = kEmptyKey;
      uint32_t bound = 0u;
      if (lane == 0 && kth_key != kEmptyKey)
        bound = max(atomicMax(tau + tok, (uint32_t)(kth_key >> 32)), (uint32_t)(kth_key >> 32));
      bound = __shfl_sync(0xFFFFFFFFu, bound, 0);
      const bool pass = res.slot >= 0 && res.key != kEmptyKey && (uint32_t)(res.key >> 32) >= bound;
      const unsigned int pm = __ballot_sync(0xFFFFFFFFu, pass);
      unsigned int at = 0u;
      if (lane == 0 && pm != 0u) at = atomicAdd(a.counter + kNCandWord + tok, (unsigned int)__popc(pm));
      at = __shfl_sync(0xFFFFFFFFu, at, 0);
      // at most K per CTA: the list never outgrows its WQL_MAX_CTAS * K slots
      if (pass)
        a.cand[(size_t)tok * WQL_MAX_CTAS * K + at + __popc(pm & ((1u << lane) - 1u))] = res.key;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) flags[1] = (ticket_add(a.counter) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (flags[1] == 0u) return;
  // The error word (set by any CTA whose bounded wait timed out, before its
  // ticket): with an error the results are replaced by "no entries".  A CTA
  // that timed out itself reports no entries directly.
  const unsigned int errv = __ldcg(err);
  if (!cta_bad) {
    // warp t ranks token t's appended candidates (m <= kMaxTok < warps)
    if (warp < m) {
      const unsigned long long* list = a.cand + (size_t)warp * WQL_MAX_CTAS * K;
      // the first 32 slots are read together with the count (slots beyond
      // it hold older entries and are masked): one round trip, not two
      const unsigned long long first = __ldcg(list + lane);
      const int c = (int)__ldcg(a.counter + kNCandWord + warp);
      LaneSlot res{kEmptyKey, -1};
      if (c <= 32) {
        res = warp_rank_of_32(lane < c ? first : kEmptyKey, c, K);
      } else {
        unsigned long long best[KT], out[KT];
#pragma unroll
        for (int i = 0; i < KT; ++i) best[i] = kEmptyKey;
        for (int i0 = lane; i0 < c; i0 += 8 * 32) {
          unsigned long long v[8];   // eight loads in flight per lane
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            const int i = i0 + 32 * b;
            v[b] = i < c ? __ldcg(list + i) : kEmptyKey;
          }
#pragma unroll
          for (int b = 0; b < 8; ++b) list_insert<KT>(best, v[b]);
        }
        warp_merge_topk_redux<KT>(best, K, out);
        res = lane_slot_of_list<KT>(out, K);
      }
      if (res.slot >= 0) {
        const bool ok = errv == 0u && res.key != kEmptyKey;
        const size_t o = (size_t)warp * K + res.slot;
        a.topk_idx[o] = ok ? key_index(res.key) : -1;
        a.topk_val[o] = ok ? key_value(res.key) : __int_as_float(0x7FC00000);
      }
    }
    __syncthreads();
  } else {
    // this CTA timed out: report no entries
    for (int i = threadIdx.x; i < m * K; i += blockDim.x) {
      a.topk_idx[i] = -1;
      a.topk_val[i] = __int_as_float(0x7FC00000);
    }
  }
  if (threadIdx.x == 0) *a.counter = 0u;       // ready for the next call
  if (threadIdx.x < m) {
    tau[threadIdx.x] = 0u;
    a.counter[kNCandWord + threadIdx.x] = 0u;
  }
}

// The offset sum of one 16-byte piece of 8 activations: off * sum(x); with
// kScaled, the halves at elements 2, 3, 6, 7 hold x/16 and weigh 1152, the
// others weigh 1032 (Int4F16Scaled).
template <typename XT, bool kScaled>
__device__ __forceinline__ float corr_piece(const uint4& v, float off) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float a = 0.f, b = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float lo = scale_bits_to_f32<XT>((uint16_t)(w[q] & 0xFFFFu));
    const float hi = scale_bits_to_f32<XT>((uint16_t)(w[q] >> 16));
    if (kScaled && (q & 1)) b += lo + hi;
    else a += lo + hi;
  }
  return kScaled ? 1032.0f * a + 1152.0f * b : off * a;
}

// tw:  packed weight, 16-row x 128-byte boxes (partial blocks)
// twb: packed weight, 256-row x 128-byte boxes (one copy per full block chunk;
//      TMA throughput is per box, so large boxes are what reach HBM speed)
// tx:  activations, 64-column boxes of all m rows (per-chunk mode only)
// Code conversion per variant: fp16 int4 with resident activations uses the
// pre-scaled-activation form (one shift per word); everything else the
// shifted OffsetCodes form.
template <int BITS, typename XT, bool XRES>
struct CodesFor {
  using type = OffsetCodes<BITS, XT>;
  static constexpr bool kScaledX = false;
  static constexpr bool kCorr = OffsetCodes<BITS, XT>::kOffset != 0.0f;
};
template <>
struct CodesFor<4, __half, true> {
  using type = Int4F16Scaled;
  static constexpr bool kScaledX = true;
  static constexpr bool kCorr = true;
};

template <int BITS, typename XT, typename ST, int NT, bool XRES>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap twb,
                  const __grid_constant__ CUtensorMap tx, const __grid_constant__ DecodeParams p) {
  using CF = CodesFor<BITS, XT, XRES>;
  using Codes = typename CF::type;
  constexpr int kUnits = BITS == 4 ? 4 : 2;        // 64-column units per chunk
  constexpr int KC = kUnits * 64;                  // codes per chunk
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;    // 1024-aligned for 128B swizzle
  uint8_t* sm = smem_raw + (base - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + p.off_bar);
  uint64_t* empty = full + kStages;
  unsigned int* flags = reinterpret_cast<unsigned int*>(empty + kStages);  // [0] bad, [1] last
  unsigned long long* red = reinterpret_cast<unsigned long long*>(sm + p.off_red);
  float* corr = reinterpret_cast<float*>(sm + p.off_corr);   // [kMaxTok][ngroups]
  float* svals = reinterpret_cast<float*>(sm + p.off_vals);
  int* blk_stage = reinterpret_cast<int*>(sm + p.off_blk);   // [kStages]
  int* blk_list = blk_stage + kStages;                        // [cap_units]
  const int U = p.unit_tiles;

  const LogitsArgs& a = p.a;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int m = a.m, n = a.n, k = a.k;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    flags[0] = 0u;
    flags[1] = 0u;
    fence_barrier_init();
  }
  __syncthreads();

  bool bad = false;

  if (warp == kConsumers) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      prefetch_tmap(&tw);
      prefetch_tmap(&twb);
      if (!XRES) prefetch_tmap(&tx);
      const uint8_t* scales = reinterpret_cast<const uint8_t*>(a.scales);
      const int xstage = kUnits * p.xbox_bytes;
      int stage = 0;
      uint32_t ephase = 0;
      int j = 0, issued = 0;
      // Work units: the CTA's first is its own index; later ones come from
      // the shared counter (CTAs that stream faster take more) or, without
      // one, in a fixed stride.  The next id is taken when a unit starts, so
      // the atomic's latency hides behind that unit's copies; an id is only
      // taken when the CTA has room to process it.
      int b = (int)blockIdx.x;
      for (int lb = 0; !bad && b < p.units_total && lb < p.cap_units; ++lb) {
        int nextb = p.units_total;
        if (lb + 1 < p.cap_units)
          nextb = p.sched ? (int)atomicAdd(p.sched, 1u) + (int)gridDim.x : b + (int)gridDim.x;
        blk_list[lb] = b;
        const int tb = b * U;
        const int ntb = min(U, p.tiles_total - tb);
        const bool sc_bulk = p.scales_aligned && (tb + ntb) * 16 <= n;
        const uint32_t sbytes = (uint32_t)(ntb * 16 * p.ngroups * 2);
        for (int c = 0; c < p.chunks; ++c, ++j) {
          // stage reuse: wait until all consumers released its previous fill
          if (j >= kStages && !bad) bad = !mbar_wait(&empty[stage], ephase ^ 1u);
          if (!bad) {
            blk_stage[stage] = b;
            uint32_t bytes = (uint32_t)(ntb * kTileBytes);
            if (!XRES) bytes += (uint32_t)(kUnits * m * 128);
            if (c == 0 && sc_bulk) bytes += sbytes;
            mbar_arrive_expect_tx(&full[stage], bytes);
            uint8_t* wdst = sm + stage * kStageWBytes;
            if (ntb == kBlockTiles) {
              tma_load_2d(wdst, &twb, c * (kChunkRowBytes / 4), tb * 16, &full[stage]);
            } else {
              for (int t = 0; t < ntb; ++t)
                tma_load_2d(wdst + t * kTileBytes, &tw, c * (kChunkRowBytes / 4), (tb + t) * 16,
                            &full[stage]);
            }
            if (!XRES) {
              uint8_t* xdst = sm + p.off_x + stage * xstage;
              for (int u = 0; u < kUnits; ++u)
                tma_load_2d(xdst + u * p.xbox_bytes, &tx, c * KC + u * 64, 0, &full[stage]);
            }
            if (c == 0 && sc_bulk)
              bulk_load(sm + p.off_s + (lb % p.nsb) * p.sbuf_bytes,
                        scales + (size_t)tb * 16 * p.ngroups * 2, sbytes, &full[stage]);
            issued = j + 1;
          }
          if (++stage == kStages) { stage = 0; ephase ^= 1u; }
        }
        b = nextb;
      }
      // Every copy this CTA issued must have landed before it can finish: the
      // latest fill of slot s completes phase (fills_of_s - 1) & 1.  On the
      // normal path the consumers already waited for all of them.
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int fills = (issued - 1 - s) / kStages + 1;
        if (!mbar_wait(&full[s], (uint32_t)((fills - 1) & 1))) bad = true;
      }
      // This producer takes no more units (its last take has returned): the
      // last producer of the grid to get here resets the counter for the
      // next launch.
      if (p.sched && atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
        p.sched[0] = 0u;
        p.sched[1] = 0u;
      }
      // End of work: one more stage, unit id -1, completed by a plain arrive
      // (after the copies above, so no copy phase is pending on its slot).
      if (!bad) {
        if (j >= kStages) bad = !mbar_wait(&empty[stage], ephase ^ 1u);
        if (!bad) {
          blk_stage[stage] = -1;
          mbar_arrive(&full[stage]);
        }
      }
    }
  } else {
    // ------------------------------ consumers -----------------------------
    const int g = lane >> 2, t = lane & 3;
    const XT* xg = reinterpret_cast<const XT*>(a.x);
    // (1) resident activations: [unit][token][64] halves, 16-byte pieces
    //     XOR-swizzled by token so fragment loads avoid bank conflicts.
    if (XRES) {
      const int pieces_per_row = k / 8;
      for (int i = threadIdx.x; i < m * pieces_per_row; i += kConsumers * 32) {
        const int tok = i / pieces_per_row, pc = i - tok * pieces_per_row;
        uint4 v = *reinterpret_cast<const uint4*>(xg + (size_t)tok * k + pc * 8);
        if constexpr (CF::kScaledX) {   // elements 2, 3, 6, 7 of each 8 -> x / 16 (exact)
          const uint32_t sixteenth = 0x2C002C00u;
          v.y = hmul2_u32(v.y, sixteenth);
          v.w = hmul2_u32(v.w, sixteenth);
        }
        const int U = pc >> 3, piece = pc & 7;
        *reinterpret_cast<uint4*>(sm + p.off_x + (U * m + tok) * 128 +
                                  ((piece ^ (tok & 7)) * 16)) = v;
      }
    }
    // (2) per (token, group): the offset the MMA sums picked up, summed from
    //     16-byte pieces (the resident copy when there is one, as the MMA
    //     sees it); absent tokens get 0
    if constexpr (CF::kCorr) {
      if (XRES) consumer_sync();
      const int G = p.gunits * 64;
      for (int i = m * p.ngroups + threadIdx.x; i < kMaxTok * p.ngroups; i += kConsumers * 32)
        corr[i] = 0.f;
      for (int pr = warp; pr < m * p.ngroups; pr += kConsumers) {
        const int tok = pr / p.ngroups, gidx = pr - tok * p.ngroups;
        float s = 0.f;
        for (int e = lane * 8; e < G; e += 256) {
          const int kk = gidx * G + e;
          uint4 v;
          if (XRES) {
            const int U = kk >> 6, piece = (kk >> 3) & 7;
            v = *reinterpret_cast<const uint4*>(sm + p.off_x + (U * m + tok) * 128 +
                                                ((piece ^ (tok & 7)) * 16));
          } else {
            v = *reinterpret_cast<const uint4*>(xg + (size_t)tok * k + kk);
          }
          s += corr_piece<XT, CF::kScaledX>(v, Codes::kOffset);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
        if (lane == 0) corr[pr] = s;
      }
    }
    consumer_sync();

    // per-lane constant shared-memory offsets
    const int r8 = lane & 7, mi = lane >> 3;
    uint32_t woff[4];   // ldmatrix address inside a 16-row tile, per unit (int8: per half unit)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int seg = (BITS == 4 ? 2 * i : 2 * i) + (mi >> 1);
      woff[i] = (uint32_t)((r8 + 8 * (mi & 1)) * kChunkRowBytes + ((seg ^ r8) * 16));
    }
    uint32_t xoff[NT][4];   // activation piece offsets inside one 64-column unit box
    bool tok_ok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tok = nt * 8 + g;
      tok_ok[nt] = tok < m;
      const int tk = tok < m ? tok : 0;
#pragma unroll
      for (int sg = 0; sg < 4; ++sg) {
        const int piece = BITS == 4 ? (4 * sg + t) : (2 * sg + (t >> 1));
        xoff[nt][sg] = (uint32_t)(tk * 128 + (((piece & 7) ^ (tk & 7)) * 16) +
                                  (BITS == 4 ? 0 : (t & 1) * 8));
      }
    }
    const uint32_t xunit_stride = XRES ? (uint32_t)(m * 128) : (uint32_t)p.xbox_bytes;

    int stage = 0;
    uint32_t fphase = 0;
    int lb = 0;
    for (;; ++lb) {
      // the stage of a unit's first chunk names the unit (-1: no more work)
      if (!bad) bad = !mbar_wait(&full[stage], fphase);
      if (bad) break;
      const int ub = blk_stage[stage];
      if (ub < 0) break;
      const int tb = ub * U;
      const int ntb = min(U, p.tiles_total - tb);
      const bool active = warp < ntb;
      const bool sc_bulk = p.scales_aligned && (tb + ntb) * 16 <= n;
      const int row_a = (tb + warp) * 16 + g, row_b = row_a + 8;
      const uint16_t* sbuf = reinterpret_cast<const uint16_t*>(sm + p.off_s +
                                                               (lb % p.nsb) * p.sbuf_bytes);
      float acc[NT][4], part[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[nt][c] = part[nt][c] = 0.f;
      uint32_t xb[NT][8];     // B fragments; lanes of absent tokens keep zeros
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 8; ++i) xb[nt][i] = 0u;
      const uint16_t* srow_a = sc_bulk ? sbuf + (warp * 16 + g) * p.ngroups
                                       : a.scales + (size_t)min(row_a, n - 1) * p.ngroups;
      const uint16_t* srow_b = sc_bulk ? sbuf + (warp * 16 + g + 8) * p.ngroups
                                       : a.scales + (size_t)min(row_b, n - 1) * p.ngroups;
      const float* corr_t0 = corr + (2 * t) * p.ngroups;      // tokens 2t, 2t+1 (+8 nt)
      int u_in_group = 0, gi = 0;

      for (int c = 0; c < p.chunks; ++c) {
        if (c > 0 && !bad) bad = !mbar_wait(&full[stage], fphase);
        if (active && !bad) {
          const uint32_t wst = base + stage * kStageWBytes + warp * kTileBytes;
          const uint32_t xst = XRES ? base + p.off_x + (uint32_t)(c * kUnits) * xunit_stride
                                    : base + p.off_x + (uint32_t)(stage * kUnits) * xunit_stride;
          const int nu = min(kUnits, (k - c * KC) / 64);   // last chunk may be partial
#pragma unroll
          for (int u = 0; u < kUnits; ++u) {
            if (u < nu) {
              // ---- activations (B fragments) for this 64-column unit ----
              const uint32_t xu = xst + u * xunit_stride;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (tok_ok[nt]) {
                  if constexpr (BITS == 4) {
#pragma unroll
                    for (int sg = 0; sg < 2; ++sg) {
                      const uint4 v = lds128(xu + xoff[nt][sg]);
                      xb[nt][4 * sg] = v.x; xb[nt][4 * sg + 1] = v.y;
                      xb[nt][4 * sg + 2] = v.z; xb[nt][4 * sg + 3] = v.w;
                    }
                  } else {
#pragma unroll
                    for (int sg = 0; sg < 4; ++sg) {
                      const uint2 v = lds64(xu + xoff[nt][sg]);
                      xb[nt][2 * sg] = v.x; xb[nt][2 * sg + 1] = v.y;
                    }
                  }
                }
              }
              // ---- weights: ldmatrix + offset codes + MMA ----
              if constexpr (BITS == 4) {
                uint32_t wv[4];
                ldmatrix_x4(wv, wst + woff[u]);
                // wv: (row g, seg 2u), (row g+8, seg 2u), (row g, seg 2u+1), (row g+8, seg 2u+1)
#pragma unroll
                for (int sg = 0; sg < 2; ++sg) {
                  uint32_t qa[4], qb[4];
                  Codes::run(wv[2 * sg], qa);
                  Codes::run(wv[2 * sg + 1], qb);
                  const uint32_t af0[4] = {qa[0], qb[0], qa[1], qb[1]};
                  const uint32_t af1[4] = {qa[2], qb[2], qa[3], qb[3]};
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt) {
                    Mma16816<XT>::run(part[nt], af0, xb[nt][4 * sg], xb[nt][4 * sg + 1], part[nt]);
                    Mma16816<XT>::run(part[nt], af1, xb[nt][4 * sg + 2], xb[nt][4 * sg + 3],
                                      part[nt]);
                  }
                }
              } else {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  uint32_t wv[4];
                  ldmatrix_x4(wv, wst + woff[2 * u + hh]);
#pragma unroll
                  for (int sg = 0; sg < 2; ++sg) {
                    uint32_t qa[2], qb[2];
                    Codes::run(wv[2 * sg], qa);
                    Codes::run(wv[2 * sg + 1], qb);
                    const uint32_t af[4] = {qa[0], qb[0], qa[1], qb[1]};
                    const int s4 = 2 * hh + sg;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                      Mma16816<XT>::run(part[nt], af, xb[nt][2 * s4], xb[nt][2 * s4 + 1],
                                        part[nt]);
                  }
                }
              }
              // ---- group end: remove the offset, apply the exact scale ----
              if (++u_in_group == p.gunits) {
                u_in_group = 0;
                const float fa = scale_bits_to_f32<ST>(srow_a[gi]);
                const float fb = scale_bits_to_f32<ST>(srow_b[gi]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  float c0 = 0.f, c1 = 0.f;
                  if constexpr (CF::kCorr) {
                    c0 = corr_t0[(nt * 8) * p.ngroups + gi];
                    c1 = corr_t0[(nt * 8 + 1) * p.ngroups + gi];
                  }
                  acc[nt][0] = fmaf(fa, part[nt][0] - c0, acc[nt][0]);
                  acc[nt][1] = fmaf(fa, part[nt][1] - c1, acc[nt][1]);
                  acc[nt][2] = fmaf(fb, part[nt][2] - c0, acc[nt][2]);
                  acc[nt][3] = fmaf(fb, part[nt][3] - c1, acc[nt][3]);
#pragma unroll
                  for (int c2 = 0; c2 < 4; ++c2) part[nt][c2] = 0.f;
                }
                ++gi;
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == kStages) { stage = 0; fphase ^= 1u; }
      }

      if (active && !bad) {
        // ---- epilogue: logits (+bias), fp32 copy for the top-K pass ----
        const int rows[2] = {row_a, row_b};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int row = rows[c >> 1];
            const int tok = nt * 8 + 2 * t + (c & 1);
            if (row < n && tok < m) {
              float v = acc[nt][c];
              if (a.bias) v += to_f32(reinterpret_cast<const XT*>(a.bias)[row]);
              reinterpret_cast<XT*>(a.logits)[(size_t)tok * n + row] = from_f32<XT>(v);
              if (a.topk > 0) {
                if (p.vals_stride > 0)
                  svals[tok * p.vals_stride + lb * U * 16 + (row - tb * 16)] = v;
                else
                  a.scratch[(size_t)tok * n + row] = v;
              }
            }
          }
      }
      if (bad) break;
    }
    if (threadIdx.x == 0) flags[2] = (unsigned int)lb;   // units this CTA processed
  }

  if (bad) atomicOr(&flags[0], 1u);
  __syncthreads();
  const bool cta_bad = flags[0] != 0u;
  if (cta_bad && threadIdx.x == 0 && p.err) atomicOr(p.err, 1u);
  if (a.topk <= 0) return;

  // ---------------- top-K: per-CTA selection, last-CTA merge ----------------
  SelWork& W = *reinterpret_cast<SelWork*>(sm);
  const float* sv = p.vals_stride > 0 ? svals : nullptr;
  const int nunits = (int)flags[2];
  if (sv) {
    if (a.topk <= 8)
      topk_tail<8, XT, true>(p, W, red, flags, nunits, blk_list, cta_bad, sv);
    else
      topk_tail<16, XT, true>(p, W, red, flags, nunits, blk_list, cta_bad, sv);
  } else {
    if (a.topk <= 8)
      topk_tail<8, XT, false>(p, W, red, flags, nunits, blk_list, cta_bad, sv);
    else
      topk_tail<16, XT, false>(p, W, red, flags, nunits, blk_list, cta_bad, sv);
  }
}

template <int BITS, typename XT, typename ST, int NT, bool XRES>
cudaError_t launch_t(const CUtensorMap& tw, const CUtensorMap& twb, const CUtensorMap& tx,
                     const DecodeParams& p, size_t smem, int ctas, cudaStream_t s) {
  auto kern = decode_kernel<BITS, XT, ST, NT, XRES>;
  static size_t configured = 0;  // per instantiation: raise the smem limit once
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  kern<<<ctas, kThreads, smem, s>>>(tw, twb, tx, p);
  note_launch();
  return cudaGetLastError();
}

// All variants for one activation dtype.
template <typename XT>
cudaError_t dispatch_x(const CUtensorMap& tw, const CUtensorMap& twb, const CUtensorMap& tx,
                       const DecodeParams& p, size_t smem, int ctas, cudaStream_t s) {
  const bool nt1 = p.a.m <= 8;
  const bool sf16 = p.a.scale_dtype == WQL_F16;
#define WQL_DECODE_CASE(B, ST)                                                                \
  if (p.x_resident) {                                                                        \
    return nt1 ? launch_t<B, XT, ST, 1, true>(tw, twb, tx, p, smem, ctas, s)                 \
               : launch_t<B, XT, ST, 2, true>(tw, twb, tx, p, smem, ctas, s);                \
  }                                                                                          \
  return nt1 ? launch_t<B, XT, ST, 1, false>(tw, twb, tx, p, smem, ctas, s)                  \
             : launch_t<B, XT, ST, 2, false>(tw, twb, tx, p, smem, ctas, s);
  if (p.a.bits == 4) {
    if (sf16) { WQL_DECODE_CASE(4, __half) }
    WQL_DECODE_CASE(4, __nv_bfloat16)
  }
  if (sf16) { WQL_DECODE_CASE(8, __half) }
  WQL_DECODE_CASE(8, __nv_bfloat16)
#undef WQL_DECODE_CASE
}

}  // namespace decode_detail
}  // namespace wql
