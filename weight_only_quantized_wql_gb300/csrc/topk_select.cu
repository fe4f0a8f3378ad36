// topk_select.cu -- top-K candidates of each token row from the rounded
// logits a logits kernel has written, with the candidates' values recomputed
// in fp32 from the packed weight ("Fused WNA16 GEMM for tied quantized
// lm_head logits", reviewer comment item 2: take the top-K of the quantised
// logits, to be rescored exactly).
//
// Why the rounded logits suffice to find the candidates: rounding to
// fp16/bf16 is monotone, so if the K-th largest rounded logit of a row is h,
// every row in the fp32 top-K has a rounded logit >= h (a row below h would
// have K rows strictly above it).  The set {rounded logit >= h} -- K rows
// plus any ties at h -- therefore contains the fp32 top-K; only those rows
// are recomputed and ranked (value descending, index ascending).
//
// Keys are the order-preserving 16-bit images of the rounded logits.  The
// row is split into ranges (the grid fills one wave); one CTA per (token,
// range):
//  * threshold: the K-th largest of 16 half-warp maxima over the range's
//    first step -- K distinct positions lie at or above it, so it bounds the
//    range's K-th largest key from below; during the scan it rises to the
//    K-th largest key that any one warp has queued (again K distinct
//    positions at or above it);
//  * every position with key >= threshold is queued (a thread first tests
//    its 32 logits of a step at once: per-half signed maxima), the range's K-th
//    largest queued key h_r found, and the positions with key >= h_r -- a
//    superset of the range's top K, and of its share of the row's top K --
//    recomputed in fp32 (a warp per position); the range's best K go to the
//    workspace;
//  * the last CTA of a token to finish (a per-token ticket in the
//    workspace, reset by that CTA) merges the ranges' K best.
// A range with too many positions above its threshold (many equal logits)
// is done exactly in chunks instead: each chunk's positions above the
// running threshold are recomputed and merged, the running K-th value
// raising the threshold.
#include <cuda_bf16.h>
#include <cuda_fp16.h>


#include "sm100.cuh"
#include "wql_common.cuh"

namespace wql {
namespace {

constexpr int kPer = 8;                          // logits per 16-byte load
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kLoads = 4;                        // 16-byte loads in flight per thread
constexpr int kStep = kThreads * kPer * kLoads;  // 8192 positions per scan step
constexpr int kCap = 1024;                       // queued / gathered positions
constexpr int kChunk = kThreads * 4;             // fallback chunk: 1024 positions (<= kCap)
constexpr int kMinRange = kStep;                 // shortest range worth its own CTA

// Order-preserving 16-bit key of an fp16 / bf16 pattern (sign bit 15 in both).
__device__ __forceinline__ unsigned int key16(unsigned int h) {
  return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}

// The fp16 / bf16 value rounded from an fp32 value, as a key.
template <typename XT>
__device__ __forceinline__ unsigned int key_of_f32(float v) {
  const XT r = from_f32<XT>(v);
  return key16((unsigned int)*reinterpret_cast<const uint16_t*>(&r));
}

// Eight raw rounded logits from position i as a uint4 (scalar loads when
// the row is not 16-byte aligned or at its end; positions >= n read as 0).
__device__ __forceinline__ uint4 load_raw(const uint16_t* row, int n, int i, bool vec) {
  if (vec && i + kPer <= n) return __ldcg(reinterpret_cast<const uint4*>(row + i));
  unsigned int h[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) h[e] = i + e < n ? (unsigned int)__ldcg(row + i + e) : 0u;
  return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                    h[6] | (h[7] << 16));
}

__device__ __forceinline__ unsigned int raw_half(const uint4& v, int e) {
  const unsigned int w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
  return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
}


// Whether any of the thread's kLoads x 8 rounded logits in cur reaches a
// non-negative threshold key (t = its low 15 bits).  Non-negative fp16 and
// bf16 patterns order like signed 16-bit integers and negative ones read as
// negative integers, so the per-half signed maximum clamped at 0 (three
// inputs per instruction) holds the largest non-negative pattern of each half
// lane; a NaN with the sign bit clear counts as above +inf, as its key does.
// Exact for every non-negative threshold.
__device__ __forceinline__ bool any_reaches_pos(const uint4 (&cur)[kLoads], uint32_t t) {
  static_assert(kLoads == 4, "the maximum tree below takes 16 words");
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&cur[0]);
  const uint32_t m0 = __vimax3_s16x2_relu(w[0], w[1], w[2]);
  const uint32_t m1 = __vimax3_s16x2_relu(w[3], w[4], w[5]);
  const uint32_t m2 = __vimax3_s16x2_relu(w[6], w[7], w[8]);
  const uint32_t m3 = __vimax3_s16x2_relu(w[9], w[10], w[11]);
  const uint32_t m4 = __vimax3_s16x2_relu(w[12], w[13], w[14]);
  const uint32_t m5 = __vimax3_s16x2_relu(m0, m1, w[15]);
  const uint32_t m = __vimax3_s16x2_relu(m2, m3, __vimax_s16x2_relu(m4, m5));
  return max(m & 0xFFFFu, m >> 16) >= t;
}

// Bit 15 (low half) and bit 31 (high half) set where a rounded logit of the
// word w has a key >= a non-negative threshold key (t2 = its low 15 bits in
// both halves): the half is non-negative and (h | 0x8000) - t keeps bit 15.
// The subtraction never borrows across halves since h | 0x8000 >= t.
__device__ __forceinline__ uint32_t reach_bits_pos(uint32_t w, uint32_t t2) {
  return (((w | 0x80008000u) - t2) & ~w) & 0x80008000u;
}

struct Hist {
  unsigned int h[256];
  unsigned int bin;        // search result: the bin holding the need-th key
  unsigned int need;       // its rank inside that bin (1-based)
};

// Warp 0: the bin holding the need-th largest key counted in H.h (from bin
// 255 down).
__device__ __forceinline__ void find_bin(Hist& H, unsigned int need) {
  const int lane = threadIdx.x & 31;
  unsigned int c[8], tot = 0;        // lane l owns bins 255 - 8l .. 248 - 8l
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = H.h[255 - 8 * lane - i];
    tot += c[i];
  }
  unsigned int incl = tot;           // inclusive prefix over lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  const unsigned int before = incl - tot;
  if (before < need && incl >= need) {
    unsigned int cum = before;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (cum + c[i] >= need && cum < need) {
        H.bin = 255u - 8u * lane - i;
        H.need = need - cum;
      }
      cum += c[i];
    }
  }
}

// The need-th largest 16-bit key among cnt keys key_at(0..cnt); every thread
// returns it.  Requires cnt >= need >= 1.  Two byte-wise histograms.
template <int NT, typename KeyAt>
__device__ unsigned int kth_key(Hist& H, int cnt, unsigned int need, KeyAt key_at) {
  for (int i = threadIdx.x; i < 256; i += NT) H.h[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < cnt; i += NT) atomicAdd(&H.h[key_at(i) >> 8], 1u);
  __syncthreads();
  if (threadIdx.x < 32) find_bin(H, need);
  __syncthreads();
  const unsigned int hi = H.bin, need2 = H.need;
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += NT) H.h[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < cnt; i += NT) {
    const unsigned int k = key_at(i);
    if ((k >> 8) == hi) atomicAdd(&H.h[k & 0xFFu], 1u);
  }
  __syncthreads();
  if (threadIdx.x < 32) find_bin(H, need2);
  __syncthreads();
  const unsigned int res = (hi << 8) | H.bin;
  __syncthreads();
  return res;
}

// One warp: the need-th largest of cnt <= 32 * kWarpKeys keys key_at(i),
// bit by bit from the top: a prefix stays if at least `need` keys are >= it.
constexpr int kWarpKeys = 16;
template <typename KeyAt>
__device__ __forceinline__ unsigned int warp_kth_key(int cnt, unsigned int need, KeyAt key_at) {
  const int lane = threadIdx.x & 31;
  unsigned int k[kWarpKeys];
#pragma unroll
  for (int j = 0; j < kWarpKeys; ++j) {
    const int i = lane + 32 * j;
    k[j] = i < cnt ? key_at(i) : 0u;
  }
  unsigned int res = 0u;
#pragma unroll 1
  for (int bit = 15; bit >= 0; --bit) {
    const unsigned int cand = res | (1u << bit);
    unsigned int c = 0;
#pragma unroll
    for (int j = 0; j < kWarpKeys; ++j) c += k[j] >= cand ? 1u : 0u;
    if (__reduce_add_sync(0xFFFFFFFFu, c) >= need) res = cand;
  }
  return res;   // keys 0 never count (positions absent from the list)
}

constexpr int kStepBytes = kStep * 2;            // one bulk-copy stage (16 KB)
constexpr int kStages = 5;                       // stages in flight (80 KB per CTA)

struct SelShared {
  uint64_t bar[kStages];                    // stage ring (bulk copies of the row)
  unsigned int cons[kStages];               // warps done with a stage's current fill
  unsigned int bad;                         // a bounded wait timed out
  Hist H;
  unsigned int count, thresh, last, nbest, nlive;
  unsigned int hmax[2 * kWarps];            // half-warp maxima of the first step
  unsigned int wkth[kWarps];                // each warp's K-th largest queued key
  unsigned long long best[WQL_MAX_TOPK];    // running fp32 top-K, descending
  unsigned int queue[kCap];                 // positions
  unsigned short qkey[kCap];                // their keys
  unsigned long long cand[kCap];            // recomputed fp32 keys
  unsigned int live[kCap];                  // positions to recompute, packed
};

// The need-th largest of cnt keys qkey[0..cnt) (block-wide; every thread
// returns it).
__device__ unsigned int queued_kth(SelShared& S, int cnt, unsigned int need) {
  if (cnt <= 32) {
    // one key per lane: the need-th largest is the smallest key with fewer
    // than `need` keys strictly above it
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const unsigned int mine = lane < cnt ? (unsigned int)S.qkey[lane] : 0u;
      unsigned int above = 0u;
#pragma unroll
      for (int j = 0; j < 32; ++j) above += __shfl_sync(0xFFFFFFFFu, mine, j) > mine ? 1u : 0u;
      const unsigned int h =
          __reduce_min_sync(0xFFFFFFFFu, (lane < cnt && above < need) ? mine : 0xFFFFFFFFu);
      if (lane == 0) S.thresh = h == 0xFFFFFFFFu ? 0u : h;
    }
    __syncthreads();
    const unsigned int h = S.thresh;
    __syncthreads();
    return h;
  }
  if (cnt <= 32 * kWarpKeys) {
    if (threadIdx.x < 32) {
      const unsigned int h =
          warp_kth_key(cnt, need, [&](int i) -> unsigned int { return S.qkey[i]; });
      if (threadIdx.x == 0) S.thresh = h;
    }
    __syncthreads();
    const unsigned int h = S.thresh;
    __syncthreads();
    return h;
  }
  return kth_key<kThreads>(S.H, cnt, need, [&](int i) -> unsigned int { return S.qkey[i]; });
}

// fp32 logit of vocab row r (a half-warp): exact q times x summed per 32-bit
// word in fp32, times the group scale, accumulated in fp32.  Each of the 16
// lanes takes words lane, lane + 16, ...; a batch's words and scales are
// loaded before any arithmetic; the activations come from shared memory.
template <typename XT>
__device__ float recompute(const LogitsArgs& a, const XT* xs, int r) {
  constexpr int kB = 8;
  const int lane = threadIdx.x & 15;
  const int k = a.k, ng = k / a.group_eff;
  const int per_word = a.bits == 4 ? 8 : 4;              // codes per 32-bit word
  const int nwords = k / per_word;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(a.qweight) + (size_t)r * nwords;
  const uint16_t* srow = a.scales + (size_t)r * ng;
  float acc = 0.f;
  for (int i0 = lane; i0 < nwords; i0 += 16 * kB) {
    uint32_t word[kB];
    uint16_t sb[kB];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int i = i0 + 16 * b;
      const bool ok = i < nwords;
      word[b] = ok ? __ldg(w + i) : 0u;
      sb[b] = ok ? ldg_u16(srow + i * per_word / a.group_eff) : (uint16_t)0;
    }
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int i = i0 + 16 * b;
      if (i >= nwords) break;
      float part = 0.f;
      if (a.bits == 4) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + 8 * i);
        const XT* xe = reinterpret_cast<const XT*>(&xv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int q = (int)((word[b] >> (4 * nibble_pos(j))) & 0xFu) - 8;
          part = fmaf(to_f32(xe[j]), (float)q, part);
        }
      } else {
        const uint2 xv = *reinterpret_cast<const uint2*>(xs + 4 * i);
        const XT* xe = reinterpret_cast<const XT*>(&xv);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int q = (int)(int8_t)((word[b] >> (8 * j)) & 0xFFu);
          part = fmaf(to_f32(xe[j]), (float)q, part);
        }
      }
      acc = fmaf(part, scale_to_f32(sb[b], a.scale_dtype), acc);
    }
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (a.bias) acc += to_f32(reinterpret_cast<const XT*>(a.bias)[r]);
  return acc;
}

// Recompute the queued positions with key >= key_min (a half-warp each) and
// fold them into the running top-K S.best (warp 0).  Ends with a barrier.
template <typename XT, int KT>
__device__ void recompute_and_merge(const LogitsArgs& a, SelShared& S, const XT* xs, int cnt,
                                    unsigned int key_min) {
  const int hw = threadIdx.x >> 4, lane = threadIdx.x & 31;
  constexpr int kHalfWarps = kThreads / 16;
  // the positions to recompute, packed (their keys are no longer needed)
  if (threadIdx.x == 0) S.nlive = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < cnt; i += kThreads)
    if (S.qkey[i] >= key_min) S.live[atomicAdd(&S.nlive, 1u)] = S.queue[i];
  __syncthreads();
  const int nlive = (int)S.nlive;
  // every half-warp runs the same number of rounds (the shuffles need both
  // halves of a warp)
  const int rounds = (nlive + kHalfWarps - 1) / kHalfWarps;
  for (int rr = 0; rr < rounds; ++rr) {
    const int i = rr * kHalfWarps + hw;
    const int r = i < nlive ? (int)S.live[i] : 0;
    const float v = recompute<XT>(a, xs, r);
    if (i < nlive && (threadIdx.x & 15) == 0) S.cand[i] = topk_key(v, (uint32_t)r);
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == 0) {
    unsigned long long list[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) list[i] = (lane == 0 && i < (int)S.nbest) ? S.best[i] : kEmptyKey;
    for (int i = lane; i < nlive; i += 32) list_insert<KT>(list, S.cand[i]);
    unsigned long long outk[KT];
    warp_merge_topk_redux<KT>(list, a.topk, outk);
    if (lane == 0) {
      int nb = 0;
#pragma unroll
      for (int i = 0; i < KT; ++i) {
        if (i < a.topk) S.best[i] = outk[i];
        nb += (i < a.topk && outk[i] != kEmptyKey) ? 1 : 0;
      }
      S.nbest = (unsigned int)nb;
    }
  }
  __syncthreads();
}

template <typename XT, int KT>
__global__ void __launch_bounds__(kThreads, 2) topk_select_kernel(const LogitsArgs a, int parts) {
  __shared__ SelShared S;
  extern __shared__ __align__(128) uint8_t ring[];   // kStages x kStepBytes, then x
  XT* xs = reinterpret_cast<XT*>(ring + (size_t)kStages * kStepBytes);
  const int tok = blockIdx.x, part = blockIdx.y, n = a.n, K = a.topk;
  const int lane = threadIdx.x & 31;
  const int per = ((n + parts - 1) / parts + kPer - 1) / kPer * kPer;
  const int lo = min(n, part * per), hi = min(n, lo + per);
  const int need = min(K, hi - lo);
  const uint16_t* row = reinterpret_cast<const uint16_t*>(a.logits) + (size_t)tok * n;
  const bool vec = (n % kPer == 0) && (reinterpret_cast<uintptr_t>(a.logits) % 16 == 0);
  if (threadIdx.x == 0) {
    S.count = 0u;
    S.thresh = 0u;
    S.nbest = 0u;
    S.bad = 0u;
  }
  if (threadIdx.x < kWarps) S.wkth[threadIdx.x] = 0u;
  griddep_launch_dependents();
  griddep_wait();   // the logits kernel before it has finished
  // ---- this range's candidates ----
  // Queue every position with key >= thresh; `keys_of(l)` gives this
  // thread's l-th group of 8 raw logits of the current step.
  // Queue every position whose key reaches thresh; each thread returns the
  // largest key it queued (0 if none).
  auto queue_step = [&](int base, unsigned int thresh, const uint4 (&cur)[kLoads]) -> unsigned int {
    unsigned int top = 0u;
    auto enqueue = [&](int pos, unsigned int key) {
      const unsigned int at = atomicAdd(&S.count, 1u);
      if (at < (unsigned int)kCap) {
        S.queue[at] = (unsigned int)pos;
        S.qkey[at] = (unsigned short)key;
      }
      top = max(top, key);
    };
    if (thresh >= 0x8000u) {
      // the common case: nothing of the thread's 32 logits reaches it
      const uint32_t t = thresh & 0x7FFFu;
      if (!any_reaches_pos(cur, t)) return 0u;
      const uint32_t t2 = t * 0x10001u;
#pragma unroll
      for (int l = 0; l < kLoads; ++l) {
        const uint32_t wv[4] = {cur[l].x, cur[l].y, cur[l].z, cur[l].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t hit = reach_bits_pos(wv[i], t2);
          if (hit == 0u) continue;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int pos = base + (l * kThreads + threadIdx.x) * kPer + 2 * i + h;
            if (((hit >> (16 * h + 15)) & 1u) != 0u && pos < hi)
              enqueue(pos, ((wv[i] >> (16 * h)) & 0xFFFFu) | 0x8000u);
          }
        }
      }
    } else {
      // a negative threshold: every key is tested
#pragma unroll
      for (int l = 0; l < kLoads; ++l) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          const int pos = base + (l * kThreads + threadIdx.x) * kPer + e;
          const unsigned int key = key16(raw_half(cur[l], e));
          if (pos < hi && key >= thresh) enqueue(pos, key);
        }
      }
    }
    return top;
  };
  // The selection threshold rises during the scan: each warp keeps, in lanes
  // 0 .. need-1, the need largest keys its threads have queued (at most one
  // per thread and step), sorted descending, and publishes the need-th of
  // them in S.wkth.  Those are keys of distinct positions of the range, so
  // each published key, and the largest of them, is a lower bound of the
  // range's need-th largest key; the published values only grow.
  unsigned int lst = 0u;
  auto raise_bound = [&](unsigned int top) {
    unsigned int hits = __ballot_sync(0xFFFFFFFFu, top != 0u);
    if (hits == 0u) return;
    while (hits != 0u) {
      const int src = __ffs(hits) - 1;
      hits &= hits - 1u;
      const unsigned int key = __shfl_sync(0xFFFFFFFFu, top, src);
      const unsigned int at =
          (unsigned int)__popc(__ballot_sync(0xFFFFFFFFu, lane < need && lst >= key));
      const unsigned int up = __shfl_up_sync(0xFFFFFFFFu, lst, 1);
      if (lane < need && (unsigned int)lane >= at) lst = (unsigned int)lane == at ? key : up;
    }
    const unsigned int kth = __shfl_sync(0xFFFFFFFFu, lst, (need - 1) & 31);
    if (lane == 0) S.wkth[threadIdx.x >> 5] = kth;
  };
  auto current_bound = [&](unsigned int t) {
    const volatile unsigned int* wk = S.wkth;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t = max(t, wk[w]);
    return t;
  };
  // threshold: need-th largest of the 16 half-warp maxima of the first
  // step (positions >= hi count as key 0, below every real key)
  auto first_threshold = [&](const uint4 (&cur)[kLoads]) -> unsigned int {
    unsigned int mx = 0u;
#pragma unroll
    for (int l = 0; l < kLoads; ++l)
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        const int pos = lo + (l * kThreads + threadIdx.x) * kPer + e;
        mx = max(mx, pos < hi ? key16(raw_half(cur[l], e)) : 0u);
      }
    const unsigned int m0 = redux_max_u32(lane < 16 ? mx : 0u);
    const unsigned int m1 = redux_max_u32(lane >= 16 ? mx : 0u);
    if (lane == 0) {
      S.hmax[2 * (threadIdx.x >> 5)] = m0;
      S.hmax[2 * (threadIdx.x >> 5) + 1] = m1;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      constexpr int kH = 2 * kWarps;
      const unsigned int mine = lane < kH ? S.hmax[lane] : 0u;
      int above = 0;
#pragma unroll
      for (int j = 0; j < kH; ++j) {
        const unsigned int o = S.hmax[j];
        above += (o > mine || (o == mine && j < lane)) ? 1 : 0;
      }
      if (lane < kH && above == need - 1) S.thresh = mine;
    }
    __syncthreads();
    return S.thresh;
  };
  unsigned int thresh = 0u;
  if (vec) {
    // bulk copies of 16 KB steps through a kStages-deep ring in shared
    // memory (ranges start and end on 8-position, 16-byte boundaries here)
    const int nsteps = (hi - lo + kStep - 1) / kStep;
    auto issue = [&](int st) {
      const int start = lo + st * kStep;
      const uint32_t bytes = (uint32_t)(min(kStep, hi - start) * 2);
      mbar_arrive_expect_tx(&S.bar[st % kStages], bytes);
      bulk_load(ring + (size_t)(st % kStages) * kStepBytes, row + start, bytes,
                &S.bar[st % kStages]);
    };
    if (threadIdx.x == 0) {
      for (int b = 0; b < kStages; ++b) {
        mbar_init(&S.bar[b], 1);
        S.cons[b] = 0u;
      }
      fence_barrier_init();
      S.bad = 0u;
      for (int st = 0; st < kStages && st < nsteps; ++st) issue(st);
    }
    // the token's activations, for the recompute (loaded while the first
    // copies are in flight)
    {
      const uint4* xg = reinterpret_cast<const uint4*>(reinterpret_cast<const XT*>(a.x) +
                                                       (size_t)tok * a.k);
      for (int i = threadIdx.x; i < a.k / 8; i += kThreads)
        reinterpret_cast<uint4*>(xs)[i] = __ldg(xg + i);
    }
    __syncthreads();
    for (int st = 0; st < nsteps; ++st) {
      const int b = st % kStages;
      if (!mbar_wait(&S.bar[b], (uint32_t)((st / kStages) & 1))) S.bad = 1u;
      uint4 cur[kLoads];
      const uint4* src = reinterpret_cast<const uint4*>(ring + (size_t)b * kStepBytes);
#pragma unroll
      for (int l = 0; l < kLoads; ++l) cur[l] = src[l * kThreads + threadIdx.x];
      if (st == 0) thresh = first_threshold(cur);     // all warps meet here once
      // the step's data is in registers: release the stage; the last warp
      // to release it refills it (no block-wide barrier per step)
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        if (atomicAdd(&S.cons[b], 1u) == (unsigned int)(kWarps - 1)) {
          S.cons[b] = 0u;
          if (st + kStages < nsteps) issue(st + kStages);
        }
      }
      if (st > 0) thresh = current_bound(thresh);
      raise_bound(queue_step(lo + st * kStep, thresh, cur));
    }
    __syncthreads();
    if (S.bad != 0u) {
      // a copy did not arrive in time (a stalled GPU): record it in the
      // error word, wait (bounded) for every stage's last fill, and report
      // nothing for this range
      if (threadIdx.x == 0) {
        atomicOr(a.counter + 1, 4u);
        for (int b = 0; b < kStages && b < nsteps; ++b) {
          const int last = b + (nsteps - 1 - b) / kStages * kStages;
          mbar_wait(&S.bar[b], (uint32_t)((last / kStages) & 1));
        }
        S.count = 0u;
      }
      __syncthreads();
    }
  } else {
    // the token's activations, for the recompute
    {
      const uint4* xg = reinterpret_cast<const uint4*>(reinterpret_cast<const XT*>(a.x) +
                                                       (size_t)tok * a.k);
      for (int i = threadIdx.x; i < a.k / 8; i += kThreads)
        reinterpret_cast<uint4*>(xs)[i] = __ldg(xg + i);
    }
    // rows not 16-byte aligned: register loads, the next step's issued
    // before the current one is compared
    uint4 cur[kLoads];
#pragma unroll
    for (int l = 0; l < kLoads; ++l)
      cur[l] = load_raw(row, hi, lo + (l * kThreads + threadIdx.x) * kPer, false);
    thresh = first_threshold(cur);
    for (int base = lo; base < hi; base += kStep) {
      uint4 nxt[kLoads];
#pragma unroll
      for (int l = 0; l < kLoads; ++l)
        nxt[l] = base + kStep < hi
                     ? load_raw(row, hi, base + kStep + (l * kThreads + threadIdx.x) * kPer, false)
                     : make_uint4(0u, 0u, 0u, 0u);
      thresh = current_bound(thresh);
      raise_bound(queue_step(base, thresh, cur));
#pragma unroll
      for (int l = 0; l < kLoads; ++l) cur[l] = nxt[l];
    }
  }
  __syncthreads();
  const int cnt = (int)S.count;
  if (need > 0 && cnt <= kCap) {
    // recompute the positions with key >= the range's K-th queued key
    const unsigned int h = queued_kth(S, cnt, (unsigned int)need);
    recompute_and_merge<XT, KT>(a, S, xs, cnt, h);
  } else if (need > 0) {
    // many positions above the threshold: the range exactly, in chunks
    unsigned int th = thresh;
    for (int base = lo; base < hi; base += kChunk) {
      if (threadIdx.x == 0) S.count = 0u;
      __syncthreads();
#pragma unroll
      for (int e = 0; e < kChunk / kThreads; ++e) {
        const int pos = base + e * kThreads + threadIdx.x;
        if (pos < hi) {
          const unsigned int key = key16((unsigned int)__ldcg(row + pos));
          if (key >= th) {
            const unsigned int at = atomicAdd(&S.count, 1u);   // < kChunk <= kCap
            S.queue[at] = (unsigned int)pos;
            S.qkey[at] = (unsigned short)key;
          }
        }
      }
      __syncthreads();
      recompute_and_merge<XT, KT>(a, S, xs, (int)S.count, th);
      // a later position enters only with an fp32 value above the K-th,
      // hence with a rounded value >= the K-th's rounded value
      if ((int)S.nbest == K) th = max(th, key_of_f32<XT>(key_value(S.best[K - 1])));
    }
  }
  // this range's best K (fp32 keys; empty entries where it has fewer)
  unsigned long long* slots = a.cand + (size_t)tok * WQL_MAX_CTAS * K;
  if (threadIdx.x < K)
    slots[(size_t)part * K + threadIdx.x] =
        threadIdx.x < (int)S.nbest ? S.best[threadIdx.x] : kEmptyKey;
  // ---- the token's last range to finish merges ----
  __syncthreads();
  unsigned int* ticket = a.tickets + tok;
  if (threadIdx.x == 0) {
    __threadfence();
    S.last = atomicAdd(ticket, 1u) == (unsigned int)(parts - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (S.last == 0u) return;
  __threadfence();
  if (threadIdx.x < 32) {
    unsigned long long list[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) list[i] = kEmptyKey;
    for (int i = lane; i < parts * K; i += 32) list_insert<KT>(list, __ldcg(slots + i));
    unsigned long long outk[KT];
    warp_merge_topk_redux<KT>(list, K, outk);
    // a timed-out wait of this call's kernels (or an earlier one's, until
    // the caller clears the error word) voids the result
    const bool failed = __ldcg(a.counter + 1) != 0u;
    const unsigned long long b = failed ? kEmptyKey : pick(outk, lane);
    if (lane < K) {
      a.topk_idx[(size_t)tok * K + lane] = b == kEmptyKey ? -1 : key_index(b);
      a.topk_val[(size_t)tok * K + lane] =
          b == kEmptyKey ? __int_as_float(0x7FC00000) : key_value(b);
    }
    if (lane == 0) *ticket = 0u;   // ready for the next call
  }
}

template <typename XT, int KT>
cudaError_t launch_t(const LogitsArgs& a, cudaStream_t s) {
  // ranges per token: one wave of CTAs (two per SM), none shorter than one
  // step, at most WQL_MAX_CTAS (the workspace's slots per token)
  int parts = (2 * device_sm_count()) / a.m;
  parts = max(1, min(parts, min(WQL_MAX_CTAS, (a.n + kMinRange - 1) / kMinRange)));
  const size_t smem = (size_t)kStages * kStepBytes + (size_t)a.k * 2;
  auto kern = topk_select_kernel<XT, KT>;
  static size_t configured = 0;
  if (smem > configured) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const cudaError_t e = launch_pdl(kern, dim3(a.m, parts), dim3(kThreads), smem, s, a, parts);
  note_launch();
  return e;
}

}  // namespace

cudaError_t launch_topk_select(const LogitsArgs& a, cudaStream_t s) {
  if (a.topk <= 0 || a.m <= 0) return cudaSuccess;
  if (a.x_dtype == WQL_F16)
    return a.topk <= 8 ? launch_t<__half, 8>(a, s) : launch_t<__half, 16>(a, s);
  return a.topk <= 8 ? launch_t<__nv_bfloat16, 8>(a, s) : launch_t<__nv_bfloat16, 16>(a, s);
}

}  // namespace wql
