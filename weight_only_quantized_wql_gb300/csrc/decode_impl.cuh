// decode_impl.cuh -- the decode kernel template (included by decode_f16.cu and
// decode_bf16.cu, which instantiate it per activation dtype).
//
// Logits of a weight-only quantised lm_head for small token
// counts (m <= 16), the bandwidth-bound decode case ("Fused WNA16 GEMM for
// tied quantized lm_head logits", Perf evals rows at M = 1; reviewer comment
// item 1: at M = 1 only the bytes moved matter).
//
// Design (sm_103a, one persistent CTA per SM):
//  * The CTA owns a contiguous range of 16-row vocab tiles, walked in blocks
//    of up to 256 rows.  Each block streams along the hidden dimension in
//    chunks of 128 packed bytes per row (256 int4 or 128 int8 codes).
//  * Warp 16 is the producer: one lane issues TMA tensor copies of every
//    chunk (16-row boxes, 128B-swizzled) and, once per block, a bulk copy of
//    the block's scale rows, into a 4-stage ring.  Activations are either
//    resident in shared memory for the whole launch or, when m*k is too
//    large for that, copied per chunk with the weights.
//  * Warps 0..15 are consumers, one 16-row tile each.  ldmatrix moves packed
//    words straight into the A-fragment layout of a warp MMA (m16n8k16, swap
//    AB: vocab rows = M, tokens = N).  A code becomes the exact 16-bit value
//    magic + u with one LOP3 (OffsetCodes); the MMA sums x*(q + offset) with
//    exact products and fp32 accumulation, and offset * sum(x) -- computed
//    once per launch for every (token, group) -- is subtracted per scale
//    group before the exact fp32 scale multiply.
//  * Top-K: fp32 logits go to a scratch row; each CTA selects its own rows'
//    top-K per token (all warps, token x row-slice), and the last CTA to
//    finish (atomic ticket, no waiting) merges all CTAs' candidates.
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

struct DecodeParams {
  LogitsArgs a;
  int tiles_total;      // ceil(n / 16)
  int chunks;           // chunks per row
  int gunits;           // 64-column units per scale group
  int ngroups;          // scale groups per row
  int x_resident;       // 1: activations staged once; 0: per chunk by TMA
  int xbox_bytes;       // per-chunk mode: bytes between activation boxes
  uint32_t off_x, off_s, off_corr, off_bar, off_red;
  int sbuf_bytes, nsb;  // scale buffer size and count
  int scales_aligned;   // scale table 16-byte aligned (bulk copies allowed)
  unsigned int* err;    // sticky error word in the workspace (null: none)
};

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

// This CTA's candidates, the ticket, and (last CTA only) the final merge.
template <int KT, typename XT>
__device__ __forceinline__ void topk_tail(const LogitsArgs& a, unsigned int* err,
                                          unsigned long long* red, unsigned int* flags,
                                          int row_begin, int row_end, bool cta_bad) {
  const int lane = threadIdx.x & 31;
  const int m = a.m, n = a.n, K = a.topk;
  if (!cta_bad) {
    unsigned long long best[KT];
    int tok;
    select_topk<KT>(
        m, K, row_end - row_begin, red,
        [&](int tk, int i) {
          const int r = row_begin + i;
          return topk_key(__ldcg(a.scratch + (size_t)tk * n + r), (uint32_t)r);
        },
        best, tok);
    if (tok >= 0) {
      const unsigned long long mine = pick(best, lane);
      if (lane < K) a.cand[((size_t)tok * WQL_MAX_CTAS + blockIdx.x) * K + lane] = mine;
      __threadfence();
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int ticket = atomicAdd(a.counter, 1u);
    flags[1] = (ticket == gridDim.x - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (flags[1] == 0u) return;
  __threadfence();
  const bool any_bad = (__ldcg(err) != 0u);
  unsigned long long best[KT];
  int tok;
  select_topk<KT>(
      m, K, any_bad ? 0 : (int)gridDim.x * K, red,
      [&](int tk, int i) { return __ldcg(a.cand + (size_t)tk * WQL_MAX_CTAS * K + i); }, best,
      tok);
  if (tok >= 0) {
    const unsigned long long mine = pick(best, lane);
    if (lane < K) {
      const bool ok = !any_bad && mine != kEmptyKey;
      a.topk_idx[(size_t)tok * K + lane] = ok ? key_index(mine) : -1;
      a.topk_val[(size_t)tok * K + lane] = ok ? key_value(mine) : __int_as_float(0x7FC00000);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *a.counter = 0u;
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
                  const __grid_constant__ CUtensorMap tx, const DecodeParams p) {
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

  const int T0 = (int)(((long long)p.tiles_total * blockIdx.x) / gridDim.x);
  const int T1 = (int)(((long long)p.tiles_total * (blockIdx.x + 1)) / gridDim.x);
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
      for (int tb = T0, blk = 0; tb < T1; tb += kBlockTiles, ++blk) {
        const int ntb = min(kBlockTiles, T1 - tb);
        const bool sc_bulk = p.scales_aligned && (tb + ntb) * 16 <= n;
        const uint32_t sbytes = (uint32_t)(ntb * 16 * p.ngroups * 2);
        for (int c = 0; c < p.chunks; ++c, ++j) {
          // stage reuse: wait until all consumers released its previous fill
          if (j >= kStages && !bad) bad = !mbar_wait(&empty[stage], ephase ^ 1u);
          if (!bad) {
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
              bulk_load(sm + p.off_s + (blk % p.nsb) * p.sbuf_bytes,
                        scales + (size_t)tb * 16 * p.ngroups * 2, sbytes, &full[stage]);
            issued = j + 1;
          }
          if (++stage == kStages) { stage = 0; ephase ^= 1u; }
        }
      }
      // Every copy this CTA issued must have landed before it can finish: the
      // latest fill of slot s completes phase (fills_of_s - 1) & 1.  On the
      // normal path the consumers already waited for all of them.
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int fills = (issued - 1 - s) / kStages + 1;
        if (!mbar_wait(&full[s], (uint32_t)((fills - 1) & 1))) bad = true;
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
    // (2) per (token, group): the offset the MMA sums picked up
    if constexpr (CF::kCorr) {
      const int G = p.gunits * 64;
      for (int pr = warp; pr < kMaxTok * p.ngroups; pr += kConsumers) {
        const int tok = pr / p.ngroups, gidx = pr - tok * p.ngroups;
        float s = 0.f;
        if (tok < m) {
          for (int e = lane; e < G; e += 32) {
            const XT xv = xg[(size_t)tok * k + gidx * G + e];
            if constexpr (CF::kScaledX) {
              const int j = e & 7;
              if (j == 2 || j == 3 || j == 6 || j == 7)
                s += 1152.0f * to_f32(__hmul(xv, __float2half_rn(0.0625f)));
              else
                s += 1032.0f * to_f32(xv);
            } else {
              s += Codes::kOffset * to_f32(xv);
            }
          }
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
    for (int tb = T0, blk = 0; tb < T1; tb += kBlockTiles, ++blk) {
      const int ntb = min(kBlockTiles, T1 - tb);
      const bool active = warp < ntb;
      const bool sc_bulk = p.scales_aligned && (tb + ntb) * 16 <= n;
      const int row_a = (tb + warp) * 16 + g, row_b = row_a + 8;
      const uint16_t* sbuf = reinterpret_cast<const uint16_t*>(sm + p.off_s +
                                                               (blk % p.nsb) * p.sbuf_bytes);
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
        if (!bad) bad = !mbar_wait(&full[stage], fphase);
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
              if (a.topk > 0) a.scratch[(size_t)tok * n + row] = v;
            }
          }
      }
    }
  }

  if (bad) atomicOr(&flags[0], 1u);
  __syncthreads();
  const bool cta_bad = flags[0] != 0u;
  if (cta_bad && threadIdx.x == 0 && p.err) atomicOr(p.err, 1u);
  if (a.topk <= 0) return;

  // ---------------- top-K: per-CTA selection, last-CTA merge ----------------
  const int row_begin = T0 * 16, row_end = min(T1 * 16, n);
  if (a.topk <= 8)
    topk_tail<8, XT>(a, p.err, red, flags, row_begin, row_end, cta_bad);
  else
    topk_tail<16, XT>(a, p.err, red, flags, row_begin, row_end, cta_bad);
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
