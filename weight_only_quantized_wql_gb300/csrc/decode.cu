// decode.cu -- logits of a weight-only quantised lm_head for small token
// counts (m <= 16), the bandwidth-bound decode case ("Fused WNA16 GEMM for
// tied quantized lm_head logits", Perf evals rows M = 1; reviewer comment
// item 1: at M = 1 only the bytes moved matter).
//
// Design (sm_103a):
//  * Swap-AB warp MMA: a warp owns a 16-row vocab tile; the packed weight is
//    operand A (dequantised in registers, never written anywhere), the tokens
//    are operand B (n = 8 per MMA, zero-padded), fp32 accumulators.
//  * Each lane streams its share of a k-step (64 or 128 hidden columns) with
//    16/8-byte non-allocating loads, PD k-steps ahead of the math.
//  * Codes become exact fp16/bf16 values with the LOP3/PRMT magic-number
//    tricks (wql_common.cuh); q*x products are exact, sums are fp32.
//  * Per-group scales are applied exactly in fp32: every MMA of a k-step
//    stays inside one scale group, so the k-step partial is multiplied by
//    s[row, group] once.
//  * Top-K: fp32 logits go to a scratch row; when its tiles are done each
//    CTA selects its own top-K per token, and the last CTA to finish merges
//    every CTA's candidates (atomic ticket, no waiting).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "wql_common.cuh"

namespace wql {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;

template <int BITS, int KS>
struct StepShape {
  // 32-bit words one lane loads per row per k-step
  static constexpr int kWordsPerLane = BITS == 4 ? KS / 32 : KS / 16;
  // bytes of packed weight per row per k-step
  static constexpr int kRowBytes = KS * BITS / 8;
  // halves of X a lane reads per token row per k-step
  static constexpr int kXHalves = BITS == 4 ? 8 * kWordsPerLane : 4 * kWordsPerLane;
};

template <int WPL>
struct WordBuf {
  uint32_t a[WPL];   // row g
  uint32_t b[WPL];   // row g + 8
  uint16_t sa, sb;   // raw scale bits for rows g, g + 8
};

template <int WPL>
__device__ __forceinline__ void load_words(uint32_t (&dst)[WPL], const uint8_t* p) {
  if constexpr (WPL == 2) {
    uint2 v = ldg_stream_u2(p);
    dst[0] = v.x; dst[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < WPL; i += 4) {
      uint4 v = ldg_stream_u4(p + 4 * i);
      dst[i] = v.x; dst[i + 1] = v.y; dst[i + 2] = v.z; dst[i + 3] = v.w;
    }
  }
}

template <int BITS, typename XT, int NT, int KS, int PD>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const LogitsArgs a) {
  using S = StepShape<BITS, KS>;
  constexpr int WPL = S::kWordsPerLane;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // X staged once per CTA: [m][k] halves; for int4 each group of 8 columns is
  // stored as (0,4,1,5,2,6,3,7) so that the (j, j+4) code pairs of a packed
  // word meet adjacent activations.
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);
  __shared__ unsigned long long warp_best[kWarps][WQL_MAX_TOPK];
  __shared__ unsigned int is_last;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;     // MMA group id: rows g and g + 8, token column g
  const int t = lane & 3;      // thread in group: k sub-range and token pair
  const int m = a.m, n = a.n, k = a.k;

  {
    const uint16_t* xg = reinterpret_cast<const uint16_t*>(a.x);
    for (int i = threadIdx.x; i < m * k; i += kThreads) {
      int row = i / k, col = i - row * k;
      int dst = col;
      if (BITS == 4) {
        int j = col & 7;
        dst = (col & ~7) + (j < 4 ? 2 * j : 2 * (j - 4) + 1);
      }
      xs[row * k + dst] = xg[i];
    }
  }
  __syncthreads();

  const int ntiles = (n + 15) >> 4;
  const int tile_begin = (int)(((long long)ntiles * blockIdx.x) / gridDim.x);
  const int tile_end = (int)(((long long)ntiles * (blockIdx.x + 1)) / gridDim.x);
  const int my_tiles = tile_end - tile_begin > warp
                           ? (tile_end - tile_begin - warp + kWarps - 1) / kWarps : 0;
  const int nks = k / KS;
  const int steps_per_group = a.group_eff / KS;
  const int ngroups = k / a.group_eff;
  const int total = my_tiles * nks;
  const size_t row_bytes = (size_t)k * BITS / 8;
  const uint8_t* qw = reinterpret_cast<const uint8_t*>(a.qweight);

  auto issue = [&](int it, WordBuf<WPL>& buf) {
    if (it < total) {
      int tile = tile_begin + warp + kWarps * (it / nks);
      int ks = it % nks;
      int r0 = tile * 16 + g, r1 = r0 + 8;
      r0 = r0 < n ? r0 : n - 1;
      r1 = r1 < n ? r1 : n - 1;
      size_t off = (size_t)ks * S::kRowBytes + (size_t)t * WPL * 4;
      load_words<WPL>(buf.a, qw + (size_t)r0 * row_bytes + off);
      load_words<WPL>(buf.b, qw + (size_t)r1 * row_bytes + off);
      if ((ks % steps_per_group) == steps_per_group - 1) {
        int gi = (ks * KS) / a.group_eff;
        buf.sa = ldg_u16(a.scales + (size_t)r0 * ngroups + gi);
        buf.sb = ldg_u16(a.scales + (size_t)r1 * ngroups + gi);
      }
    }
  };

  float acc[NT][4];
  float part[NT][4];
  WordBuf<WPL> ring[PD];
#pragma unroll
  for (int s = 0; s < PD; ++s) issue(s, ring[s]);

  const bool want_scratch = a.topk > 0;

  for (int base = 0; base < total; base += PD) {
#pragma unroll
    for (int s = 0; s < PD; ++s) {
      const int it = base + s;
      if (it < total) {
        const int ks = it % nks;
        if (ks == 0) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;
        }
        if ((ks % steps_per_group) == 0) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) part[nt][c] = 0.f;
        }
        // ---- B fragments (activations) for this k-step ----
        uint32_t xb[NT][S::kXHalves / 2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int tok = nt * 8 + g;
          if (tok < m) {
            const uint4* src = reinterpret_cast<const uint4*>(
                xs + (size_t)tok * k + ks * KS + t * S::kXHalves);
#pragma unroll
            for (int v = 0; v < S::kXHalves / 8; ++v) {
              uint4 q4 = src[v];
              xb[nt][4 * v] = q4.x; xb[nt][4 * v + 1] = q4.y;
              xb[nt][4 * v + 2] = q4.z; xb[nt][4 * v + 3] = q4.w;
            }
          } else {
#pragma unroll
            for (int v = 0; v < S::kXHalves / 2; ++v) xb[nt][v] = 0u;
          }
        }
        // ---- dequantise operand A and multiply ----
        WordBuf<WPL>& cur = ring[s];
        if constexpr (BITS == 4) {
#pragma unroll
          for (int w = 0; w < WPL; ++w) {
            uint32_t pa[4], pb[4];
            Int4Dequant<XT>::run(cur.a[w], pa);
            Int4Dequant<XT>::run(cur.b[w], pb);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t afrag[4] = {pa[2 * h], pb[2 * h], pa[2 * h + 1], pb[2 * h + 1]};
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                Mma16816<XT>::run(part[nt], afrag, xb[nt][4 * w + 2 * h],
                                  xb[nt][4 * w + 2 * h + 1], part[nt]);
              }
            }
          }
        } else {
#pragma unroll
          for (int w = 0; w < WPL; ++w) {
            uint32_t pa[2], pb[2];
            Int8Dequant<XT>::run(cur.a[w], pa);
            Int8Dequant<XT>::run(cur.b[w], pb);
            const uint32_t afrag[4] = {pa[0], pb[0], pa[1], pb[1]};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              Mma16816<XT>::run(part[nt], afrag, xb[nt][2 * w], xb[nt][2 * w + 1], part[nt]);
            }
          }
        }
        if ((ks % steps_per_group) == steps_per_group - 1) {
          const float sa = scale_to_f32(cur.sa, a.scale_dtype);
          const float sb = scale_to_f32(cur.sb, a.scale_dtype);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            acc[nt][0] = fmaf(sa, part[nt][0], acc[nt][0]);
            acc[nt][1] = fmaf(sa, part[nt][1], acc[nt][1]);
            acc[nt][2] = fmaf(sb, part[nt][2], acc[nt][2]);
            acc[nt][3] = fmaf(sb, part[nt][3], acc[nt][3]);
          }
        }
        // refill this ring slot PD k-steps ahead
        issue(it + PD, ring[s]);
        if (ks == nks - 1) {
          const int tile = tile_begin + warp + kWarps * (it / nks);
          const int rows[2] = {tile * 16 + g, tile * 16 + g + 8};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int row = rows[c >> 1];
              const int tok = nt * 8 + 2 * t + (c & 1);
              if (row < n && tok < m) {
                float v = acc[nt][c];
                if (a.bias) v += to_f32(reinterpret_cast<const XT*>(a.bias)[row]);
                reinterpret_cast<XT*>(a.logits)[(size_t)tok * n + row] = from_f32<XT>(v);
                if (want_scratch) a.scratch[(size_t)tok * n + row] = v;
              }
            }
          }
        }
      }
    }
  }

  if (a.topk <= 0) return;

  // ---------------- per-CTA top-K of this CTA's rows ----------------
  __syncthreads();
  __threadfence_block();
  const int row_begin = tile_begin * 16;
  const int row_end = min(tile_end * 16, n);
  const int K = a.topk;
  for (int tok = 0; tok < m; ++tok) {
    unsigned long long list[WQL_MAX_TOPK];
#pragma unroll
    for (int i = 0; i < WQL_MAX_TOPK; ++i) list[i] = kEmptyKey;
    const float* src = a.scratch + (size_t)tok * n;
    for (int r = row_begin + threadIdx.x; r < row_end; r += kThreads)
      list_insert<WQL_MAX_TOPK>(list, topk_key(__ldcg(src + r), (uint32_t)r));
    unsigned long long best[WQL_MAX_TOPK];
    warp_merge_topk<WQL_MAX_TOPK>(list, K, best);
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < WQL_MAX_TOPK; ++i) warp_best[warp][i] = best[i];
    }
    __syncthreads();
    if (warp == 0) {
      unsigned long long l2[WQL_MAX_TOPK];
#pragma unroll
      for (int i = 0; i < WQL_MAX_TOPK; ++i) l2[i] = kEmptyKey;
      if (lane < kWarps) {
#pragma unroll
        for (int i = 0; i < WQL_MAX_TOPK; ++i) l2[i] = warp_best[lane][i];
      }
      warp_merge_topk<WQL_MAX_TOPK>(l2, K, best);
      const unsigned long long mine = pick(best, lane);
      if (lane < K) {
        a.cand[((size_t)tok * WQL_MAX_CTAS + blockIdx.x) * K + lane] = mine;
        __threadfence();
      }
    }
    __syncthreads();
  }

  // ---------------- last CTA merges every CTA's candidates ----------------
  if (threadIdx.x == 0) {
    __threadfence();
    unsigned int ticket = atomicAdd(a.counter, 1u);
    is_last = (ticket == gridDim.x - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int ncand = gridDim.x * K;
  for (int tok = warp; tok < m; tok += kWarps) {
    unsigned long long list[WQL_MAX_TOPK];
#pragma unroll
    for (int i = 0; i < WQL_MAX_TOPK; ++i) list[i] = kEmptyKey;
    const unsigned long long* src = a.cand + (size_t)tok * WQL_MAX_CTAS * K;
    for (int i = lane; i < ncand; i += 32) list_insert<WQL_MAX_TOPK>(list, __ldcg(src + i));
    unsigned long long best[WQL_MAX_TOPK];
    warp_merge_topk<WQL_MAX_TOPK>(list, K, best);
    const unsigned long long mine = pick(best, lane);
    if (lane < K) {
      a.topk_idx[(size_t)tok * K + lane] = key_index(mine);
      a.topk_val[(size_t)tok * K + lane] = key_value(mine);
    }
  }
  if (threadIdx.x == 0) *a.counter = 0u;
}

template <int BITS, typename XT, int NT, int KS, int PD>
cudaError_t launch_t(const LogitsArgs& a, cudaStream_t s) {
  auto kern = decode_kernel<BITS, XT, NT, KS, PD>;
  const size_t smem = (size_t)a.m * a.k * sizeof(uint16_t);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const int ntiles = (a.n + 15) / 16;
  int ctas = device_sm_count();
  // at least one tile per warp where the vocab is small
  int by_tiles = (ntiles + kWarps - 1) / kWarps;
  if (ctas > by_tiles) ctas = by_tiles;
  if (ctas < 1) ctas = 1;
  if (ctas > WQL_MAX_CTAS) ctas = WQL_MAX_CTAS;
  decode_kernel<BITS, XT, NT, KS, PD><<<ctas, kThreads, smem, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

template <typename XT>
cudaError_t dispatch_x(const LogitsArgs& a, cudaStream_t s) {
  const bool g64 = (a.group_eff % 128) != 0;   // group_eff is a multiple of 64
  const int nt = a.m <= 8 ? 1 : 2;
  if (a.bits == 4) {
    if (g64) return nt == 1 ? launch_t<4, XT, 1, 64, 4>(a, s) : launch_t<4, XT, 2, 64, 4>(a, s);
    return nt == 1 ? launch_t<4, XT, 1, 128, 3>(a, s) : launch_t<4, XT, 2, 128, 3>(a, s);
  }
  if (g64) return nt == 1 ? launch_t<8, XT, 1, 64, 3>(a, s) : launch_t<8, XT, 2, 64, 3>(a, s);
  return nt == 1 ? launch_t<8, XT, 1, 128, 2>(a, s) : launch_t<8, XT, 2, 128, 2>(a, s);
}

}  // namespace

cudaError_t launch_decode(const LogitsArgs& a, cudaStream_t s) {
  if (a.x_dtype == WQL_F16) return dispatch_x<__half>(a, s);
  return dispatch_x<__nv_bfloat16>(a, s);
}

}  // namespace wql
