// embed.cu -- tied-embedding gather ("Fused WNA16 GEMM for tied quantized
// lm_head logits", Purpose: the tied head's quantised weight is also the
// input embedding): out[i, :] = RN_out(q[ids[i], :] * s[ids[i], group]).
//
// Memory-bound and tiny next to the logits: a thread turns 8 codes of one
// row (one int4 word or two int8 words, consecutive threads on consecutive
// words, so a warp reads 128 or 256 contiguous bytes of the packed row) into
// 8 outputs stored as one 16-byte write, four such pieces per pass with all
// their loads issued before any is used (the id load heads a chain of two).  The product of a code (at most 8
// bits) and a scale (11- or 8-bit significand) is exact in fp32, so the one
// rounding is the conversion to the output dtype, round-to-nearest-even.
// Grid-stride over (token, 8-element piece) pairs; an id outside [0, n)
// gives a row of zeros.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "embed.cuh"

namespace wql {
namespace {

// element 8w + j of a row sits in nibble 4 * (j % 2) + j / 2 of word w
__device__ __forceinline__ int int4_code(uint32_t word, int j) {
  return (int)((word >> (4 * (4 * (j & 1) + (j >> 1)))) & 15u) - 8;
}

template <int BITS, typename OT>
__global__ void __launch_bounds__(256) embed_gather_kernel(const EmbedArgs a) {
  constexpr int kU = 4;                             // pieces per thread per pass (loads first)
  const int pieces = a.k / 8;                       // 8-element pieces per row
  const int ng = a.k / a.group_eff;
  const long long total = (long long)a.t * pieces;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long p0 = (long long)blockIdx.x * blockDim.x + threadIdx.x; p0 < total;
       p0 += kU * stride) {
    int tok[kU], pc[kU], id[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long p = p0 + u * stride;
      tok[u] = (int)(min(p, total - 1) / pieces);
      pc[u] = (int)(min(p, total - 1) - (long long)tok[u] * pieces);
      id[u] = p < total ? __ldg(a.ids + tok[u]) : -1;
    }
    uint32_t w0[kU], w1[kU];
    uint16_t sb[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      w0[u] = w1[u] = 0u;
      sb[u] = 0;
      if (id[u] >= 0 && id[u] < a.n) {
        sb[u] = __ldg(a.scales + (size_t)id[u] * ng + (pc[u] * 8) / a.group_eff);
        if constexpr (BITS == 4) {
          w0[u] = __ldg(reinterpret_cast<const uint32_t*>(a.qweight) + (size_t)id[u] * pieces +
                        pc[u]);
        } else {
          const uint2 w = __ldg(reinterpret_cast<const uint2*>(a.qweight) +
                                (size_t)id[u] * pieces + pc[u]);
          w0[u] = w.x;
          w1[u] = w.y;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (p0 + u * stride >= total) break;
      uint32_t o[4] = {0u, 0u, 0u, 0u};
      if (id[u] >= 0 && id[u] < a.n) {
        const float s = scale_to_f32(sb[u], a.scale_dtype);
        int q[8];
        if constexpr (BITS == 4) {
#pragma unroll
          for (int j = 0; j < 8; ++j) q[j] = int4_code(w0[u], j);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            q[j] = (int)(int8_t)((w0[u] >> (8 * j)) & 0xFFu);
            q[4 + j] = (int)(int8_t)((w1[u] >> (8 * j)) & 0xFFu);
          }
        }
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          const OT lo = from_f32<OT>((float)q[j] * s);     // exact product, one rounding
          const OT hi = from_f32<OT>((float)q[j + 1] * s);
          o[j / 2] = (uint32_t)*reinterpret_cast<const uint16_t*>(&lo) |
                     ((uint32_t)*reinterpret_cast<const uint16_t*>(&hi) << 16);
        }
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<OT*>(a.out) + (size_t)tok[u] * a.k + pc[u] * 8) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

template <int BITS, typename OT>
cudaError_t launch_t(const EmbedArgs& a, cudaStream_t s) {
  const long long total = (long long)a.t * (a.k / 8);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)device_sm_count() * 32;  // 8 blocks per SM resident, 4 passes
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  embed_gather_kernel<BITS, OT><<<(unsigned)blocks, 256, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_embed_gather(const EmbedArgs& a, cudaStream_t s) {
  if (a.t == 0 || a.k == 0) return cudaSuccess;
  if (a.bits == 4)
    return a.out_dtype == WQL_F16 ? launch_t<4, __half>(a, s) : launch_t<4, __nv_bfloat16>(a, s);
  return a.out_dtype == WQL_F16 ? launch_t<8, __half>(a, s) : launch_t<8, __nv_bfloat16>(a, s);
}

}  // namespace wql
