// quantize.cu -- load-time quantisation and packing of an lm_head weight
// (radiance_lmhead_int4.py, quantize_int4_rows and module constants; int8
// per the W8 rows of "Fused WNA16 GEMM for tied quantized lm_head logits").
//
// One thread owns one scale group (G columns, or the whole row).  Per tried
// clip ratio r it forms s = RN_sdtype(max(amax *f32 c_r, 1e-8f)) with
// c_r = fl32(r / qmax), picks q = clamp(rint(w /f32 s)) (q = 0 if s rounded
// to zero) and, when several ratios are tried, sums (q*s - w)^2 in binary64
// in column order with no fused multiply-add, keeping the first ratio with
// the strictly smallest error.  Every operation is the IEEE operation the
// definition names, so the result is bit-exact on any conforming machine.
// The weight is streamed from global memory (L1-cached re-reads); no fp32
// copy of the matrix is made.  The fp8 e4m3 per-row and the zero-point int4
// formats (wql_quantize_ex) follow their own definitions below.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "wql_common.cuh"

namespace wql {
namespace {

template <typename WT>
__device__ __forceinline__ float load_w(const WT* p, int64_t i) { return to_f32(p[i]); }

__device__ __forceinline__ uint16_t round_scale(float v, int sdt) {
  return sdt == WQL_F16 ? __half_as_ushort(__float2half_rn(v))
                        : __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ int code_of(float w, float s, int qmin, int qmax) {
  if (s == 0.0f) return 0;
  float r = rintf(__fdiv_rn(w, s));
  r = fminf(fmaxf(r, (float)qmin), (float)qmax);
  return (int)r;
}

// fp8 e4m3 codes of one row (WQL_FMT_E4M3): s = RN(max(amax * fl32(1/448),
// 1e-8)), q = RN_e4m3(clamp(w / s, -448, 448)) with ties to even (the
// conversion's own rounding; the clamp keeps NaN, which converts to NaN).
template <typename WT>
__device__ void quantize_e4m3_row(const QuantizeArgs& a, const WT* w, int64_t gid) {
  const int G = a.group_eff;
  float amax = 0.0f;
  for (int j = 0; j < G; ++j) amax = fmaxf(amax, fabsf(load_w(w, j)));
  float prod = __fmul_rn(amax, a.ratio_c[0]);
  prod = prod < 1e-8f ? 1e-8f : prod;
  const uint16_t sbits = round_scale(prod, a.scale_dtype);
  const float s = scale_to_f32(sbits, a.scale_dtype);
  a.scales[gid] = sbits;
  uint32_t* out = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(a.qweight) + gid * (int64_t)G);
  for (int j4 = 0; j4 < G; j4 += 4) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t c = 0;
      if (s != 0.0f) {
        float t = __fdiv_rn(load_w(w, j4 + j), s);
        if (t > 448.0f) t = 448.0f;
        if (t < -448.0f) t = -448.0f;
        c = (uint32_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
      }
      word |= c << (8 * j);
    }
    out[j4 / 4] = word;
  }
}

// Zero-point int4 codes of one group (WQL_FMT_ASYM): with lo = min(0, w)
// and hi = max(0, w), s = RN(max((hi - lo) * fl32(1/15), 1e-8)),
// z = clamp(rint(-lo / s), 0, 15), q = clamp(rint(w / s) + z, 0, 15).
template <typename WT>
__device__ void quantize_asym_group(const QuantizeArgs& a, const WT* w, int64_t row, int64_t gi,
                                    int64_t gid) {
  const int G = a.group_eff;
  float lo = 0.0f, hi = 0.0f;
  for (int j = 0; j < G; ++j) {
    const float v = load_w(w, j);
    if (v < lo) lo = v;
    if (v > hi) hi = v;
  }
  float prod = __fmul_rn(__fsub_rn(hi, lo), a.ratio_c[0]);
  prod = prod < 1e-8f ? 1e-8f : prod;
  const uint16_t sbits = round_scale(prod, a.scale_dtype);
  const float s = scale_to_f32(sbits, a.scale_dtype);
  a.scales[gid] = sbits;
  int z = 0;
  if (s != 0.0f) z = min(max((int)rintf(__fdiv_rn(-lo, s)), 0), 15);
  a.zeros[gid] = (uint8_t)z;
  uint32_t* out = reinterpret_cast<uint32_t*>(a.qweight) + (row * a.k + gi * (int64_t)G) / 8;
  for (int j8 = 0; j8 < G; j8 += 8) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int q = 0;
      if (s != 0.0f) q = min(max((int)rintf(__fdiv_rn(load_w(w, j8 + j), s)) + z, 0), 15);
      word |= (uint32_t)q << (4 * nibble_pos(j));
    }
    out[j8 / 8] = word;
  }
}

template <typename WT>
__global__ void __launch_bounds__(128) quantize_kernel(const QuantizeArgs a) {
  const int64_t ngroups = a.k / a.group_eff;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= a.n * ngroups) return;
  const int64_t row = gid / ngroups;
  const int64_t gi = gid - row * ngroups;
  const int G = a.group_eff;
  const WT* w = reinterpret_cast<const WT*>(a.w) + row * a.k + gi * (int64_t)G;
  if (a.format == WQL_FMT_E4M3) {
    quantize_e4m3_row(a, w, gid);
    return;
  }
  if (a.format == WQL_FMT_ASYM) {
    quantize_asym_group(a, w, row, gi, gid);
    return;
  }
  const int qmax = a.bits == 4 ? 7 : 127;
  const int qmin = a.bits == 4 ? -8 : -127;

  float amax = 0.0f;
  for (int j = 0; j < G; ++j) amax = fmaxf(amax, fabsf(load_w(w, j)));

  int best = 0;
  if (a.nratios > 1) {
    double best_err = 0.0;
    for (int ri = 0; ri < a.nratios; ++ri) {
      float prod = __fmul_rn(amax, a.ratio_c[ri]);
      prod = prod < 1e-8f ? 1e-8f : prod;
      const float s = scale_to_f32(round_scale(prod, a.scale_dtype), a.scale_dtype);
      double err = 0.0;
      for (int j = 0; j < G; ++j) {
        const float wv = load_w(w, j);
        const int q = code_of(wv, s, qmin, qmax);
        const double d = __dsub_rn(__dmul_rn((double)q, (double)s), (double)wv);
        err = __dadd_rn(err, __dmul_rn(d, d));
      }
      if (ri == 0 || err < best_err) {
        best_err = err;
        best = ri;
      }
    }
  }
  float prod = __fmul_rn(amax, a.ratio_c[best]);
  prod = prod < 1e-8f ? 1e-8f : prod;
  const uint16_t sbits = round_scale(prod, a.scale_dtype);
  const float s = scale_to_f32(sbits, a.scale_dtype);
  a.scales[gid] = sbits;

  if (a.bits == 4) {
    uint32_t* out = reinterpret_cast<uint32_t*>(a.qweight) + (row * a.k + gi * (int64_t)G) / 8;
    for (int j8 = 0; j8 < G; j8 += 8) {
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int q = code_of(load_w(w, j8 + j), s, qmin, qmax);
        word |= (uint32_t)(q + 8) << (4 * nibble_pos(j));
      }
      out[j8 / 8] = word;
    }
  } else {
    uint32_t* out = reinterpret_cast<uint32_t*>(
        reinterpret_cast<int8_t*>(a.qweight) + row * a.k + gi * (int64_t)G);
    for (int j4 = 0; j4 < G; j4 += 4) {
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = code_of(load_w(w, j4 + j), s, qmin, qmax);
        word |= ((uint32_t)q & 0xFFu) << (8 * j);
      }
      out[j4 / 4] = word;
    }
  }
}

__global__ void pack_kernel(const uint8_t* nib, int64_t words, uint32_t* out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= words) return;
  const uint2 v = *reinterpret_cast<const uint2*>(nib + 8 * i);
  uint32_t word = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t b = ((j < 4 ? v.x : v.y) >> (8 * (j & 3))) & 15u;
    word |= b << (4 * nibble_pos(j));
  }
  out[i] = word;
}

__global__ void unpack_kernel(const uint32_t* packed, int64_t words, uint8_t* out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= words) return;
  const uint32_t w = packed[i];
  uint2 v = make_uint2(0u, 0u);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t b = (w >> (4 * nibble_pos(j))) & 15u;
    if (j < 4) v.x |= b << (8 * j); else v.y |= b << (8 * (j - 4));
  }
  *reinterpret_cast<uint2*>(out + 8 * i) = v;
}

}  // namespace

cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t s) {
  const int64_t groups = a.n * (a.k / a.group_eff);
  const int threads = 128;
  const int64_t blocks = (groups + threads - 1) / threads;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  switch (a.w_dtype) {
    case WQL_F32: quantize_kernel<float><<<(unsigned)blocks, threads, 0, s>>>(a); break;
    case WQL_F16: quantize_kernel<__half><<<(unsigned)blocks, threads, 0, s>>>(a); break;
    default: quantize_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, s>>>(a); break;
  }
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t* nib, int64_t n, int64_t k, uint32_t* out, cudaStream_t s) {
  const int64_t words = n * (k / 8);
  const int64_t blocks = (words + 255) / 256;
  pack_kernel<<<(unsigned)blocks, 256, 0, s>>>(nib, words, out);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* packed, int64_t n, int64_t k, uint8_t* out,
                          cudaStream_t s) {
  const int64_t words = n * (k / 8);
  const int64_t blocks = (words + 255) / 256;
  unpack_kernel<<<(unsigned)blocks, 256, 0, s>>>(packed, words, out);
  note_launch();
  return cudaGetLastError();
}

}  // namespace wql
