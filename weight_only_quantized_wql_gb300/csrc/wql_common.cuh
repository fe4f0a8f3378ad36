// wql_common.cuh -- device helpers and internal launcher declarations shared
// by the libwql CUDA sources (sm_103a).  Nothing here is part of the C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wql.h"

namespace wql {

// ---------------------------------------------------------------------------
// Host-side bookkeeping
// ---------------------------------------------------------------------------
void note_launch();                 // one kernel launched through the library
int device_sm_count();              // SMs of the current device (cached)
wql_status record_cuda_error(cudaError_t e);  // keep the text for wql_last_error()

// Packed int4 layout: element 8i + j of a row is the nibble at position
// nibble_pos(j) of word i -- even elements in bits 0..15, odd in 16..31 -- so
// that masking one nibble per 16-bit half yields the adjacent pair (j, j+1).
__host__ __device__ constexpr int nibble_pos(int j) { return 4 * (j % 2) + j / 2; }

// ---------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Scale table entries are raw 16-bit patterns; `sdt` says how to read them.
__device__ __forceinline__ float scale_to_f32(uint16_t bits, int sdt) {
  return sdt == WQL_F16 ? __half2float(__ushort_as_half(bits))
                        : __bfloat162float(__ushort_as_bfloat16(bits));
}

__device__ __forceinline__ uint16_t ldg_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ldg_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ldg_stream_u2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Integer code -> 16-bit float pairs without int->float converts.
//
// A 16-bit float whose exponent field says [1024, 2048) (fp16, pattern 0x64xx)
// or [128, 256) (bf16, pattern 0x43xx) has unit spacing, so OR-ing a small
// unsigned integer u into its low mantissa bits yields exactly 1024 + u (or
// 128 + u); one packed subtract then gives the signed code exactly.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t d;
  // (a & b) | c  ->  lookup table 0xEA
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One packed 32-bit word (element j at nibble_pos(j)) -> four packed pairs of
// exact codes q = nibble - 8 in natural order:
//   out[p] = (q[2p], q[2p + 1]) for p = 0..3  (low half = first element).
template <typename XT> struct Int4Dequant;

template <> struct Int4Dequant<__half> {
  static __device__ __forceinline__ void run(uint32_t w, uint32_t out[4]) {
    const uint32_t kMagic = 0x64006400u;      // (1024, 1024)
    const uint32_t kSub = 0x64086408u;        // (1032, 1032)
    const uint32_t kOneSixteenth = 0x2C002C00u; // (1/16, 1/16)
    const uint32_t kNeg72 = 0xD480D480u;      // (-72, -72)
    uint32_t hi = w >> 8;
    // nibbles in bits 0..3 of each half: 1024 + u; in bits 4..7: 1024 + 16u,
    // which x/16 - 72 turns into u - 8.
    out[0] = hsub2_u32(lop3_and_or(w, 0x000F000Fu, kMagic), kSub);
    out[1] = hfma2_u32(lop3_and_or(w, 0x00F000F0u, kMagic), kOneSixteenth, kNeg72);
    out[2] = hsub2_u32(lop3_and_or(hi, 0x000F000Fu, kMagic), kSub);
    out[3] = hfma2_u32(lop3_and_or(hi, 0x00F000F0u, kMagic), kOneSixteenth, kNeg72);
  }
};

template <> struct Int4Dequant<__nv_bfloat16> {
  static __device__ __forceinline__ void run(uint32_t w, uint32_t out[4]) {
    const uint32_t kMagic = 0x43004300u;      // (128, 128)
    const uint32_t kOne = 0x3F803F80u;        // (1, 1)
    const uint32_t kNeg136 = 0xC308C308u;     // (-136, -136)
    out[0] = bfma2_u32(lop3_and_or(w, 0x000F000Fu, kMagic), kOne, kNeg136);
    out[1] = bfma2_u32(lop3_and_or(w >> 4, 0x000F000Fu, kMagic), kOne, kNeg136);
    out[2] = bfma2_u32(lop3_and_or(w >> 8, 0x000F000Fu, kMagic), kOne, kNeg136);
    out[3] = bfma2_u32(lop3_and_or(w >> 12, 0x000F000Fu, kMagic), kOne, kNeg136);
  }
};

// One 32-bit word of four int8 codes (element j in byte j) -> two packed
// pairs in natural order: out[0] = (q0, q1), out[1] = (q2, q3).
template <typename XT> struct Int8Dequant;

template <> struct Int8Dequant<__half> {
  static __device__ __forceinline__ void run(uint32_t w, uint32_t out[2]) {
    const uint32_t b = w ^ 0x80808080u;       // byte = q + 128 in [1, 255]
    const uint32_t kSub = 0x64806480u;        // (1152, 1152) = 1024 + 128
    out[0] = hsub2_u32(prmt(b, 0x64646464u, 0x4140u), kSub);
    out[1] = hsub2_u32(prmt(b, 0x64646464u, 0x4342u), kSub);
  }
};

template <> struct Int8Dequant<__nv_bfloat16> {
  // bf16 has no unit-spaced binade wide enough for 8-bit codes: go through
  // the fp32 pattern 0x4B0000xx = 2^23 + byte, then pack (exact for |q|<=127).
  static __device__ __forceinline__ void run(uint32_t w, uint32_t out[2]) {
    const uint32_t b = w ^ 0x80808080u;
    const float kOff = 8388736.0f;            // 2^23 + 128
    float f0 = __uint_as_float(prmt(b, 0x4B000000u, 0x7440u)) - kOff;
    float f1 = __uint_as_float(prmt(b, 0x4B000000u, 0x7441u)) - kOff;
    float f2 = __uint_as_float(prmt(b, 0x4B000000u, 0x7442u)) - kOff;
    float f3 = __uint_as_float(prmt(b, 0x4B000000u, 0x7443u)) - kOff;
    __nv_bfloat162 p0 = __floats2bfloat162_rn(f0, f1);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(f2, f3);
    out[0] = *reinterpret_cast<uint32_t*>(&p0);
    out[1] = *reinterpret_cast<uint32_t*>(&p1);
  }
};

// ---------------------------------------------------------------------------
// Offset codes for the decode path: the same magic-number trick without the
// packed subtract.  Each 16-bit value is exactly kMagic + u (u the unsigned
// code), so an MMA with activations x accumulates sum x*(q + kOffset) and the
// caller subtracts kOffset * sum(x) once per scale group.  Products are exact
// (<= 11 x 11 significant bits); the subtraction happens in fp32.
// kOffset == 0 marks a variant that already yields exact q.
// ---------------------------------------------------------------------------
template <int BITS, typename XT> struct OffsetCodes;

template <> struct OffsetCodes<4, __half> {   // 1024 + u, u = q + 8
  static constexpr float kOffset = 1032.0f;
  static constexpr int kPairs = 4;
  static __device__ __forceinline__ void run(uint32_t w, uint32_t (&out)[4]) {
    const uint32_t m = 0x64006400u;
    out[0] = lop3_and_or(w, 0x000F000Fu, m);
    out[1] = lop3_and_or(w >> 4, 0x000F000Fu, m);
    out[2] = lop3_and_or(w >> 8, 0x000F000Fu, m);
    out[3] = lop3_and_or(w >> 12, 0x000F000Fu, m);
  }
};

template <> struct OffsetCodes<4, __nv_bfloat16> {   // 128 + u, u = q + 8
  static constexpr float kOffset = 136.0f;
  static constexpr int kPairs = 4;
  static __device__ __forceinline__ void run(uint32_t w, uint32_t (&out)[4]) {
    const uint32_t m = 0x43004300u;
    out[0] = lop3_and_or(w, 0x000F000Fu, m);
    out[1] = lop3_and_or(w >> 4, 0x000F000Fu, m);
    out[2] = lop3_and_or(w >> 8, 0x000F000Fu, m);
    out[3] = lop3_and_or(w >> 12, 0x000F000Fu, m);
  }
};

template <> struct OffsetCodes<8, __half> {   // 1024 + b, b = q + 128
  static constexpr float kOffset = 1152.0f;
  static constexpr int kPairs = 2;
  static __device__ __forceinline__ void run(uint32_t w, uint32_t (&out)[2]) {
    const uint32_t b = w ^ 0x80808080u;
    out[0] = prmt(b, 0x64646464u, 0x4140u);
    out[1] = prmt(b, 0x64646464u, 0x4342u);
  }
};

template <> struct OffsetCodes<8, __nv_bfloat16> {   // exact q (no offset)
  static constexpr float kOffset = 0.0f;
  static constexpr int kPairs = 2;
  static __device__ __forceinline__ void run(uint32_t w, uint32_t (&out)[2]) {
    Int8Dequant<__nv_bfloat16>::run(w, out);
  }
};

// fp8 e4m3 codes (four per word, element j in byte j) -> two packed pairs in
// natural order, exact: every e4m3 value is an fp16 normal or zero (the
// subnormals m * 2^-9 included) and fits bf16's 8-bit mantissa too.
template <typename XT> struct E4M3Codes;
template <> struct E4M3Codes<__half> {
  static constexpr float kOffset = 0.0f;
  static constexpr int kPairs = 2;
  static __device__ __forceinline__ void run(uint32_t w, uint32_t (&out)[2]) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    out[0] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
    out[1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
  }
};
template <> struct E4M3Codes<__nv_bfloat16> {
  static constexpr float kOffset = 0.0f;
  static constexpr int kPairs = 2;
  static __device__ __forceinline__ void run(uint32_t w, uint32_t (&out)[2]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw r =
          __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w >> (16 * h)) & 0xFFFFu), __NV_E4M3);
      const __nv_bfloat162 b = __floats2bfloat162_rn(__half2float(__ushort_as_half(r.x)),
                                                     __half2float(__ushort_as_half(r.y)));
      out[h] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
};

// fp16 int4 with activations pre-scaled by 1/16 at the elements held in
// nibbles 1 and 3 of each half-word (elements 2, 3, 6, 7 of a word): those
// nibbles stay where they are and read as 1024 + 16u, so only one shift per
// word is needed.  With x' = x/16 there, x'*(1024 + 16u) = 16x'*(q + 72), so
// the per-group offset is 1032*sum(x) over the other elements plus
// 1152*sum(x') over these.
struct Int4F16Scaled {
  static constexpr float kOffset = 1032.0f;   // of elements 0, 1, 4, 5
  static __device__ __forceinline__ void run(uint32_t w, uint32_t (&out)[4]) {
    const uint32_t m = 0x64006400u;
    const uint32_t hi = w >> 8;
    out[0] = lop3_and_or(w, 0x000F000Fu, m);    // elements 0, 1: 1024 + u
    out[1] = lop3_and_or(w, 0x00F000F0u, m);    // elements 2, 3: 1024 + 16u
    out[2] = lop3_and_or(hi, 0x000F000Fu, m);   // elements 4, 5
    out[3] = lop3_and_or(hi, 0x00F000F0u, m);   // elements 6, 7
  }
};

template <typename ST>
__device__ __forceinline__ float scale_bits_to_f32(uint16_t bits);
template <>
__device__ __forceinline__ float scale_bits_to_f32<__half>(uint16_t bits) {
  return __half2float(__ushort_as_half(bits));
}
template <>
__device__ __forceinline__ float scale_bits_to_f32<__nv_bfloat16>(uint16_t bits) {
  return __uint_as_float((uint32_t)bits << 16);
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core MMA (m16n8k16, fp32 accumulate)
// ---------------------------------------------------------------------------
template <typename XT> struct Mma16816;

template <> struct Mma16816<__half> {
  static __device__ __forceinline__ void run(float d[4], const uint32_t a[4], uint32_t b0,
                                             uint32_t b1, const float c[4]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]),
          "f"(c[1]), "f"(c[2]), "f"(c[3]));
  }
};

template <> struct Mma16816<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float d[4], const uint32_t a[4], uint32_t b0,
                                             uint32_t b1, const float c[4]) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]),
          "f"(c[1]), "f"(c[2]), "f"(c[3]));
  }
};

// ---------------------------------------------------------------------------
// Top-K keys: one 64-bit integer per (value, index) so that a larger key
// ranks higher -- value descending, then index ascending.  -0 counts as +0
// and NaN ranks below everything.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long topk_key(float v, uint32_t idx) {
  uint32_t o;
  if (v != v) {
    o = 0u;
  } else {
    uint32_t b = __float_as_uint(v + 0.0f);
    o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ float key_value(unsigned long long key) {
  uint32_t o = (uint32_t)(key >> 32);
  uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}
__device__ __forceinline__ int32_t key_index(unsigned long long key) {
  return (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}
constexpr unsigned long long kEmptyKey = 0ull;   // ranks below every real entry

// Insert `key` into a descending register list of K entries (static indexing).
template <int K>
__device__ __forceinline__ void list_insert(unsigned long long (&list)[K], unsigned long long key) {
  if (key <= list[K - 1]) return;
#pragma unroll
  for (int i = K - 1; i > 0; --i) {
    unsigned long long prev = list[i - 1];
    bool shift = key > prev;
    list[i] = shift ? prev : (key > list[i] ? key : list[i]);
  }
  if (key > list[0]) list[0] = key;
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
  uint32_t lo = (uint32_t)v, hi = (uint32_t)(v >> 32);
  lo = __shfl_xor_sync(0xFFFFFFFFu, lo, m);
  hi = __shfl_xor_sync(0xFFFFFFFFu, hi, m);
  return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    unsigned long long o = shfl_xor_u64(v, m);
    v = o > v ? o : v;
  }
  return v;
}

// Merge the 32 lanes' descending lists into the warp's top `kk` keys (kk <=
// K), returned in descending order in `out` on every lane.  Keys are unique.
template <int K>
__device__ __forceinline__ void warp_merge_topk(unsigned long long (&list)[K], int kk,
                                                unsigned long long (&out)[K]) {
#pragma unroll
  for (int r = 0; r < K; ++r) {
    if (r < kk) {
      unsigned long long best = warp_max_u64(list[0]);
      out[r] = best;
      if (list[0] == best && best != kEmptyKey) {
#pragma unroll
        for (int i = 0; i < K - 1; ++i) list[i] = list[i + 1];
        list[K - 1] = kEmptyKey;
      }
    } else {
      out[r] = kEmptyKey;
    }
  }
}

__device__ __forceinline__ uint32_t redux_max_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// Same contract as warp_merge_topk, with each round's warp maximum taken by two
// hardware reductions (value half, then index half among the tied lanes).
template <int K>
__device__ __forceinline__ void warp_merge_topk_redux(unsigned long long (&list)[K], int kk,
                                                      unsigned long long (&out)[K]) {
#pragma unroll
  for (int r = 0; r < K; ++r) {
    if (r < kk) {
      const uint32_t hi = (uint32_t)(list[0] >> 32), lo = (uint32_t)list[0];
      const uint32_t mhi = redux_max_u32(hi);
      const uint32_t mlo = redux_max_u32(hi == mhi ? lo : 0u);
      const unsigned long long best = ((unsigned long long)mhi << 32) | mlo;
      out[r] = best;
      if (list[0] == best && best != kEmptyKey) {
#pragma unroll
        for (int i = 0; i < K - 1; ++i) list[i] = list[i + 1];
        list[K - 1] = kEmptyKey;
      }
    } else {
      out[r] = kEmptyKey;
    }
  }
}

// best[lane] without dynamic register indexing (which would go to local memory)
template <int K>
__device__ __forceinline__ unsigned long long pick(const unsigned long long (&v)[K], int i) {
  unsigned long long r = kEmptyKey;
#pragma unroll
  for (int j = 0; j < K; ++j) r = (j == i) ? v[j] : r;
  return r;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: the kernels of the logits path (decode,
// tensor-core, top-K selection, rescoring) are launched so that each may
// start while the preceding kernel on the stream finishes; each reads
// nothing another kernel may write (its inputs, the workspace) and writes
// nothing before griddep_wait(), which returns once the preceding kernel has
// completed and its writes are visible (the decode kernel's early weight
// copies under WQL_WEIGHT_STATIC are the one documented exception).
// griddep_launch_dependents() lets the following kernel launch early.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---------------------------------------------------------------------------
// Internal launchers
// ---------------------------------------------------------------------------
struct QuantizeArgs {
  const void* w;
  int w_dtype;
  int64_t n, k;
  int bits, group_eff, scale_dtype, nratios;
  float ratio_c[5];          // fl32(r / qmax), computed on the host in binary64
  void* qweight;
  uint16_t* scales;
  int format;                // wql_format
  uint8_t* zeros;            // WQL_FMT_ASYM: [n, k / group_eff]
};
cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t s);
cudaError_t launch_pack(const uint8_t* nib, int64_t n, int64_t k, uint32_t* out, cudaStream_t s);
cudaError_t launch_unpack(const uint32_t* packed, int64_t n, int64_t k, uint8_t* out,
                          cudaStream_t s);

struct LogitsArgs {
  const void* x;
  int x_dtype;
  int m;                      // token rows in this launch
  const void* qweight;
  const uint16_t* scales;
  int bits, group_eff, scale_dtype;
  int n, k;
  const void* bias;
  void* logits;
  int topk;
  int32_t* topk_idx;
  float* topk_val;
  unsigned int* counter;      // zero between calls; the last CTA resets it
  unsigned long long* cand;   // [m][WQL_MAX_CTAS][topk] keys
  unsigned int* tickets;      // [256] per-token tickets of the top-K selection
                              // (zero between calls)
  int weights_static;         // 1: no kernel that may precede this launch on the
                              // stream writes qweight / scales
  int format;                 // wql_format of the weight
  const uint8_t* zeros;       // WQL_FMT_ASYM: [n, k / group_eff] zero points
};
// Diagnostics (wql_debug_set_waits): the budget of the tensor-core kernel's
// in-loop waits, in SM cycles, and whether its MMA warp first stalls on a
// barrier nothing arrives on.
long long diag_wait_budget();
int diag_stall_mma();

// The code format of a weight (wql_weight.format without its flag bits).
inline int weight_format(const wql_weight* w) { return w->format & WQL_FMT_MASK; }

// Host checks shared by the logits entry points (no CUDA call): argument
// validity, the weight's format, sizes and alignment.  On WQL_OK, *g_out is
// the effective group (k for one scale per row).
wql_status check_logits_args(const void* x, int32_t x_dtype, int64_t m, const wql_weight* w,
                             const void* bias, const void* logits_out, int32_t topk,
                             const void* topk_idx, const void* topk_val, int64_t* g_out);

// Bandwidth-bound path for m <= 16 (warp MMA fed straight from global memory,
// split over vocab rows).  `err` is the workspace's sticky error word.
cudaError_t launch_decode(const LogitsArgs& a, unsigned int* err, cudaStream_t s);
size_t decode_smem_bytes(int m, int k, int bits, int group_eff, int topk, int format);
// Most token rows one decode launch takes for this shape (0: none fits).
int decode_max_tokens(int k, int bits, int group_eff, int topk, int format);
// Tensor-core path for 16 < m <= 256 (fp16 activations and scales): logits
// only (a.topk is ignored; launch_topk_select follows it).
bool tc_supported(const LogitsArgs& a);
cudaError_t launch_tc(const LogitsArgs& a, unsigned int* err, cudaStream_t s);
// Top-K of each token row from the rounded logits already written to
// a.logits, candidates recomputed in fp32 from the packed weight.
cudaError_t launch_topk_select(const LogitsArgs& a, cudaStream_t s);

struct RescoreArgs {
  const void* x;
  int x_dtype;
  int m, n, k;
  const void* w_ref;
  const void* bias;
  int topk;
  int32_t* topk_idx;
  float* topk_val;
  void* logits;
};
cudaError_t launch_rescore(const RescoreArgs& a, cudaStream_t s);

// Workspace layout shared by the launchers and wql_workspace_size().
struct WorkspaceLayout {
  size_t counter_off, tickets_off, cand_off, total;
};
WorkspaceLayout workspace_layout(int64_t m, int64_t n, int32_t topk);

}  // namespace wql
