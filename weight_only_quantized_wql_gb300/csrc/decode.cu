// decode.cu -- launch planning for the small-token-count logits kernel
// (decode_impl.cuh): shared-memory layout, variant choice and grid size.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_impl.cuh"

namespace wql {
namespace {

using decode_detail::kMaxTok;
using decode_detail::kPD;
using decode_detail::round_up_u32;
using decode_detail::warps_of;

constexpr size_t kSmemLimit = 227 * 1024;

struct Plan {
  bool gw2;          // int4 whose 128-column steps span two scale groups
  int nt;            // 8-column MMA n-tiles
  int warps;         // warps per CTA
  int cap;           // candidate buffer entries per (warp, token)
  int step_cols, s_real, s, corr_pitch, corr_floats, nunits, xsum_off;
  uint32_t xpitch;
  uint32_t off_x, off_zero, off_corr, off_ring, off_list, off_cnt, off_misc, off_ugrp;
  size_t smem;
};

// Shared memory of one launch with m token rows: x resident (m rows of
// xpitch bytes), the zero region, offset sums, the warps' weight rings
// (reused at the end for the slots of tiles cut between warps and for the
// top-K survivors), (top-K) the warps' candidate buffers, counts and
// thresholds, the small words and head stashes, and the unit -> group table.
Plan plan(int m, int k, int bits, int group, int topk, int format, int cap) {
  Plan P{};
  P.gw2 = bits == 4 && (group % 128) != 0;
  P.step_cols = bits == 4 ? 128 : 64;
  P.s_real = (k + P.step_cols - 1) / P.step_cols;
  P.s = (P.s_real + kPD - 1) / kPD * kPD;
  if (P.gw2) P.nt = m <= 4 ? 1 : m <= 8 ? 2 : 4;
  else P.nt = m <= 8 ? 1 : 2;
  P.warps = warps_of(P.nt);
  P.cap = cap;
  P.xpitch = (uint32_t)P.s_real * (uint32_t)P.step_cols * 2u;
  P.corr_pitch = 2 * P.s_real;
  P.corr_floats = P.gw2 ? kMaxTok * P.corr_pitch : P.s_real * kMaxTok;
  // zero points: the plain sums of x per step follow the offset sums
  P.xsum_off = P.corr_floats;
  if (format == WQL_FMT_ASYM) P.corr_floats *= 2;
  P.nunits = bits == 4 ? 2 * P.s_real : P.s_real;
  const bool tk = topk > 0;
  uint32_t off = 0;
  P.off_x = off;
  off += (uint32_t)m * P.xpitch;
  P.off_zero = round_up_u32(off, 128);
  off = P.off_zero + decode_detail::kZeroBytes;
  P.off_corr = round_up_u32(off, 16);
  off = P.off_corr + (uint32_t)P.corr_floats * 4u;
  P.off_ring = round_up_u32(off, 128);
  off = P.off_ring + (uint32_t)(P.warps * decode_detail::kRingBytes);
  P.off_list = round_up_u32(off, 16);
  off = P.off_list + (tk ? (uint32_t)(P.warps * m * P.cap * 8) : 0u);
  P.off_cnt = round_up_u32(off, 16);
  off = P.off_cnt + (tk ? (uint32_t)(2 * P.warps * m * 4) : 0u);
  P.off_misc = round_up_u32(off, 16);
  off = P.off_misc + 256u + (uint32_t)(P.warps * 32 * P.nt * 4 * 4);
  P.off_ugrp = round_up_u32(off, 16);
  off = P.off_ugrp + (uint32_t)P.nunits * 2u;
  P.smem = off;
  return P;
}

// Candidate buffers of 32 entries per (warp, token) (fewer compactions),
// else of K + 16 (the least the appends of one tile need after a compaction)
// when the larger ones do not fit.
Plan plan(int m, int k, int bits, int group, int topk, int format) {
  const Plan P = plan(m, k, bits, group, topk, format, 32);
  if (P.smem <= kSmemLimit || topk <= 0) return P;
  return plan(m, k, bits, group, topk, format, topk + 16);
}

}  // namespace

namespace decode_detail {
template <typename XT, typename ST>
cudaError_t dispatch_xs(const DecodeParams& p, bool gw2, bool lin, int nt, size_t smem, int ctas,
                        cudaStream_t s);
extern template cudaError_t dispatch_xs<__half, __half>(const DecodeParams&, bool, bool, int,
                                                        size_t, int, cudaStream_t);
extern template cudaError_t dispatch_xs<__half, __nv_bfloat16>(const DecodeParams&, bool, bool,
                                                               int, size_t, int, cudaStream_t);
extern template cudaError_t dispatch_xs<__nv_bfloat16, __half>(const DecodeParams&, bool, bool,
                                                               int, size_t, int, cudaStream_t);
extern template cudaError_t dispatch_xs<__nv_bfloat16, __nv_bfloat16>(const DecodeParams&, bool,
                                                                      bool, int, size_t, int,
                                                                      cudaStream_t);
}  // namespace decode_detail

size_t decode_smem_bytes(int m, int k, int bits, int group_eff, int topk, int format) {
  return plan(m, k, bits, group_eff, topk, format).smem;
}

int decode_max_tokens(int k, int bits, int group_eff, int topk, int format) {
  for (int m = kMaxTok; m >= 1; --m)
    if (plan(m, k, bits, group_eff, topk, format).smem <= kSmemLimit) return m;
  return 0;
}

cudaError_t launch_decode(const LogitsArgs& a, unsigned int* err, cudaStream_t s) {
  (void)err;   // the decode kernel has no waits that can time out
  if (a.m < 1 || a.m > kMaxTok) return cudaErrorInvalidConfiguration;
  const Plan P = plan(a.m, a.k, a.bits, a.group_eff, a.topk, a.format);
  if (a.format == WQL_FMT_ASYM && (P.gw2 || a.zeros == nullptr))
    return cudaErrorInvalidConfiguration;
  if (P.smem > kSmemLimit) return cudaErrorInvalidConfiguration;
  if (a.topk > 0 && (a.counter == nullptr || a.cand == nullptr))
    return cudaErrorInvalidConfiguration;
  decode_detail::DecodeParams p{};
  p.a = a;
  p.tiles = (a.n + 15) / 16;
  p.S = P.s;
  p.S_real = P.s_real;
  p.group = a.group_eff;
  p.ngroups = a.k / a.group_eff;
  p.nunits = P.nunits;
  p.off_ugrp = P.off_ugrp;
  p.row_bytes = a.k * a.bits / 8;
  p.corr_pitch = P.corr_pitch;
  p.xpitch = P.xpitch;
  p.off_x = P.off_x;
  p.off_zero = P.off_zero;
  p.off_corr = P.off_corr;
  p.off_ring = P.off_ring;
  p.off_list = P.off_list;
  p.off_cnt = P.off_cnt;
  p.off_misc = P.off_misc;
  p.cap = P.cap;
  p.xsum_off = P.xsum_off;
  p.corr_floats = P.corr_floats;
  // linear scale addressing: with two group halves per step, groups of 64
  // columns, no half step at a row's end and 4-byte aligned scale rows (one
  // 32-bit load per row); otherwise one group per step
  const bool lin = P.gw2 ? (a.group_eff == 64 && a.k % 128 == 0 &&
                            reinterpret_cast<uintptr_t>(a.scales) % 4 == 0)
                         : a.group_eff == P.step_cols;
  p.early_weights = a.weights_static ? 1 : 0;
  int ctas = device_sm_count();
  if (ctas > WQL_MAX_CTAS) ctas = WQL_MAX_CTAS;
  if (ctas > p.tiles) ctas = p.tiles;
  p.tpc = p.tiles / ctas;
  p.tex = p.tiles - p.tpc * ctas;
  p.rpt = P.s / kPD;
  const bool xh = a.x_dtype == WQL_F16, sh = a.scale_dtype == WQL_F16;
  using decode_detail::dispatch_xs;
  if (xh && sh) return dispatch_xs<__half, __half>(p, P.gw2, lin, P.nt, P.smem, ctas, s);
  if (xh) return dispatch_xs<__half, __nv_bfloat16>(p, P.gw2, lin, P.nt, P.smem, ctas, s);
  if (sh) return dispatch_xs<__nv_bfloat16, __half>(p, P.gw2, lin, P.nt, P.smem, ctas, s);
  return dispatch_xs<__nv_bfloat16, __nv_bfloat16>(p, P.gw2, lin, P.nt, P.smem, ctas, s);
}

}  // namespace wql
