// decode.cu -- launch planning for the small-token-count logits kernel
// (decode_impl.cuh): shared-memory layout, activation residency, tensor maps,
// grid size and variant dispatch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_impl.cuh"

namespace wql {
namespace {

using decode_detail::kBlockTiles;
using decode_detail::kChunkRowBytes;
using decode_detail::kMaxTok;
using decode_detail::kStageWBytes;
using decode_detail::kStages;
using decode_detail::kThreads;
using decode_detail::kWarpsAll;
using decode_detail::round_up_u32;

struct Layout {
  int chunks, ngroups, nsb, sbuf_bytes, xbox_bytes, x_resident;
  uint32_t off_x, off_s, off_corr, off_bar, off_red;
  size_t smem;
};

Layout plan(int m, int k, int bits, int group_eff, bool allow_resident) {
  Layout L{};
  const int row_bytes = k * bits / 8;
  const int units = bits == 4 ? 4 : 2;
  L.chunks = (row_bytes + kChunkRowBytes - 1) / kChunkRowBytes;
  L.ngroups = k / group_eff;
  L.sbuf_bytes = (int)round_up_u32((uint32_t)(kBlockTiles * 16 * L.ngroups * 2), 128u);
  L.nsb = 1 + (kStages - 1 + L.chunks - 1) / L.chunks;
  L.xbox_bytes = (int)round_up_u32((uint32_t)m * 128u, 1024u);
  L.x_resident = allow_resident ? 1 : 0;
  uint32_t off = kStages * kStageWBytes;
  L.off_x = off;
  off += L.x_resident ? round_up_u32((uint32_t)m * (uint32_t)k * 2u, 1024u)
                      : (uint32_t)(kStages * units * L.xbox_bytes);
  L.off_s = off;
  off += L.nsb * L.sbuf_bytes;
  L.off_corr = round_up_u32(off, 16);
  off = L.off_corr + kMaxTok * L.ngroups * 4;
  L.off_bar = round_up_u32(off, 64);
  off = L.off_bar + 2 * kStages * 8 + 16;
  L.off_red = round_up_u32(off, 64);
  off = L.off_red + kWarpsAll * WQL_MAX_TOPK * 8;
  L.smem = off + 1024;   // slack for aligning the base to 1024
  return L;
}

constexpr size_t kSmemLimit = 227 * 1024;

Layout choose(int m, int k, int bits, int group_eff) {
  Layout L = plan(m, k, bits, group_eff, true);
  if (L.smem <= kSmemLimit) return L;
  return plan(m, k, bits, group_eff, false);
}

}  // namespace

namespace decode_detail {
template <typename XT>
cudaError_t dispatch_x(const CUtensorMap& tw, const CUtensorMap& twb, const CUtensorMap& tx,
                       const DecodeParams& p, size_t smem, int ctas, cudaStream_t s);
extern template cudaError_t dispatch_x<__half>(const CUtensorMap&, const CUtensorMap&,
                                              const CUtensorMap&, const DecodeParams&, size_t,
                                              int, cudaStream_t);
extern template cudaError_t dispatch_x<__nv_bfloat16>(const CUtensorMap&, const CUtensorMap&,
                                                     const CUtensorMap&, const DecodeParams&,
                                                     size_t, int, cudaStream_t);
}  // namespace decode_detail

size_t decode_smem_bytes(int m, int k, int bits, int group_eff) {
  return choose(m, k, bits, group_eff).smem;
}

cudaError_t launch_decode(const LogitsArgs& a, unsigned int* err, cudaStream_t s) {
  const Layout L = choose(a.m, a.k, a.bits, a.group_eff);
  if (L.smem > kSmemLimit || a.m > kMaxTok) return cudaErrorInvalidConfiguration;
  decode_detail::DecodeParams p{};
  p.a = a;
  p.err = err;
  p.tiles_total = (a.n + 15) / 16;
  p.chunks = L.chunks;
  p.gunits = a.group_eff / 64;
  p.ngroups = L.ngroups;
  p.x_resident = L.x_resident;
  p.xbox_bytes = L.xbox_bytes;
  p.scales_aligned = (reinterpret_cast<uintptr_t>(a.scales) % 16) == 0;
  p.sbuf_bytes = L.sbuf_bytes;
  p.nsb = L.nsb;
  p.off_x = L.off_x;
  p.off_s = L.off_s;
  p.off_corr = L.off_corr;
  p.off_bar = L.off_bar;
  p.off_red = L.off_red;

  const int row_bytes = a.k * a.bits / 8;
  CUtensorMap tw, twb, tx;
  cudaError_t e = make_tmap_2d(&tw, a.qweight, 4, (uint64_t)row_bytes / 4, (uint64_t)a.n,
                               (uint64_t)row_bytes, kChunkRowBytes / 4, 16, Swizzle::k128B);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&twb, a.qweight, 4, (uint64_t)row_bytes / 4, (uint64_t)a.n,
                   (uint64_t)row_bytes, kChunkRowBytes / 4, kBlockTiles * 16, Swizzle::k128B);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d(&tx, a.x, 2, (uint64_t)a.k, (uint64_t)a.m, (uint64_t)a.k * 2, 64,
                   (uint32_t)a.m, Swizzle::k128B);
  if (e != cudaSuccess) return e;

  int ctas = device_sm_count();
  if (ctas > p.tiles_total) ctas = p.tiles_total;
  if (ctas > WQL_MAX_CTAS) ctas = WQL_MAX_CTAS;
  if (ctas < 1) ctas = 1;
  if (a.x_dtype == WQL_F16)
    return decode_detail::dispatch_x<__half>(tw, twb, tx, p, L.smem, ctas, s);
  return decode_detail::dispatch_x<__nv_bfloat16>(tw, twb, tx, p, L.smem, ctas, s);
}

}  // namespace wql
