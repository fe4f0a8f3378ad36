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
  uint32_t off_x, off_s, off_corr, off_bar, off_red, off_blk, off_vals;
  int vals_stride;
  size_t smem;
};

// vals_rows > 0: room for the fp32 logits of that many rows per token (the
// top-K input), with a row stride of 4 mod 32 words so that the epilogue's
// stores of one instruction fall in distinct banks.
Layout plan(int m, int k, int bits, int group_eff, bool allow_resident, int cap_units,
            int vals_rows) {
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
  L.off_blk = round_up_u32(off, 16);
  off = L.off_blk + (uint32_t)(kStages + cap_units) * 4u;
  if (vals_rows > 0) {
    L.vals_stride = (int)round_up_u32((uint32_t)vals_rows, 32u) + 4;
    L.off_vals = round_up_u32(off, 16);
    off = L.off_vals + (uint32_t)m * (uint32_t)L.vals_stride * 4u;
  }
  L.smem = off + 1024;   // slack for aligning the base to 1024
  return L;
}

constexpr size_t kSmemLimit = 227 * 1024;

// Preference: resident activations first (they serve the whole main loop),
// then the top-K logits in shared memory rather than a global scratch row.
Layout choose(int m, int k, int bits, int group_eff, int cap_units, int vals_rows) {
  Layout L{};
  for (int res = 1; res >= 0; --res) {
    if (vals_rows > 0) {
      L = plan(m, k, bits, group_eff, res != 0, cap_units, vals_rows);
      if (L.smem <= kSmemLimit) return L;
    }
    L = plan(m, k, bits, group_eff, res != 0, cap_units, 0);
    if (L.smem <= kSmemLimit) return L;
  }
  return L;
}

// Work split.  A unit is kBlockTiles 16-row tiles (one TMA box per chunk
// when full), halved while there are too few for about three per CTA.  CTAs take units from a counter in the workspace, so those whose
// copies stream faster take more; cap_units bounds one CTA's share (room for
// its unit list and top-K rows) and is never below an even share.
struct Split {
  int ctas, unit_tiles, units_total, cap_units;
};

Split split_work(int tiles_total, bool dynamic) {
  Split w{};
  int ctas = device_sm_count();
  if (ctas > WQL_MAX_CTAS) ctas = WQL_MAX_CTAS;
  if (ctas < 1) ctas = 1;
  // a power of two, so that a row's place in a CTA's list is a shift and mask
  int u = kBlockTiles;
  while (u > 1 && tiles_total < 3 * u * ctas) u >>= 1;
  w.unit_tiles = u;
  w.units_total = (tiles_total + u - 1) / u;
  w.ctas = ctas < w.units_total ? ctas : w.units_total;
  const int even = (w.units_total + w.ctas - 1) / w.ctas;
  w.cap_units = dynamic ? (2 * even < 64 ? 2 * even : (even > 64 ? even : 64)) : even;
  return w;
}

// the shared-memory need does not depend on the split beyond the unit list
constexpr int kPlanCapUnits = 64;

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
  return choose(m, k, bits, group_eff, kPlanCapUnits, 0).smem;
}

cudaError_t launch_decode(const LogitsArgs& a, unsigned int* err, cudaStream_t s) {
  const int tiles_total = (a.n + 15) / 16;
  const bool dynamic = a.counter != nullptr;
  const Split w = split_work(tiles_total, dynamic);
  const int ctas = w.ctas;
  // a CTA's top-K rows: at most cap_units units of unit_tiles tiles
  const int rows_cta = a.topk > 0 ? w.cap_units * w.unit_tiles * 16 : 0;
  const Layout L = choose(a.m, a.k, a.bits, a.group_eff, w.cap_units, rows_cta);
  if (L.smem > kSmemLimit || a.m > kMaxTok) return cudaErrorInvalidConfiguration;
  decode_detail::DecodeParams p{};
  p.a = a;
  p.err = err;
  p.tiles_total = tiles_total;
  p.unit_tiles = w.unit_tiles;
  p.unit_rows_log2 = 4;
  while ((16 << (p.unit_rows_log2 - 4)) < w.unit_tiles * 16) ++p.unit_rows_log2;
  p.units_total = w.units_total;
  p.cap_units = w.cap_units;
  p.sched = dynamic ? a.counter + 2 : nullptr;
  p.off_blk = L.off_blk;
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
  p.off_vals = L.off_vals;
  p.vals_stride = L.vals_stride;

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

  if (a.x_dtype == WQL_F16)
    return decode_detail::dispatch_x<__half>(tw, twb, tx, p, L.smem, ctas, s);
  return decode_detail::dispatch_x<__nv_bfloat16>(tw, twb, tx, p, L.smem, ctas, s);
}

}  // namespace wql
