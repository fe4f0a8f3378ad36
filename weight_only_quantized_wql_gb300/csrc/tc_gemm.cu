// tc_gemm.cu -- logits of a weight-only quantised lm_head for larger token
// counts (m > 16) on the 5th-generation tensor cores ("Fused WNA16 GEMM for
// tied quantized lm_head logits", Perf evals rows M = 32 and M = 256, where
// the product becomes a dense contraction).
//
// Design (sm_103a, one persistent CTA per SM, fp16 activations):
//  * Swap AB: a 128-row vocab tile is the MMA M dimension, the tokens
//    (padded to a multiple of 16, at most 256) are N; the fp32 accumulator
//    lives in tensor memory, double-buffered (2N <= 512 columns) so one
//    tile's epilogue overlaps the next tile's MMAs.
//  * Warp 0 (one lane) streams, by TMA, the packed weight in chunks of 128
//    bytes per row (256 int4 / 128 int8 codes; 128-row 128B-swizzled boxes)
//    and -- unless they stay resident for the whole launch -- the
//    activations in 64-column boxes.
//  * Warps 2..17 dequantise, as two groups of eight that fill A stages in
//    turn; a stage holds two consecutive 64-column blocks (32 KB).  Within
//    a group, thread pair (r, r+128) owns row r of the tile: per block it
//    turns 32 codes into exact fp16 q (magic-number LOP3/PRMT), multiplies
//    by the row's group scale (one fp16 rounding of q*s) and writes its
//    half of the 128B-swizzled K-major A row the tensor core reads.
//  * Warp 1 allocates tensor memory and runs the issue loop as a whole warp
//    (warp-uniform indices and descriptors); one elected lane issues
//    tcgen05.mma (kind::f16, 128 x N x 16), eight per A stage, committing to
//    mbarriers that release the A / activation buffers and hand finished
//    accumulators to the epilogue.
//  * Warps 18..21 (one per TMEM lane quarter) read the accumulator with
//    tcgen05.ld, add the bias, round to fp16, transpose each 32 x 32 block
//    through shared memory and store the logits with 16-byte stores.  Top-K
//    candidates are chosen afterwards from these logits (topk_select.cu).
//  * Every mbarrier wait is bounded; on a timeout the CTA records an error
//    in the workspace, skips the remaining work and still frees its TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm100.cuh"
#include "wql_common.cuh"

namespace wql {
namespace {

constexpr int kTileRows = 128;
constexpr int kWarps = 22;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerWarp = 0, kMmaWarp = 1, kDequantWarp0 = 2, kEpilogueWarp0 = 18;
constexpr int kDequantGroups = 2, kGroupWarps = 8;
constexpr int kDequantWarps = kDequantGroups * kGroupWarps, kEpilogueWarps = 4;
constexpr int kWChunkBytes = kTileRows * 128;     // one packed-weight chunk (16 KB)
constexpr int kABytes = kTileRows * 128;          // one 64-column fp16 A block (16 KB)
constexpr int kStageBlocks = 2;                   // A blocks per stage: 8 MMAs per handshake
constexpr int kAStageBytes = kStageBlocks * kABytes;
constexpr int kMaxWStages = 8, kMinWStages = 3;   // packed-weight ring: as deep as smem allows
constexpr int kMinAStages = 2, kMaxAStages = 3;   // A ring: 3 stages where smem allows
static_assert(kStageBlocks == kDequantGroups, "each group fills one block of every stage");
static_assert(kEpilogueWarp0 == kDequantWarp0 + kDequantWarps, "warp roles overlap");
constexpr int kStageBytes = kEpilogueWarps * 32 * 32 * 2;   // logits staging, all warps

struct TcParams {
  LogitsArgs a;
  int tiles_total;      // ceil(n / 128)
  int npad;             // tokens padded to a multiple of 16
  int kblocks;          // k / 64
  int chunks;           // packed chunks per row
  int ngroups;
  int x_resident;       // activations staged once per CTA
  int xstages;          // activation ring depth when not resident
  int acc_bufs;         // 1 or 2 accumulators in TMEM
  int wstages;          // packed-weight ring depth (kMinWStages..kMaxWStages)
  int astages;          // A ring depth (kMinAStages..kMaxAStages)
  uint32_t tmem_cols;   // power of two >= acc_bufs * npad
  uint32_t off_w, off_a, off_x, off_bar, off_s;
  uint32_t off_st;      // per-epilogue-warp logits staging (32 tokens x 32 rows fp16)
  int vec_store;        // logits rows 16-byte aligned: 16-byte stores allowed
  int sbuf_bytes;       // one tile's scale rows (128 x ngroups halves), 0 = no staging
  int scales_aligned;   // scale table 16-byte aligned
  unsigned int* err;
  long long wait_budget;  // SM cycles a wait on a ring slot or on data may take
  int diag_stall;         // diagnostics: the MMA warp first waits on a barrier
                          // nothing arrives on (the timeout path runs)
};

__host__ __device__ constexpr uint32_t rup(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// ---- tcgen05 / UMMA helpers (inline PTX) ----
// Shared-memory matrix descriptor for a K-major, 128B-swizzled operand whose
// 8-row x 128-byte atoms are stacked 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);          // start address
  d |= (uint64_t)1u << 16;                          // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset: 8 rows
  d |= (uint64_t)1u << 46;                          // descriptor version for sm_100
  d |= (uint64_t)2u << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, fp16 A/B, fp32 D, both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_f16(int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(kTileRows >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One lane of the (fully active) warp: true there, false elsewhere.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xFFFFFFFF;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0u;
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Exact fp16 codes q (pairs in natural order) times the fp16 scale pair s2.
__device__ __forceinline__ void int4_q_times_s(uint32_t w, uint32_t s2, uint32_t (&out)[4]) {
  uint32_t q[4];
  Int4Dequant<__half>::run(w, q);
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = hmul2_u32(q[i], s2);
}
__device__ __forceinline__ void int8_q_times_s(uint32_t w, uint32_t s2, uint32_t (&out)[2]) {
  uint32_t q[2];
  Int8Dequant<__half>::run(w, q);
  out[0] = hmul2_u32(q[0], s2);
  out[1] = hmul2_u32(q[1], s2);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1)
    tc_logits_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
                     const TcParams p) {
  constexpr int kBlocksPerChunk = BITS == 4 ? 4 : 2;   // 64-column blocks per packed chunk
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.off_bar);
  uint64_t* w_full = bars;
  uint64_t* w_empty = w_full + kMaxWStages;
  uint64_t* a_full = w_empty + kMaxWStages;
  uint64_t* a_empty = a_full + kMaxAStages;
  uint64_t* x_full = a_empty + kMaxAStages;
  uint64_t* x_empty = x_full + 4;
  uint64_t* acc_full = x_empty + 4;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* s_full = acc_empty + 2;        // per-tile scale rows (2 slots)
  uint64_t* s_empty = s_full + 2;
  uint64_t* stall_bar = s_empty + 2;       // never arrived on (diagnostics)
  uint64_t* drain_bar = stall_bar + 1;     // the MMA warp's last MMAs, on a timeout
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  unsigned int* flags = tmem_slot + 1;   // [0] bad

  const LogitsArgs& a = p.a;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = a.n, m = a.m;
  const int T0 = (int)(((long long)p.tiles_total * blockIdx.x) / gridDim.x);
  const int T1 = (int)(((long long)p.tiles_total * (blockIdx.x + 1)) / gridDim.x);
  const int ntiles = T1 - T0;
  const uint32_t xblock_bytes = (uint32_t)p.npad * 128u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.wstages; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], kDequantWarps);
    }
    for (int s = 0; s < p.astages; ++s) {
      mbar_init(&a_full[s], kDequantWarps);    // both groups, one block each
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&x_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], kEpilogueWarps);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kDequantWarps);
    }
    mbar_init(stall_bar, 1);
    mbar_init(drain_bar, 1);
    flags[0] = 0u;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    // tensor-memory accumulators (one warp allocates; freed by the same warp)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // barriers and tensor memory are set up; from here on the kernel reads its
  // inputs and the workspace and writes its outputs
  griddep_launch_dependents();
  griddep_wait();
  const uint32_t tmem_base = *tmem_slot;
  bool bad = false;

  if (warp == kProducerWarp) {
    // ------------------------------ TMA producers ------------------------------
    // Lane 0 streams the packed weight and the scale rows; lane 1 the
    // activations (once when resident, else through their ring), so neither
    // stream waits for the other's free slots.
    if (lane == 0) {
      prefetch_tmap(&tw);
      int ws = 0;
      uint32_t wph = 0;
      int wfills = 0, sfills = 0;
      const uint8_t* scales = reinterpret_cast<const uint8_t*>(a.scales);
      for (int t = T0; t < T1 && !bad; ++t) {
        // this tile's scale rows, when the tile is whole and the table aligned
        if (p.sbuf_bytes > 0 && p.scales_aligned && (t + 1) * kTileRows <= n) {
          const int slot = sfills & 1;
          if (sfills >= 2) bad = !mbar_wait(&s_empty[slot], (uint32_t)(((sfills - 2) >> 1) & 1), p.wait_budget);
          if (bad) break;
          const uint32_t sbytes = (uint32_t)(kTileRows * p.ngroups * 2);
          mbar_arrive_expect_tx(&s_full[slot], sbytes);
          bulk_load(sm + p.off_s + slot * p.sbuf_bytes,
                    scales + (size_t)t * kTileRows * p.ngroups * 2, sbytes, &s_full[slot]);
          ++sfills;
        }
        for (int c = 0; c < p.chunks && !bad; ++c) {
          if (wfills >= p.wstages) bad = !mbar_wait(&w_empty[ws], wph ^ 1u, p.wait_budget);
          if (bad) break;
          mbar_arrive_expect_tx(&w_full[ws], (uint32_t)kWChunkBytes);
          tma_load_2d(sm + p.off_w + ws * kWChunkBytes, &tw, c * 32, t * kTileRows, &w_full[ws]);
          ++wfills;
          if (++ws == p.wstages) { ws = 0; wph ^= 1u; }
        }
      }
      // every issued copy lands before the CTA can finish
      for (int s = 0; s < 2 && s < sfills; ++s)
        if (!mbar_wait(&s_full[s], (uint32_t)(((sfills - 1 - s) >> 1) & 1))) bad = true;
      for (int s = 0; s < p.wstages && s < wfills; ++s)
        if (!mbar_wait(&w_full[s], (uint32_t)(((wfills - 1 - s) / p.wstages) & 1))) bad = true;
    } else if (lane == 1 && ntiles > 0) {
      prefetch_tmap(&tx);
      if (p.x_resident) {
        // all activation blocks once, on x_full[0]; a box always moves npad
        // rows (rows >= m are zero-filled and counted)
        mbar_arrive_expect_tx(&x_full[0], (uint32_t)p.kblocks * xblock_bytes);
        for (int kb = 0; kb < p.kblocks; ++kb)
          tma_load_2d(sm + p.off_x + kb * xblock_bytes, &tx, kb * 64, 0, &x_full[0]);
        if (!mbar_wait(&x_full[0], 0u)) bad = true;
      } else {
        int xs = 0, xfills = 0;
        uint32_t xph = 0;
        for (int t = T0; t < T1 && !bad; ++t)
          for (int kb = 0; kb < p.kblocks && !bad; ++kb) {
            if (xfills >= p.xstages) bad = !mbar_wait(&x_empty[xs], xph ^ 1u, p.wait_budget);
            if (bad) break;
            mbar_arrive_expect_tx(&x_full[xs], xblock_bytes);
            tma_load_2d(sm + p.off_x + xs * xblock_bytes, &tx, kb * 64, 0, &x_full[xs]);
            ++xfills;
            if (++xs == p.xstages) { xs = 0; xph ^= 1u; }
          }
        for (int s = 0; s < p.xstages && s < xfills; ++s)
          if (!mbar_wait(&x_full[s], (uint32_t)(((xfills - 1 - s) / p.xstages) & 1))) bad = true;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer ------------------------------
    // The whole warp runs the issue loop, so stage indices and operand
    // descriptors are warp-uniform values; one elected lane issues the
    // tcgen05 instructions (single-thread instructions) and their commits.
    // One A-stage handshake covers kStageBlocks blocks (8 MMAs), which
    // halves the waits per MMA: this one warp's loop sets the pace when the
    // MMAs themselves are short.  The descriptors are built once and advanced
    // by additions (the start-address field counts 16-byte units; every
    // operand lies below 256 KB, so the field never carries).
    const bool leader = elect_one();
    const uint32_t idesc = idesc_f16(p.npad);
    const uint64_t adesc0 = smem_desc_sw128(base + p.off_a);
    const uint64_t xdesc0 = smem_desc_sw128(base + p.off_x);
    const uint64_t xstep = (uint64_t)(xblock_bytes >> 4);
    constexpr uint64_t kAStep = (uint64_t)(kABytes >> 4);
    constexpr uint64_t kKStep = 32u >> 4;          // 16 fp16 columns of a K-major row
    int as = 0, xs = 0, acc = 0;
    uint32_t aph = 0, xph = 0, accph = 0;
    int tiles_done = 0;
    bool issued = false;
    if (p.diag_stall) bad = !mbar_wait(stall_bar, 0u, p.wait_budget);
    if (p.x_resident && T0 < T1 && !bad) bad = !mbar_wait(&x_full[0], 0u, p.wait_budget);
    for (int t = T0; t < T1; ++t, ++tiles_done) {
      // wait for the epilogue to have drained this accumulator buffer
      if (!bad && tiles_done >= p.acc_bufs) bad = !mbar_wait(&acc_empty[acc], accph ^ 1u, p.wait_budget);
      if (__any_sync(0xFFFFFFFFu, bad)) { bad = true; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.npad);
      for (int kb0 = 0; kb0 < p.kblocks; kb0 += kStageBlocks) {
        bad = !mbar_wait(&a_full[as], aph, p.wait_budget);
        if (__any_sync(0xFFFFFFFFu, bad)) { bad = true; break; }
        tc_fence_after();
        const int nb = min(kStageBlocks, p.kblocks - kb0);
        const uint64_t ad0 = adesc0 + (uint64_t)as * (kStageBlocks * kAStep);
        for (int sb = 0; sb < nb; ++sb) {
          const int kb = kb0 + sb;
          if (!p.x_resident) {
            bad = !mbar_wait(&x_full[xs], xph, p.wait_budget);
            if (__any_sync(0xFFFFFFFFu, bad)) { bad = true; break; }
            tc_fence_after();
          }
          const uint64_t ad = ad0 + (uint64_t)sb * kAStep;
          const uint64_t xd = xdesc0 + (uint64_t)(p.x_resident ? kb : xs) * xstep;
          if (leader) {
            umma_f16(d_tmem, ad, xd, idesc, kb > 0 ? 1u : 0u);
            umma_f16(d_tmem, ad + kKStep, xd + kKStep, idesc, 1u);
            umma_f16(d_tmem, ad + 2 * kKStep, xd + 2 * kKStep, idesc, 1u);
            umma_f16(d_tmem, ad + 3 * kKStep, xd + 3 * kKStep, idesc, 1u);
            if (!p.x_resident) umma_commit(&x_empty[xs]);   // activation block consumed
          }
          issued = true;
          __syncwarp();
          if (!p.x_resident && ++xs == p.xstages) { xs = 0; xph ^= 1u; }
        }
        if (bad) break;
        if (leader) umma_commit(&a_empty[as]);  // A stage consumed
        __syncwarp();
        if (++as == p.astages) { as = 0; aph ^= 1u; }
      }
      if (bad) break;
      if (leader) umma_commit(&acc_full[acc]);  // accumulator ready for the epilogue
      __syncwarp();
      if (++acc == p.acc_bufs) { acc = 0; accph ^= 1u; }
    }
    if (bad && issued) {
      // after a timeout: the MMAs already issued finish before TMEM is freed
      if (leader) umma_commit(drain_bar);
      __syncwarp();
      mbar_wait(drain_bar, 0u);
    }
  } else if (warp < kEpilogueWarp0) {
    // ------------------------------ dequantisers ------------------------------
    // A stages hold kStageBlocks consecutive 64-column blocks; group g
    // fills block g of every stage, so a stage is ready after one block's
    // time.  Stages are numbered js = 0, 1, ... over the CTA's tiles and use
    // A buffer js % astages.  Each packed chunk holds whole stages; both
    // groups wait for it and release it.
    const int dq = warp - kDequantWarp0;                   // 0..15
    const int grp = dq / kGroupWarps;
    const int tdq = (dq % kGroupWarps) * 32 + lane;        // 0..255 within the group
    const int r = tdq & (kTileRows - 1);                   // row of the tile
    const int half = tdq >> 7;                             // which 32 codes of a block
    const uint32_t sw = (uint32_t)(r & 7);
    int ws = 0;
    uint32_t wph = 0;
    int sfills = 0;
    const int spt = (p.kblocks + kStageBlocks - 1) / kStageBlocks;   // stages per tile
    const int gblocks = a.group_eff / 64;                  // 64-column blocks per group
    for (int t = T0; t < T1; ++t) {
      const unsigned int js0 = (unsigned int)((t - T0) * spt);
      const int row = min(t * kTileRows + r, n - 1);
      const bool staged = p.sbuf_bytes > 0 && p.scales_aligned && (t + 1) * kTileRows <= n;
      const int slot = sfills & 1;
      const uint16_t* srow;
      if (staged) {
        if (!bad) bad = !mbar_wait(&s_full[slot], (uint32_t)((sfills >> 1) & 1), p.wait_budget);
        srow = reinterpret_cast<const uint16_t*>(sm + p.off_s + slot * p.sbuf_bytes) +
               r * p.ngroups;
      } else {
        srow = a.scales + (size_t)row * p.ngroups;
      }
      // The scale of this group's block in each of the tile's stages,
      // preloaded (stage st's in half st & 1 of sk[st >> 1]) when a row has 8
      // or 16 groups and a tile at most 8 stages: one or two 16-byte loads
      // of the row instead of a 2-byte load per block, whose 16- or 32-byte
      // row stride puts 4 or 8 rows of a warp on one shared-memory bank.
      const bool pre = spt <= 8 && (p.ngroups == 8 || p.ngroups == 16) && gblocks <= 2 &&
                       (staged || p.scales_aligned);
      uint32_t sk[4] = {0u, 0u, 0u, 0u};
      if (pre && !bad) {
        uint32_t wv[8];
        const uint4* src = reinterpret_cast<const uint4*>(srow);
        const uint4 v0 = staged ? src[0] : __ldg(src);
        const uint4 v1 = p.ngroups == 16 ? (staged ? src[1] : __ldg(src + 1)) : v0;
        wv[0] = v0.x; wv[1] = v0.y; wv[2] = v0.z; wv[3] = v0.w;
        wv[4] = v1.x; wv[5] = v1.y; wv[6] = v1.z; wv[7] = v1.w;
        if (gblocks == 2) {
          // stage st uses group st: words 0..3 as they are
          sk[0] = wv[0]; sk[1] = wv[1]; sk[2] = wv[2]; sk[3] = wv[3];
        } else {
          // stage st uses group 2 st + grp: half grp of word st, paired up
          const uint32_t sel = grp ? 0x7632u : 0x5410u;
#pragma unroll
          for (int j = 0; j < 4; ++j) sk[j] = prmt(wv[2 * j], wv[2 * j + 1], sel);
        }
      }
      int cur_chunk = -1;
      for (int st = 0; st < spt; ++st) {
        const int kb = st * kStageBlocks + grp;            // this group's block
        const bool have = kb < p.kblocks;                  // (absent in an odd tail stage)
        // the chunk holding this stage (a stage never spans two chunks)
        const int c = (st * kStageBlocks) / kBlocksPerChunk;
        if (c != cur_chunk) {
          if (cur_chunk >= 0) {
            // a warp that gave up releases nothing more: the producer then
            // times out too instead of refilling a slot whose copy may fly
            bad = __any_sync(0xFFFFFFFFu, bad);
            if (lane == 0 && !bad) mbar_arrive(&w_empty[ws]);
            if (++ws == p.wstages) { ws = 0; wph ^= 1u; }
          }
          if (!bad) bad = !mbar_wait(&w_full[ws], wph, p.wait_budget);
          cur_chunk = c;
        }
        const unsigned int js = js0 + (unsigned int)st;
        const int as = (int)(js % (unsigned int)p.astages);
        // the buffer's previous fill (astages stages back) must be consumed
        if (js >= (unsigned int)p.astages && !bad)
          bad = !mbar_wait(&a_empty[as], ((js / (unsigned int)p.astages) & 1u) ^ 1u, p.wait_budget);
        if (have && !bad) {
          const int b = kb % kBlocksPerChunk;
          const uint32_t wrow = base + p.off_w + ws * kWChunkBytes + r * 128;
          uint16_t sbits;
          if (pre) {
            const int q = st >> 1;
            const uint32_t wsel = q == 0 ? sk[0] : q == 1 ? sk[1] : q == 2 ? sk[2] : sk[3];
            sbits = (uint16_t)((st & 1) ? (wsel >> 16) : (wsel & 0xFFFFu));
          } else {
            const int gi = kb / gblocks;
            sbits = staged ? srow[gi] : ldg_u16(srow + gi);
          }
          const uint32_t s2 = (uint32_t)sbits | ((uint32_t)sbits << 16);
          const uint32_t arow = base + p.off_a + as * kAStageBytes + grp * kABytes + r * 128;
          if constexpr (BITS == 4) {
            // 16 packed bytes = 32 codes = A chunks 4*half .. 4*half+3
            const uint32_t piece = (uint32_t)(2 * b + half) ^ sw;
            const uint4 v = lds128(wrow + piece * 16);
            const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int wdi = 0; wdi < 4; ++wdi) {
              uint32_t o[4];
              int4_q_times_s(words[wdi], s2, o);
              const uint32_t chunk = (uint32_t)(4 * half + wdi) ^ sw;
              st_shared_v4(arow + chunk * 16, o[0], o[1], o[2], o[3]);
            }
          } else {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int h = 2 * half + h2;                // 16 codes per packed piece
              const uint32_t piece = (uint32_t)(4 * b + h) ^ sw;
              const uint4 v = lds128(wrow + piece * 16);
              uint32_t o0[2], o1[2], o2[2], o3[2];
              int8_q_times_s(v.x, s2, o0);
              int8_q_times_s(v.y, s2, o1);
              int8_q_times_s(v.z, s2, o2);
              int8_q_times_s(v.w, s2, o3);
              st_shared_v4(arow + (((uint32_t)(2 * h) ^ sw) * 16), o0[0], o0[1], o1[0], o1[1]);
              st_shared_v4(arow + (((uint32_t)(2 * h + 1) ^ sw) * 16), o2[0], o2[1], o3[0],
                           o3[1]);
            }
          }
          fence_async_smem();                   // generic-proxy writes -> tensor core
        }
        bad = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0 && !bad) mbar_arrive(&a_full[as]);
      }
      if (cur_chunk >= 0) {
        bad = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0 && !bad) mbar_arrive(&w_empty[ws]);
        if (++ws == p.wstages) { ws = 0; wph ^= 1u; }
      }
      if (staged) {
        bad = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0 && !bad) mbar_arrive(&s_empty[slot]);
        ++sfills;
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    uint32_t* st = reinterpret_cast<uint32_t*>(sm + p.off_st + quarter * 2048);
    const bool odd = (lane & 1) != 0;
    int acc = 0;
    uint32_t accph = 0;
    for (int t = T0; t < T1; ++t) {
      if (!bad) bad = !mbar_wait(&acc_full[acc], accph, p.wait_budget);
      bad = __any_sync(0xFFFFFFFFu, bad);
      tc_fence_after();
      const int row = t * kTileRows + r;
      const float bias = (a.bias && row < n)
                             ? __half2float(reinterpret_cast<const __half*>(a.bias)[row])
                             : 0.f;
      const uint32_t taddr =
          tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * p.npad);
      const int wrow0 = t * kTileRows + quarter * 32;   // first row of this warp
      for (int c0 = 0; c0 < p.npad && !bad; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(taddr + (uint32_t)c0, v);
        // pair adjacent rows (one shuffle per token pair), stage the warp's
        // 32 rows x 32 tokens as fp16, then write every token's 64-byte run
        // of rows with 16-byte stores
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float f0 = __uint_as_float(v[j]) + bias;
          const float f1 = __uint_as_float(v[j + 1]) + bias;
          const float recv = __shfl_xor_sync(0xFFFFFFFFu, odd ? f0 : f1, 1);
          // even lane: token j, rows (lane, lane + 1); odd: token j + 1, rows (lane - 1, lane)
          const __half2 h = odd ? __floats2half2_rn(recv, f1) : __floats2half2_rn(f0, recv);
          st[(odd ? j + 1 : j) * 16 + (lane >> 1)] = *reinterpret_cast<const uint32_t*>(&h);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int id = i * 32 + lane;
          const int tk = id >> 2, part = id & 3;
          const int tok = c0 + tk;
          const int rs = wrow0 + part * 8;
          const uint4 val = *reinterpret_cast<const uint4*>(st + tk * 16 + part * 4);
          if (tok < m) {
            __half* dst = reinterpret_cast<__half*>(a.logits) + (size_t)tok * n + rs;
            if (p.vec_store && rs + 8 <= n) {
              *reinterpret_cast<uint4*>(dst) = val;
            } else {
              const uint32_t w4[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (rs + e < n)
                  reinterpret_cast<uint16_t*>(dst)[e] = (uint16_t)(w4[e >> 1] >> (16 * (e & 1)));
            }
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !bad) mbar_arrive(&acc_empty[acc]);
      if (++acc == p.acc_bufs) { acc = 0; accph ^= 1u; }
    }
  }

  if (bad) atomicOr(&flags[0], 1u);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(p.tmem_cols)
                 : "memory");
  }
  if (flags[0] != 0u && threadIdx.x == 0 && p.err) atomicOr(p.err, 2u);
}

struct TcLayout {
  uint32_t off_w, off_a, off_x, off_bar, off_s, off_st;
  size_t smem;
  int x_resident, xstages, sbuf_bytes, wstages, astages;
};

// Shared memory: packed-weight ring, A stages, activations (resident for the
// whole launch when that still leaves a ring of kMinWStages, else a ring of
// 64-column blocks), then barriers, scale rows and the logits staging.  The
// weight ring takes what is left, up to kMaxWStages chunks: it is what keeps
// enough bytes in flight when the kernel is bound by HBM (small m).
TcLayout tc_plan_a(int npad, int k, int ngroups, int astages) {
  TcLayout L{};
  L.astages = astages;
  const uint32_t xblock = (uint32_t)npad * 128u;
  const int kblocks = k / 64;
  const uint32_t sbuf = rup((uint32_t)(kTileRows * ngroups * 2), 128u);
  L.sbuf_bytes = (2 * sbuf <= 24u * 1024u) ? (int)sbuf : 0;   // else direct scale loads
  const uint32_t tail = 512 + 128 + 2 * L.sbuf_bytes + 128 + kStageBytes + 128 + 1024;
  const uint32_t limit = 227u * 1024u;
  const uint32_t fixed = (uint32_t)astages * kAStageBytes + tail;
  const uint32_t resident = (uint32_t)kblocks * xblock;
  uint32_t xbytes;
  if (fixed + resident + kMinWStages * kWChunkBytes <= limit) {
    L.x_resident = 1;
    L.xstages = 1;
    xbytes = resident;
  } else {
    L.x_resident = 0;
    L.xstages = (fixed + 3 * xblock + kMinWStages * kWChunkBytes <= limit) ? 3 : 2;
    xbytes = L.xstages * xblock;
  }
  const uint32_t room = limit > fixed + xbytes ? limit - fixed - xbytes : 0;
  L.wstages = (int)(room / kWChunkBytes);
  if (L.wstages > kMaxWStages) L.wstages = kMaxWStages;
  uint32_t off = 0;
  L.off_w = off;
  off += (uint32_t)L.wstages * kWChunkBytes;
  L.off_a = off;
  off += (uint32_t)astages * kAStageBytes;
  L.off_x = off;
  off += xbytes;
  L.off_bar = rup(off, 64);
  off = L.off_bar + 512;
  L.off_s = rup(off, 128);
  off = L.off_s + 2 * L.sbuf_bytes;
  L.off_st = rup(off, 128);
  off = L.off_st + kStageBytes;
  L.smem = off + 1024;
  return L;
}

// Shared memory: packed-weight ring, A stages, activations (resident for the
// whole launch when that still leaves a ring of kMinWStages, else a ring of
// 64-column blocks), then barriers, scale rows and the logits staging.  The
// weight ring takes what is left, up to kMaxWStages chunks (it keeps bytes
// in flight when the kernel is bound by HBM).  A third A stage measured no
// faster than a deeper weight ring at m = 32, and does not fit at m = 256.
TcLayout tc_plan(int npad, int k, int ngroups) {
  return tc_plan_a(npad, k, ngroups, kMinAStages);
}

template <int BITS>
cudaError_t tc_launch_t(const CUtensorMap& tw, const CUtensorMap& tx, const TcParams& p,
                        size_t smem, int ctas, cudaStream_t s) {
  auto kern = tc_logits_kernel<BITS>;
  static size_t configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const cudaError_t e = launch_pdl(kern, dim3((unsigned)ctas), dim3(kThreads), smem, s, tw, tx, p);
  note_launch();
  return e;
}

}  // namespace

bool tc_supported(const LogitsArgs& a) {
  if (a.x_dtype != WQL_F16 || a.scale_dtype != WQL_F16) return false;
  if (a.m < 1 || a.m > 256 || a.k % 64 != 0) return false;
  const int npad = (a.m + 15) / 16 * 16;
  const TcLayout L = tc_plan(npad, a.k, a.k / a.group_eff);
  return L.wstages >= 2 && L.smem <= 227u * 1024u;
}

cudaError_t launch_tc(const LogitsArgs& a, unsigned int* err, cudaStream_t s) {
  if (!tc_supported(a)) return cudaErrorInvalidConfiguration;
  TcParams p{};
  p.a = a;
  p.err = err;
  p.wait_budget = diag_wait_budget();
  p.diag_stall = diag_stall_mma();
  p.tiles_total = (a.n + kTileRows - 1) / kTileRows;
  p.npad = (a.m + 15) / 16 * 16;
  p.kblocks = a.k / 64;
  const int row_bytes = a.k * a.bits / 8;
  p.chunks = (row_bytes + 127) / 128;
  p.ngroups = a.k / a.group_eff;
  p.acc_bufs = (2 * p.npad <= 512) ? 2 : 1;
  uint32_t cols = 32;
  while (cols < (uint32_t)(p.acc_bufs * p.npad)) cols <<= 1;
  p.tmem_cols = cols;
  const TcLayout L = tc_plan(p.npad, a.k, p.ngroups);
  p.sbuf_bytes = L.sbuf_bytes;
  p.off_s = L.off_s;
  p.scales_aligned = (reinterpret_cast<uintptr_t>(a.scales) % 16) == 0;
  p.x_resident = L.x_resident;
  p.xstages = L.xstages;
  p.wstages = L.wstages;
  p.astages = L.astages;
  p.off_w = L.off_w;
  p.off_a = L.off_a;
  p.off_x = L.off_x;
  p.off_bar = L.off_bar;
  p.off_st = L.off_st;
  p.vec_store = (a.n % 8 == 0) && (reinterpret_cast<uintptr_t>(a.logits) % 16 == 0);

  CUtensorMap tw, tx;
  cudaError_t e = make_tmap_2d(&tw, a.qweight, 4, (uint64_t)row_bytes / 4, (uint64_t)a.n,
                               (uint64_t)row_bytes, 32, kTileRows, Swizzle::k128B);
  if (e != cudaSuccess) return e;
  // activation boxes: 64 columns x npad rows (rows >= m read as zero)
  e = make_tmap_2d(&tx, a.x, 2, (uint64_t)a.k, (uint64_t)a.m, (uint64_t)a.k * 2, 64,
                   (uint32_t)p.npad, Swizzle::k128B);
  if (e != cudaSuccess) return e;
  int ctas = device_sm_count();
  if (ctas > p.tiles_total) ctas = p.tiles_total;
  if (ctas > WQL_MAX_CTAS) ctas = WQL_MAX_CTAS;
  return a.bits == 4 ? tc_launch_t<4>(tw, tx, p, L.smem, ctas, s)
                     : tc_launch_t<8>(tw, tx, p, L.smem, ctas, s);
}

}  // namespace wql
