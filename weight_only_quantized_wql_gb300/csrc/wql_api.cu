// wql_api.cu -- the extern "C" entry points declared in include/wql.h.
//
// Every entry point validates its arguments on the host before it touches
// the CUDA runtime, so bad arguments never launch anything and never need a
// GPU to be diagnosed.  Kernel choice by token count lives here.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <string>

#include <cudaTypedefs.h>

#include <mutex>

#include "sm100.cuh"
#include "wql_common.cuh"
#include "embed.cuh"

namespace wql {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void resolve_encoder() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t cols,
                         uint64_t rows, uint64_t row_stride_bytes, uint32_t box_cols,
                         uint32_t box_rows, Swizzle swz) {
  std::call_once(g_encode_once, resolve_encoder);
  if (!g_encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const CUresult r = g_encode(
      map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE,
      swz == Swizzle::k128B ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
std::atomic<uint64_t> g_launches{0};
thread_local std::string g_last_error;
constexpr int kDecodeMaxTokens = 16;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool half_dtype(int d) { return d == WQL_F16 || d == WQL_BF16; }

wql_status cuda_fail(cudaError_t e) {
  g_last_error = cudaGetErrorString(e);
  return WQL_ECUDA;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

wql_status record_cuda_error(cudaError_t e) { return cuda_fail(e); }

int device_sm_count() {
  static thread_local int cached_dev = -1;
  static thread_local int cached_sms = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev != cached_dev) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      sms = 1;
    cached_dev = dev;
    cached_sms = sms;
  }
  return cached_sms;
}

WorkspaceLayout workspace_layout(int64_t m, int64_t n, int32_t topk) {
  WorkspaceLayout l{};
  l.counter_off = 0;
  size_t off = 256;
  // fixed place (any m): per-token tickets of the top-K selection
  l.tickets_off = off;
  if (topk > 0) off += 256 * sizeof(unsigned int);
  l.cand_off = off;
  if (topk > 0) off += round_up((size_t)m * WQL_MAX_CTAS * (size_t)topk * 8, 256);
  (void)n;
  l.total = off;
  return l;
}

namespace {
std::atomic<long long> g_wait_budget{0};
std::atomic<int> g_stall_mma{0};
}  // namespace

long long diag_wait_budget() {
  const long long b = g_wait_budget.load(std::memory_order_relaxed);
  return b > 0 ? b : kWaitBudgetCycles;
}
int diag_stall_mma() { return g_stall_mma.load(std::memory_order_relaxed); }

wql_status check_logits_args(const void* x, int32_t x_dtype, int64_t m, const wql_weight* w,
                             const void* bias, const void* logits_out, int32_t topk,
                             const void* topk_idx, const void* topk_val, int64_t* g_out) {
  if (!w || m < 0 || w->n < 0 || w->k <= 0 || w->group < 0) return WQL_EINVAL;
  const int fmt = weight_format(w);
  if ((w->format & ~(WQL_FMT_MASK | WQL_WEIGHT_STATIC)) != 0 ||
      (fmt != WQL_FMT_SYM && fmt != WQL_FMT_E4M3 && fmt != WQL_FMT_ASYM))
    return WQL_EINVAL;
  if (topk < 0 || topk > WQL_MAX_TOPK) return WQL_EINVAL;
  const int64_t n = w->n, k = w->k;
  if (m > 0 && n > 0) {
    if (!x || !w->qweight || !w->scales) return WQL_EINVAL;
    // logits_out may be NULL only for candidates alone (top-K on)
    if (!logits_out && topk == 0) return WQL_EINVAL;
    if (topk > 0 && (!topk_idx || !topk_val)) return WQL_EINVAL;
    if (topk > n) return WQL_EINVAL;
    if (fmt == WQL_FMT_ASYM && !w->zeros) return WQL_EINVAL;
  }
  if (w->bits != 4 && w->bits != 8) return WQL_EUNSUPPORTED;
  if (fmt == WQL_FMT_E4M3 && (w->bits != 8 || w->group != 0)) return WQL_EUNSUPPORTED;
  if (fmt == WQL_FMT_ASYM && (w->bits != 4 || w->group == 0 || w->group % 128 != 0))
    return WQL_EUNSUPPORTED;
  if (!half_dtype(x_dtype) || !half_dtype(w->scale_dtype)) return WQL_EUNSUPPORTED;
  const int64_t g = w->group == 0 ? k : w->group;
  if (k % 64 != 0 || g % 64 != 0 || k % g != 0) return WQL_EUNSUPPORTED;
  if (n >= (int64_t(1) << 31) || m >= (int64_t(1) << 31) || k >= (int64_t(1) << 30))
    return WQL_EUNSUPPORTED;
  if (!aligned(x, 16) || !aligned(w->qweight, 16) || !aligned(w->scales, 2) ||
      !aligned(logits_out, 2) || !aligned(bias, 2))
    return WQL_EUNSUPPORTED;
  *g_out = g;
  return WQL_OK;
}

}  // namespace wql

using namespace wql;

extern "C" {

const char* wql_status_string(wql_status status) {
  switch (status) {
    case WQL_OK: return "WQL_OK: success";
    case WQL_EINVAL: return "WQL_EINVAL: invalid argument";
    case WQL_EUNSUPPORTED: return "WQL_EUNSUPPORTED: unsupported configuration";
    case WQL_ECUDA: return "WQL_ECUDA: CUDA error";
    case WQL_EWORKSPACE: return "WQL_EWORKSPACE: workspace missing or too small";
  }
  return "unknown wql_status";
}

const char* wql_last_error(void) { return g_last_error.c_str(); }

uint64_t wql_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

size_t wql_workspace_size(int64_t m, int64_t n, int32_t topk) {
  if (m < 0 || n < 0 || topk < 0 || topk > WQL_MAX_TOPK) return 0;
  return workspace_layout(m, n, topk).total;
}

wql_status wql_quantize(const void* w, int32_t w_dtype, int64_t n, int64_t k, int32_t bits,
                        int32_t group, int32_t scale_dtype, int32_t clip, void* qweight_out,
                        void* scales_out, cudaStream_t stream) {
  return wql_quantize_ex(w, w_dtype, n, k, WQL_FMT_SYM, bits, group, scale_dtype, clip,
                         qweight_out, scales_out, nullptr, stream);
}

wql_status wql_quantize_ex(const void* w, int32_t w_dtype, int64_t n, int64_t k, int32_t format,
                           int32_t bits, int32_t group, int32_t scale_dtype, int32_t clip,
                           void* qweight_out, void* scales_out, void* zeros_out,
                           cudaStream_t stream) {
  if (n < 0 || k <= 0 || group < 0) return WQL_EINVAL;
  if (n > 0 && (!w || !qweight_out || !scales_out)) return WQL_EINVAL;
  if (clip != WQL_CLIP_RTN && clip != WQL_CLIP_MSE) return WQL_EINVAL;
  if (format != WQL_FMT_SYM && format != WQL_FMT_E4M3 && format != WQL_FMT_ASYM)
    return WQL_EINVAL;
  if (format == WQL_FMT_ASYM && n > 0 && !zeros_out) return WQL_EINVAL;
  if (format == WQL_FMT_E4M3 && (bits != 8 || group != 0 || clip != WQL_CLIP_RTN))
    return WQL_EUNSUPPORTED;
  if (format == WQL_FMT_ASYM && (bits != 4 || group == 0 || group % 128 != 0 ||
                                 clip != WQL_CLIP_RTN))
    return WQL_EUNSUPPORTED;
  if (bits != 4 && bits != 8) return WQL_EUNSUPPORTED;
  if (w_dtype != WQL_F32 && !half_dtype(w_dtype)) return WQL_EUNSUPPORTED;
  if (!half_dtype(scale_dtype)) return WQL_EUNSUPPORTED;
  const int64_t g = group == 0 ? k : group;
  if (k % 8 != 0 || k % g != 0 || g % 8 != 0) return WQL_EUNSUPPORTED;
  if (!aligned(w, 16) || !aligned(qweight_out, 16) || !aligned(scales_out, 2))
    return WQL_EUNSUPPORTED;
  if (n == 0) return WQL_OK;
  if (g > (1 << 30)) return WQL_EUNSUPPORTED;
  QuantizeArgs a{};
  a.w = w;
  a.w_dtype = w_dtype;
  a.n = n;
  a.k = k;
  a.bits = bits;
  a.group_eff = (int)g;
  a.scale_dtype = scale_dtype;
  a.nratios = clip == WQL_CLIP_MSE ? 5 : 1;
  static const double kRatios[5] = {1.0, 0.95, 0.9, 0.85, 0.8};
  // the largest code magnitude the scale maps amax (or, asymmetric, the
  // group's range) to
  const double qmax = format == WQL_FMT_E4M3 ? 448.0 : format == WQL_FMT_ASYM ? 15.0
                      : bits == 4 ? 7.0 : 127.0;
  for (int i = 0; i < 5; ++i) a.ratio_c[i] = (float)(kRatios[i] / qmax);
  a.qweight = qweight_out;
  a.scales = static_cast<uint16_t*>(scales_out);
  a.format = format;
  a.zeros = static_cast<uint8_t*>(zeros_out);
  cudaError_t e = launch_quantize(a, stream);
  return e == cudaSuccess ? WQL_OK : cuda_fail(e);
}

wql_status wql_pack(const uint8_t* nibbles, int64_t n, int64_t k, int32_t* packed_out,
                    cudaStream_t stream) {
  if (n < 0 || k < 0) return WQL_EINVAL;
  if (n > 0 && k > 0 && (!nibbles || !packed_out)) return WQL_EINVAL;
  if (k % 8 != 0) return WQL_EUNSUPPORTED;
  if (!aligned(nibbles, 8) || !aligned(packed_out, 4)) return WQL_EUNSUPPORTED;
  if (n == 0 || k == 0) return WQL_OK;
  cudaError_t e = launch_pack(nibbles, n, k, reinterpret_cast<uint32_t*>(packed_out), stream);
  return e == cudaSuccess ? WQL_OK : cuda_fail(e);
}

wql_status wql_unpack(const int32_t* packed, int64_t n, int64_t k, uint8_t* nibbles_out,
                      cudaStream_t stream) {
  if (n < 0 || k < 0) return WQL_EINVAL;
  if (n > 0 && k > 0 && (!packed || !nibbles_out)) return WQL_EINVAL;
  if (k % 8 != 0) return WQL_EUNSUPPORTED;
  if (!aligned(packed, 4) || !aligned(nibbles_out, 8)) return WQL_EUNSUPPORTED;
  if (n == 0 || k == 0) return WQL_OK;
  cudaError_t e = launch_unpack(reinterpret_cast<const uint32_t*>(packed), n, k, nibbles_out,
                                stream);
  return e == cudaSuccess ? WQL_OK : cuda_fail(e);
}

wql_status wql_logits(const void* x, int32_t x_dtype, int64_t m, const wql_weight* w,
                      const void* bias, void* logits_out, int32_t topk, int32_t* topk_idx,
                      float* topk_val, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  int64_t g = 0;
  const wql_status st = check_logits_args(x, x_dtype, m, w, bias, logits_out, topk, topk_idx,
                                          topk_val, &g);
  if (st != WQL_OK) return st;
  const int64_t n = w->n, k = w->k;
  if (m == 0 || n == 0) return WQL_OK;
  const WorkspaceLayout lay = workspace_layout(m, n, topk);
  // top-K needs a workspace; any workspace given (top-K or not) holds the
  // kernels' counter block, so it must be large enough and aligned
  if (topk > 0 && !workspace) return WQL_EWORKSPACE;
  if (workspace && (ws_bytes < lay.total || !aligned(workspace, 256))) return WQL_EWORKSPACE;
  const int esz = 2;
  // tokens per decode launch: 16, fewer when x for 16 rows does not fit in
  // shared memory next to the rest
  const int dchunk = decode_max_tokens((int)k, w->bits, (int)g, topk, weight_format(w));
  if (dchunk < 1) return WQL_EUNSUPPORTED;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  // No workspace (allowed when topk == 0): the kernels skip the error word.
  unsigned int* err_word =
      ws ? reinterpret_cast<unsigned int*>(ws + lay.counter_off) + 1 : nullptr;
  LogitsArgs base{};
  base.x_dtype = x_dtype;
  base.qweight = w->qweight;
  base.scales = static_cast<const uint16_t*>(w->scales);
  base.bits = w->bits;
  base.group_eff = (int)g;
  base.scale_dtype = w->scale_dtype;
  base.n = (int)n;
  base.k = (int)k;
  base.bias = bias;
  base.topk = topk;
  base.format = weight_format(w);
  base.weights_static = (w->format & WQL_WEIGHT_STATIC) ? 1 : 0;
  base.zeros = static_cast<const uint8_t*>(w->zeros);
  // the counter block also schedules the decode kernel's work units
  if (ws) base.counter = reinterpret_cast<unsigned int*>(ws + lay.counter_off);
  if (topk > 0) {
    base.cand = reinterpret_cast<unsigned long long*>(ws + lay.cand_off);
    base.tickets = reinterpret_cast<unsigned int*>(ws + lay.tickets_off);
  }
  // Token counts above 16 go to the tensor-core kernel (up to 256 tokens per
  // launch) when it supports the dtype combination; otherwise the decode
  // kernel runs on 16-token slices.
  LogitsArgs probe = base;
  probe.m = (int)(m < 256 ? m : 256);
  // (fp8 and zero-point weights, and candidates alone, take the decode
  // kernel's 16-token slices at every m)
  const bool use_tc = m > kDecodeMaxTokens && weight_format(w) == WQL_FMT_SYM && logits_out &&
                      tc_supported(probe);
  // decode slices of balanced size (16 tokens that do not fit one launch run
  // as 8 + 8, not 15 + 1: the weight is streamed once per slice either way)
  const int64_t nslices = (m + dchunk - 1) / dchunk;
  const int64_t chunk = use_tc ? 256 : (m + nslices - 1) / nslices;
  for (int64_t m0 = 0; m0 < m; m0 += chunk) {
    const int64_t mc = (m - m0) < chunk ? (m - m0) : chunk;
    LogitsArgs a = base;
    a.x = static_cast<const unsigned char*>(x) + (size_t)m0 * k * esz;
    a.m = (int)mc;
    a.logits = logits_out ? static_cast<unsigned char*>(logits_out) + (size_t)m0 * n * esz
                          : nullptr;
    if (topk > 0) {
      a.topk_idx = topk_idx + (size_t)m0 * topk;
      a.topk_val = topk_val + (size_t)m0 * topk;
    }
    cudaError_t e;
    if (use_tc && mc > kDecodeMaxTokens) {
      // logits on the tensor cores, then the top-K from the rounded logits
      LogitsArgs g = a;
      g.topk = 0;
      e = launch_tc(g, err_word, stream);
      if (e == cudaSuccess && a.topk > 0) e = launch_topk_select(a, stream);
    } else
      e = launch_decode(a, err_word, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return WQL_OK;
}

wql_status wql_embed_gather(const int32_t* ids, int64_t t, const wql_weight* w,
                            int32_t out_dtype, void* out, cudaStream_t stream) {
  if (!w || t < 0 || w->n < 0 || w->k <= 0 || w->group < 0) return WQL_EINVAL;
  const int fmt = weight_format(w);
  if ((w->format & ~(WQL_FMT_MASK | WQL_WEIGHT_STATIC)) != 0 ||
      (fmt != WQL_FMT_SYM && fmt != WQL_FMT_E4M3 && fmt != WQL_FMT_ASYM))
    return WQL_EINVAL;
  if (fmt != WQL_FMT_SYM) return WQL_EUNSUPPORTED;
  const int64_t n = w->n, k = w->k;
  if (t > 0 && (!ids || !out)) return WQL_EINVAL;
  if (t > 0 && n > 0 && (!w->qweight || !w->scales)) return WQL_EINVAL;
  if (w->bits != 4 && w->bits != 8) return WQL_EUNSUPPORTED;
  if (!half_dtype(out_dtype) || !half_dtype(w->scale_dtype)) return WQL_EUNSUPPORTED;
  const int64_t g = w->group == 0 ? k : w->group;
  if (k % 8 != 0 || g % 8 != 0 || k % g != 0) return WQL_EUNSUPPORTED;
  if (n >= (int64_t(1) << 31) || t >= (int64_t(1) << 31) || k >= (int64_t(1) << 30))
    return WQL_EUNSUPPORTED;
  if (!aligned(ids, 4) || !aligned(w->qweight, 8) || !aligned(w->scales, 2) || !aligned(out, 16))
    return WQL_EUNSUPPORTED;
  if (t == 0) return WQL_OK;
  EmbedArgs a{};
  a.ids = ids;
  a.t = (int)t;
  a.qweight = w->qweight;
  a.scales = static_cast<const uint16_t*>(w->scales);
  a.bits = w->bits;
  a.group_eff = (int)g;
  a.scale_dtype = w->scale_dtype;
  a.n = (int)n;
  a.k = (int)k;
  a.out_dtype = out_dtype;
  a.out = out;
  cudaError_t e = launch_embed_gather(a, stream);
  return e == cudaSuccess ? WQL_OK : cuda_fail(e);
}

wql_status wql_topk_rescore(const void* x, int32_t x_dtype, int64_t m, const void* w_ref,
                            int32_t wref_dtype, int64_t n, int64_t k, const void* bias,
                            int32_t topk, int32_t* topk_idx, float* topk_val,
                            void* logits_inout, cudaStream_t stream) {
  if (m < 0 || n < 0 || k <= 0) return WQL_EINVAL;
  if (topk < 0 || topk > WQL_MAX_TOPK || topk > n) return WQL_EINVAL;
  if (m > 0 && topk > 0 && (!x || !w_ref || !topk_idx || !topk_val || !logits_inout))
    return WQL_EINVAL;
  if (!half_dtype(x_dtype) || wref_dtype != x_dtype) return WQL_EUNSUPPORTED;
  if (k % 8 != 0) return WQL_EUNSUPPORTED;
  if (n >= (int64_t(1) << 31) || m >= (int64_t(1) << 31)) return WQL_EUNSUPPORTED;
  if (!aligned(x, 16) || !aligned(w_ref, 16) || !aligned(logits_inout, 2) || !aligned(bias, 2))
    return WQL_EUNSUPPORTED;
  if (m == 0 || n == 0 || topk == 0) return WQL_OK;
  RescoreArgs a{};
  a.x = x;
  a.x_dtype = x_dtype;
  a.m = (int)m;
  a.n = (int)n;
  a.k = (int)k;
  a.w_ref = w_ref;
  a.bias = bias;
  a.topk = topk;
  a.topk_idx = topk_idx;
  a.topk_val = topk_val;
  a.logits = logits_inout;
  cudaError_t e = launch_rescore(a, stream);
  return e == cudaSuccess ? WQL_OK : cuda_fail(e);
}

wql_status wql_debug_set_waits(int64_t budget_cycles, int32_t stall_mma) {
  if (budget_cycles < 0 || (stall_mma != 0 && stall_mma != 1)) return WQL_EINVAL;
  g_wait_budget.store(budget_cycles, std::memory_order_relaxed);
  g_stall_mma.store(stall_mma, std::memory_order_relaxed);
  return WQL_OK;
}

}  // extern "C"
