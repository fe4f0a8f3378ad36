// noalloc.cu -- wql_logits_noalloc: logits (+ top-K candidates) for callers
// that cannot give the library a workspace buffer.
//
// Who needs it.  wql_logits wants a caller-owned device workspace for the
// decode kernel's scratch.  Some callers have no way to make one: a host
// program that links only this C library and has no device allocator of its
// own, or a serving loop that reserves all of its device memory when it
// starts and must not allocate while it runs (an allocation there can fail
// under memory pressure, synchronise the device, or break the memory plan
// the loop was sized with).  For them the scratch lives in one fixed-size
// array in device memory that belongs to this library's image.  The CUDA
// runtime reserves it when it loads this file's module on a device; this
// entry point itself allocates nothing, and neither does anything it calls.
//
// What the area holds (the decode kernel's workspace, for at most 16 token
// rows per launch): the ticket counter, the sticky error word, the
// per-token top-K bounds and candidate counts (one 256-byte block), the top-K
// candidates, and the fp32 logits that the top-K selection reads back when they do not
// fit in shared memory.  The 256-byte block must be zero when a launch
// starts; every call clears it on its own stream before its first launch.  The rest is
// written before it is read within each launch.
//
// One area per device, shared by every call on that device: calls that can
// be in flight at the same time (on different streams, or from different
// host threads without ordering between them) race on it and corrupt each
// other's results.  Serialise them.
#include <mutex>

#include <cuda.h>

#include "wql_common.cuh"

namespace wql {
namespace {

constexpr size_t kAreaBytes = WQL_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch area.  Without an initialiser it is zero-filled when the
// module is loaded and takes no room in the library file.
static __device__ __align__(256) unsigned char g_noalloc_area[kAreaBytes];

// Device address of the area, per device ordinal, with the identity of the
// context it was looked up in: the address belongs to the module as that
// context loaded it.  A context torn down and created again (cudaDeviceReset,
// for one) loads the module afresh, possibly elsewhere, so an address is only
// reused while the device's current context has the same unique id.
struct AreaSlot {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;
};
AreaSlot g_area[kMaxDevices];
std::mutex g_setup_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_fn_once;

void resolve_ctx_fns() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
}

// Unique id of the calling thread's current context (0 if none).
cudaError_t current_ctx_id(unsigned long long* id) {
  std::call_once(g_ctx_fn_once, resolve_ctx_fns);
  if (!g_ctx_current || !g_ctx_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  *id = 0;
  if (ctx && g_ctx_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// Address of the area on the current device.  The set-up -- with that device
// current, cudaGetSymbolAddress, which also makes the runtime load the module
// there -- runs on the first call per device and again whenever the device's
// context has been replaced since.  A failed lookup is not kept, so a later
// call tries again.
cudaError_t area_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // id 0: no context is current yet on this thread (the lookup below makes
  // the device's primary context current, and its id is read after it)
  unsigned long long id = 0;
  e = current_ctx_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  AreaSlot& slot = g_area[dev];
  if (slot.ptr == nullptr || slot.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_area);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    e = current_ctx_id(&id);
    if (e != cudaSuccess) return e;
    slot.ptr = p;
    slot.ctx_id = id;
  }
  *out = slot.ptr;
  return cudaSuccess;
}


}  // namespace
}  // namespace wql

using namespace wql;

extern "C" wql_status wql_logits_noalloc(const void* x, int32_t x_dtype, int64_t m,
                                         const wql_weight* w, const void* bias,
                                         void* logits_out, int32_t topk, int32_t* topk_idx,
                                         float* topk_val, cudaStream_t stream) {
  // Host checks first: a rejected call makes no CUDA call at all.
  int64_t g = 0;
  const wql_status st = check_logits_args(x, x_dtype, m, w, bias, logits_out, topk, topk_idx,
                                          topk_val, &g);
  if (st != WQL_OK) return st;
  const int64_t n = w->n, k = w->k;
  if (m == 0 || n == 0) return WQL_OK;
  const int max_tokens = decode_max_tokens((int)k, w->bits, (int)g, topk, weight_format(w));
  if (max_tokens < 1) return WQL_EUNSUPPORTED;
  // balanced slices (16 tokens that do not fit one launch run as 8 + 8)
  const int64_t nslices = (m + max_tokens - 1) / max_tokens;
  const int slice_tokens = (int)((m + nslices - 1) / nslices);
  const int64_t slice_max = m < slice_tokens ? m : slice_tokens;
  // Every slice reuses the same area, so one slice's layout is the need.
  const WorkspaceLayout lay = workspace_layout(slice_max, n, topk);
  if (lay.total > kAreaBytes) return WQL_EWORKSPACE;

  void* area = nullptr;
  cudaError_t e = area_on_current_device(&area);
  if (e != cudaSuccess) return record_cuda_error(e);
  unsigned char* ws = static_cast<unsigned char*>(area);
  unsigned int* counter = reinterpret_cast<unsigned int*>(ws + lay.counter_off);
  unsigned int* err_word = counter + 1;
  // The counter block (ticket counter, error word, per-token top-K bounds and
  // candidate counts) starts every call at zero.
  e = cudaMemsetAsync(counter, 0, 256, stream);
  if (e != cudaSuccess) return record_cuda_error(e);

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
  base.counter = counter;   // also schedules the decode kernel's work units
  if (topk > 0) {
    base.cand = reinterpret_cast<unsigned long long*>(ws + lay.cand_off);
  }
  const size_t esz = 2;
  for (int64_t m0 = 0; m0 < m; m0 += slice_tokens) {
    const int64_t mc = (m - m0) < slice_tokens ? (m - m0) : slice_tokens;
    LogitsArgs a = base;
    a.x = static_cast<const unsigned char*>(x) + (size_t)m0 * (size_t)k * esz;
    a.m = (int)mc;
    a.logits = logits_out ? static_cast<unsigned char*>(logits_out) + (size_t)m0 * (size_t)n * esz
                          : nullptr;
    if (topk > 0) {
      a.topk_idx = topk_idx + (size_t)m0 * topk;
      a.topk_val = topk_val + (size_t)m0 * topk;
    }
    e = launch_decode(a, err_word, stream);
    if (e != cudaSuccess) return record_cuda_error(e);
  }
  return WQL_OK;
}
