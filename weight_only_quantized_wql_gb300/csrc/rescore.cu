// rescore.cu -- exact top-K rescoring ("Fused WNA16 GEMM for tied quantized
// lm_head logits", reviewer comment item 2): the K candidate rows found on
// the quantised logits are recomputed from the unquantised weight, written
// back into the logits and re-ranked.
//
// One CTA per token row, one warp per candidate.  A warp streams its weight
// row with 16-byte loads; fp16 x fp16 (or bf16 x bf16) products are exact in
// fp32 and are summed in fp32, then reduced across the warp.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "wql_common.cuh"

namespace wql {
namespace {

template <typename XT>
__device__ __forceinline__ float dot8(uint4 xa, uint4 wa, float acc) {
  const XT* xv = reinterpret_cast<const XT*>(&xa);
  const XT* wv = reinterpret_cast<const XT*>(&wa);
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = fmaf(to_f32(xv[i]), to_f32(wv[i]), acc);
  return acc;
}

template <typename XT>
__global__ void __launch_bounds__(WQL_MAX_TOPK * 32) rescore_kernel(const RescoreArgs a) {
  __shared__ unsigned long long keys[WQL_MAX_TOPK];
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = a.topk;
  griddep_launch_dependents();
  griddep_wait();   // the candidates and logits of the kernels before it
  if (warp < K) {
    const int idx = a.topk_idx[(size_t)row * K + warp];
    if (idx < 0 || idx >= a.n) {
      // not a vocab row: nothing is read or scattered; it ranks last as (-1, NaN)
      if (lane == 0) keys[warp] = (unsigned long long)(K - warp);
    } else {
    const uint4* xr = reinterpret_cast<const uint4*>(reinterpret_cast<const XT*>(a.x) +
                                                     (size_t)row * a.k);
    const uint4* wr = reinterpret_cast<const uint4*>(reinterpret_cast<const XT*>(a.w_ref) +
                                                     (size_t)idx * a.k);
    float acc = 0.f;
    for (int c = lane; c < a.k / 8; c += 32) acc = dot8<XT>(__ldg(xr + c), __ldg(wr + c), acc);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, m);
    if (lane == 0) {
      if (a.bias) acc += to_f32(reinterpret_cast<const XT*>(a.bias)[idx]);
      reinterpret_cast<XT*>(a.logits)[(size_t)row * a.n + idx] = from_f32<XT>(acc);
      keys[warp] = topk_key(acc, (uint32_t)idx);
    }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // re-rank the K rescored candidates: value descending, index ascending
    // keys are distinct (distinct indices), so the ranks form a permutation
    unsigned long long mine = lane < K ? keys[lane] : kEmptyKey;
    int rank = 0;
    for (int j = 0; j < K; ++j) rank += keys[j] > mine ? 1 : 0;
    if (lane < K) {
      const bool valid = mine > (unsigned long long)WQL_MAX_TOPK;
      a.topk_idx[(size_t)row * K + rank] = valid ? key_index(mine) : -1;
      a.topk_val[(size_t)row * K + rank] = valid ? key_value(mine) : __int_as_float(0x7FC00000);
    }
  }
}

}  // namespace

cudaError_t launch_rescore(const RescoreArgs& a, cudaStream_t s) {
  const int threads = a.topk * 32;
  const cudaError_t e =
      a.x_dtype == WQL_F16
          ? launch_pdl(rescore_kernel<__half>, dim3(a.m), dim3(threads), 0, s, a)
          : launch_pdl(rescore_kernel<__nv_bfloat16>, dim3(a.m), dim3(threads), 0, s, a);
  note_launch();
  return e;
}

}  // namespace wql
