// embed.cuh -- arguments and launcher of the tied-embedding gather
// (embed.cu), shared with the C-ABI layer (wql_api.cu).
#pragma once

#include "wql_common.cuh"

namespace wql {

// out[i, :] = RN_out(q[ids[i], :] * s) (zeros for an id outside [0, n)).
struct EmbedArgs {
  const int32_t* ids;
  int t;                      // token ids
  const void* qweight;        // int4: uint32 [n, k/8]; int8: int8 [n, k]
  const uint16_t* scales;     // [n, k / group_eff]
  int bits, group_eff, scale_dtype;
  int n, k;
  int out_dtype;              // WQL_F16 or WQL_BF16
  void* out;                  // [t, k]
};
cudaError_t launch_embed_gather(const EmbedArgs& a, cudaStream_t s);

}  // namespace wql
