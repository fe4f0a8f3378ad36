// decode_bf16.cu -- instantiates the decode kernel variants for bf16 activations
// (split from the other dtype so the two compile in parallel).
#include "decode_impl.cuh"

namespace wql {
namespace decode_detail {
template cudaError_t dispatch_x<__nv_bfloat16>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                      const DecodeParams&, size_t, int, cudaStream_t);
}  // namespace decode_detail
}  // namespace wql
