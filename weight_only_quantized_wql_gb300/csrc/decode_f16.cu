// decode_f16.cu -- instantiates the decode kernel variants for fp16 activations
// (split from the other dtype so the two compile in parallel).
#include "decode_impl.cuh"

namespace wql {
namespace decode_detail {
template cudaError_t dispatch_x<__half>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                      const DecodeParams&, size_t, int, cudaStream_t);
}  // namespace decode_detail
}  // namespace wql
