// decode_xf16_sbf16.cu -- instantiates the decode kernel variants for f16
// activations and bf16 scales (one unit per dtype pair, compiled in parallel).
#include "decode_impl.cuh"

namespace wql {
namespace decode_detail {
template cudaError_t dispatch_xs<__half, __nv_bfloat16>(const DecodeParams&, bool, bool, int, size_t, int,
                                     cudaStream_t);
}  // namespace decode_detail
}  // namespace wql
