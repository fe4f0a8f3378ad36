// decode_xf16_sf16.cu -- instantiates the decode kernel variants for f16
// activations and f16 scales (one unit per dtype pair, compiled in parallel).
#include "decode_impl.cuh"

namespace wql {
namespace decode_detail {
template cudaError_t dispatch_xs<__half, __half>(const DecodeParams&, bool, bool, int, size_t, int,
                                     cudaStream_t);
}  // namespace decode_detail
}  // namespace wql
