// decode_xbf16_sbf16.cu -- instantiates the decode kernel variants for bf16
// activations and bf16 scales (one unit per dtype pair, compiled in parallel).
#include "decode_impl.cuh"

namespace wql {
namespace decode_detail {
template cudaError_t dispatch_xs<__nv_bfloat16, __nv_bfloat16>(const DecodeParams&, bool, bool, int, size_t, int,
                                     cudaStream_t);
}  // namespace decode_detail
}  // namespace wql
