// Instantiation of the attention backward (pre-pass, main kernel, dQ
// conversion) for head dim 64, fp16 and bf16, dense and packed sequences.
#include "bwd_kernel.cuh"

namespace attn {
namespace bwd {
template cudaError_t launch_bwd<64, false>(const BwdParams&, const uint16_t*, const uint16_t*,
                                          const float*, uint8_t*, int32_t*, long long,
                                          uint16_t*, int, cudaStream_t);
template cudaError_t launch_bwd<64, true>(const BwdParams&, const uint16_t*, const uint16_t*,
                                         const float*, uint8_t*, int32_t*, long long, uint16_t*,
                                         int, cudaStream_t);
}  // namespace bwd
}  // namespace attn
