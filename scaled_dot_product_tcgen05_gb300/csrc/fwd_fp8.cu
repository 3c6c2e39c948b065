// Instantiation of the e4m3 attention forward (head dim 128; bf16 or fp16 output)
// and of its V transpose.
#include "fwd_fp8_kernel.cuh"

namespace attn {
namespace fp8 {
template cudaError_t launch_fwd_fp8<true>(const Fp8Params&, const uint8_t*, uint8_t*, int,
                                          cudaStream_t);
template cudaError_t launch_fwd_fp8<false>(const Fp8Params&, const uint8_t*, uint8_t*, int,
                                           cudaStream_t);
}  // namespace fp8
}  // namespace attn
