// Instantiation of the fused attention forward for head dim 64, f16 inputs:
// the single-CTA kernel and the CTA-pair (2-SM MMA) kernel.
#include "fwd_kernel_2sm.cuh"

namespace attn {
template cudaError_t launch_fwd<64, false>(const FwdParams&, int, cudaStream_t);
namespace pair {
template cudaError_t launch_fwd_2sm<64, false>(const FwdParams&, int, cudaStream_t);
}  // namespace pair
}  // namespace attn
