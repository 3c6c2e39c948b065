// Instantiation of the fused attention forward for head dim 128, f16 inputs.
#include "fwd_kernel.cuh"

namespace attn {
template cudaError_t launch_fwd<128, false>(const FwdParams&, int, cudaStream_t);
}  // namespace attn
