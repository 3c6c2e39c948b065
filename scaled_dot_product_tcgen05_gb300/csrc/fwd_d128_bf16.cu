// Instantiation of the fused attention forward for head dim 128, bf16 inputs.
#include "fwd_kernel.cuh"

namespace attn {
template cudaError_t launch_fwd<128, true>(const FwdParams&, int, cudaStream_t);
}  // namespace attn
