// Instantiation of the KV-cache decode kernel for head dim 128 (fp16 and bf16;
// 1, up to 4 and up to 16 new queries per sequence) and of the merge kernel.
#include "decode_kernel.cuh"
#include "merge_kernel.cuh"

namespace attn {
namespace dec {
template cudaError_t launch_decode<128, 1, false>(const DecParams&, int, cudaStream_t);
template cudaError_t launch_decode<128, 4, false>(const DecParams&, int, cudaStream_t);
template cudaError_t launch_decode<128, 16, false>(const DecParams&, int, cudaStream_t);
template cudaError_t launch_decode<128, 1, true>(const DecParams&, int, cudaStream_t);
template cudaError_t launch_decode<128, 4, true>(const DecParams&, int, cudaStream_t);
template cudaError_t launch_decode<128, 16, true>(const DecParams&, int, cudaStream_t);
template cudaError_t launch_merge<uint16_t, false>(const uint16_t*, const float*, int, int, int,
                                                   int, int, void*, float*, cudaStream_t);
template cudaError_t launch_merge<uint16_t, true>(const uint16_t*, const float*, int, int, int,
                                                  int, int, void*, float*, cudaStream_t);
}  // namespace dec
}  // namespace attn
