// Merge of attention results computed over disjoint key sets.
//
// For P partial results (O_p, LSE_p) of the same queries over disjoint key
// sets, attention over the union of the sets is
//   w_p = exp(LSE_p - M), M = max_p LSE_p,
//   O = sum_p w_p O_p / sum_p w_p,   LSE = M + ln sum_p w_p,
// the combine step of the ring attention on page "长文本处理性能断层真相", §1
// (each GPU attends over its slice of the tokens); the decode path uses it for
// the key chunks of one sequence.  Rows whose parts are all -inf get O = 0 and
// LSE = -inf.
//
// One CTA per output row (b, s, h): each of the 8 warps computes the weights
// (lanes over parts), accumulates its share of the parts (lanes over the head
// dim, several parts' loads in flight), and the warps' sums are added through
// shared memory.  The work is a few bytes per part and row: latency, not
// bandwidth, sets its time, hence the spread over warps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fwd_kernel.cuh"

namespace attn {
namespace dec {

constexpr int kMergeWarps = 8;
constexpr int kMergeMaxD = 1024;

// Layouts: o_parts [P, B, S, H, D] (fp32 or 16-bit), lse_parts [P, B, H, S];
// o [B, S, H, D] (16-bit), lse [B, H, S].
template <typename Tin, bool BF16>
__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(
    const Tin* __restrict__ o_parts, const float* __restrict__ lse_parts, int P, int B, int S,
    int H, int D, void* o, float* lse) {
  extern __shared__ float acc_s[];  // [kMergeWarps][D]
  const long long row = blockIdx.x;  // (b * S + s) * H + h
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = static_cast<int>(row % H);
  const long long bs = row / H;
  const int s = static_cast<int>(bs % S);
  const int b = static_cast<int>(bs / S);
  const long long lrow = (static_cast<long long>(b) * H + h) * S + s;
  const long long lstride = static_cast<long long>(B) * H * S;
  const long long ostride = static_cast<long long>(B) * S * H * D;

  float M = -INFINITY;
  for (int q = lane; q < P; q += 32) M = fmaxf(M, lse_parts[q * lstride + lrow]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float z = 0.0f;
  if (M != -INFINITY)
    for (int q = lane; q < P; q += 32) z += __expf(lse_parts[q * lstride + lrow] - M);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);

  for (int d0 = 0; d0 < D; d0 += 32) {
    const int d = d0 + lane;
    float acc = 0.0f;
    if (M != -INFINITY && d < D) {
#pragma unroll 4
      for (int q = warp; q < P; q += kMergeWarps) {
        const float lp = lse_parts[q * lstride + lrow];
        float x;
        if constexpr (sizeof(Tin) == 4) {
          x = o_parts[q * ostride + row * D + d];
        } else {
          const uint16_t raw =
              reinterpret_cast<const uint16_t*>(o_parts)[q * ostride + row * D + d];
          x = BF16 ? __uint_as_float(static_cast<uint32_t>(raw) << 16)
                   : __half2float(__ushort_as_half(raw));
        }
        acc += (lp == -INFINITY ? 0.0f : __expf(lp - M)) * x;
      }
    }
    if (d < D) acc_s[warp * D + d] = acc;
  }
  __syncthreads();
  uint16_t* const O = static_cast<uint16_t*>(o);
  for (int d = threadIdx.x; d < D; d += kMergeWarps * 32) {
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) sum += acc_s[w * D + d];
    const float v = M == -INFINITY ? 0.0f : sum / z;
    O[row * D + d] = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
                          : __half_as_ushort(__float2half_rn(v));
  }
  if (threadIdx.x == 0) lse[lrow] = M == -INFINITY ? -INFINITY : M + __logf(z);
}

template <typename Tin, bool BF16>
cudaError_t launch_merge(const Tin* o_parts, const float* lse_parts, int P, int B, int S, int H,
                         int D, void* o, float* lse, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * S * H;
  if (rows == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(kMergeWarps) * D * sizeof(float);
  const void* fn = reinterpret_cast<const void*>(&attn_merge_kernel<Tin, BF16>);
  static std::atomic<unsigned long long> opted{0};  // opted in for the largest head dim
  cudaError_t e = smem_opt_in(fn, kMergeWarps * kMergeMaxD * static_cast<int>(sizeof(float)),
                              opted);
  if (e != cudaSuccess) return e;
  attn_merge_kernel<Tin, BF16><<<static_cast<unsigned>(rows), kMergeWarps * 32, smem, stream>>>(
      o_parts, lse_parts, P, B, S, H, D, o, lse);
  return cudaGetLastError();
}

}  // namespace dec
}  // namespace attn
