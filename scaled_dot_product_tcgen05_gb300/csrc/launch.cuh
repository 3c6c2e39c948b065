// Host-side kernel choice and launch shared by the C entry points.
#pragma once

#include <cstdlib>

#include "fwd_kernel.cuh"
#include "fwd_kernel_2sm.cuh"

namespace attn {

extern template cudaError_t launch_fwd<64, false>(const FwdParams&, int, cudaStream_t);
extern template cudaError_t launch_fwd<64, true>(const FwdParams&, int, cudaStream_t);
extern template cudaError_t launch_fwd<128, false>(const FwdParams&, int, cudaStream_t);
extern template cudaError_t launch_fwd<128, true>(const FwdParams&, int, cudaStream_t);
namespace pair {
extern template cudaError_t launch_fwd_2sm<64, false>(const FwdParams&, int, cudaStream_t);
extern template cudaError_t launch_fwd_2sm<64, true>(const FwdParams&, int, cudaStream_t);
extern template cudaError_t launch_fwd_2sm<128, false>(const FwdParams&, int, cudaStream_t);
extern template cudaError_t launch_fwd_2sm<128, true>(const FwdParams&, int, cudaStream_t);
}  // namespace pair

// Fills the visibility fields of `p` (see FwdParams) from the C arguments:
// window_left / window_right = -1 leave that side unbounded, causal bounds the
// right side at the diagonal, rows below global_q see all keys.  Returns false
// for a request the rules reject (a negative size other than -1, or a right
// window wider than 0 together with causal).
inline bool set_mask(FwdParams& p, int causal, int window_left, int window_right, int global_q) {
  if (window_left < -1 || window_right < -1 || global_q < 0) return false;
  if (causal && window_right > 0) return false;
  p.causal = causal ? 1 : 0;
  p.win_left = window_left < 0 ? kUnbounded : (window_left < kUnbounded ? window_left : kUnbounded);
  p.win_right = causal ? 0
                       : (window_right < 0 ? kUnbounded
                                           : (window_right < kUnbounded ? window_right : kUnbounded));
  p.global_q = global_q;
  return true;
}

struct LaunchInfo {
  int grid = 0;
  int smem = 0;
  bool pair = false;
};

// Upper bound of the work units of a call with `rows_per_unit` query rows per unit.
inline long long units_bound(bool varlen, int B, int H, long long rows_q, int Sq,
                             int rows_per_unit) {
  return varlen ? static_cast<long long>(H) * ((rows_q + rows_per_unit - 1) / rows_per_unit + B)
                : static_cast<long long>(B) * H * ((Sq + rows_per_unit - 1) / rows_per_unit);
}

// Paired row blocks (FwdParams::pair_blocks) balance the workers' loads when
// each worker gets many units; with few units per worker they would only halve
// the parallelism.
inline int pair_blocks_for(long long units, long long workers) {
  return units >= 16 * workers ? 1 : 0;
}

// Row-block-major unit order (FwdParams::block_major) for dense calls whose K
// and V (all batches and heads) take at most half of the 129 MB L2: their
// heads need no locality, and a global heaviest-first order balances the
// workers when each gets only a few units (B=8 H=12 S=2048 causal: the
// busiest worker's share falls from 1.19 to 1.06 times the mean for single
// CTAs, and from 1.17 to 1.01 for CTA pairs).
inline int block_major_for(bool varlen, int B, int H, int Sk, int D) {
  const long long kv_bytes = 4LL * B * H * static_cast<long long>(Sk) * D;  // 16-bit K and V
  return !varlen && kv_bytes <= 64LL * 1024 * 1024 ? 1 : 0;
}

// Kernel choice.  Head dim 128 runs on CTA pairs with 2-SM MMAs.  Head dim 64
// runs on CTA pairs without a causal mask and on single CTAs with one (measured
// on GB300: pairs 689 vs 648 TFLOP/s at B=8 H=12 S=2048 non-causal, single
// CTAs 521 vs 470 causal, within 2-3 % of each other on long sequences).
// ATTN_PAIR=0 forces single CTAs, ATTN_PAIR=1 CTA pairs (cross-checks).  The
// grid is persistent: at most one CTA per SM.
inline cudaError_t launch_forward(const FwdParams& params, int D, bool bf16, bool varlen, int B,
                                  int H, long long rows_q, int Sq, int sms, cudaStream_t s,
                                  LaunchInfo* info) {
  FwdParams p = params;
  const char* sel = std::getenv("ATTN_PAIR");
  const bool forced = sel != nullptr && (sel[0] == '0' || sel[0] == '1');
  const bool use_pair =
      sms >= 2 && (forced ? sel[0] == '1' : (D == 128 || p.causal == 0));
  if (use_pair) {
    const long long units = units_bound(varlen, B, H, rows_q, Sq, pair::kUR);
    const long long pairs = units < sms / 2 ? units : sms / 2;
    p.pair_blocks = pair_blocks_for(units, pairs);
    p.block_major = block_major_for(varlen, B, H, p.Sk, D);
    info->grid = static_cast<int>(2 * pairs);
    info->smem = D == 64 ? pair::fwd_2sm_smem_bytes<64>(p) : pair::fwd_2sm_smem_bytes<128>(p);
    info->pair = true;
    if (pairs <= 0) return cudaSuccess;
    if (D == 64)
      return bf16 ? pair::launch_fwd_2sm<64, true>(p, info->grid, s)
                  : pair::launch_fwd_2sm<64, false>(p, info->grid, s);
    return bf16 ? pair::launch_fwd_2sm<128, true>(p, info->grid, s)
                : pair::launch_fwd_2sm<128, false>(p, info->grid, s);
  }
  const long long units = units_bound(varlen, B, H, rows_q, Sq, kUnitRows);
  info->grid = static_cast<int>(units < sms ? units : sms);
  info->pair = false;
  p.pair_blocks = pair_blocks_for(units, info->grid);
  p.block_major = block_major_for(varlen, B, H, p.Sk, D);
  if (D == 64) {
    info->smem = fwd_smem_bytes<64>(p);
    if (info->grid <= 0) return cudaSuccess;
    return bf16 ? launch_fwd<64, true>(p, info->grid, s) : launch_fwd<64, false>(p, info->grid, s);
  }
  info->smem = fwd_smem_bytes<128>(p);
  if (info->grid <= 0) return cudaSuccess;
  return bf16 ? launch_fwd<128, true>(p, info->grid, s) : launch_fwd<128, false>(p, info->grid, s);
}

}  // namespace attn
