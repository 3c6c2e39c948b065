// Fused attention forward with 8-bit (e4m3) Q, K, V and per-tensor scales.
//
// What it computes: the same O and LSE as attn_fwd, for inputs given as e4m3
// codes and one dequantisation factor per tensor (q = q_e4m3 * q_scale, ...):
//   O_i = sum_j softmax_j(scale * q_i . k_j) v_j,  LSE_i = ln sum_j exp(scale q_i . k_j).
// Page "深度学习算子优化：从TFLOPS幻觉到FlashAttention实战", §3 names low-precision
// operands as a memory and throughput lever of the fused kernel; the online
// softmax is the same as the 16-bit path.
//
// GB300 mapping (the 16-bit single-CTA kernel with kind::f8f6f4 products):
//   * S = Q K^T with tcgen05.mma.kind::f8f6f4 (e4m3 x e4m3, fp32 accumulator,
//     K = 32 per instruction); a 128 x 128 e4m3 tile is one 16 KiB
//     128-byte-swizzled block, so D = 128 needs a single TMA box per tile;
//   * the scores' scale folds all three factors: c = scale q_s k_s log2 e;
//   * P is kept as e4m3 for O += P V: p' = 2^(c s - m + 4), four per TMEM
//     column.  The running max m is replaced (and O rescaled) once the row max
//     exceeds it by 2^4, so p' <= 2^8 stays below the e4m3 maximum (448) while
//     probabilities down to 2^-10 of the max stay in its normal range; the row
//     sum that normalises O adds the same rounded values, so the factor and
//     the rounding bias cancel; O is multiplied by v_s / l;
//   * V enters as its transpose V^T [H, D, keys] so that both products use
//     K-major operands (a separate pass writes it, keys padded per sequence
//     to a multiple of 16 so every TMA box starts 16-byte aligned).
// Roles as in the 16-bit kernel: warps 0-7 softmax (two query tiles, one
// thread per row), warp 8 issues the MMAs, warp 9 the TMA copies; every wait
// is bounded.
#pragma once

#include "fwd_kernel.cuh"

namespace attn {
namespace fp8 {

constexpr int D = 128;
constexpr int kStages = 4;
constexpr float kOffsetLog2 = 4.0f;   // p' = 2^offset p
constexpr float kRescaleLog2F8 = 4.0f;  // offset + threshold <= log2(448)

struct Fp8Params {
  FwdParams f;        // tm_q, tm_k: [rows, H, 128] e4m3, box 128 x 1 x 128; tm_v: V^T
  int sk_pad;         // keys per sequence in V^T (Sk rounded up to 16)
  float o_mul;        // v_scale: O = acc * o_mul / l
};

struct Layout8 {
  static constexpr int kTile = 16384;  // 128 rows x 128 B
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTiles * kTile;
  static constexpr int kVOff = kKOff + kStages * kTile;
  static constexpr int kBarOff = kVOff + kStages * kTile;
  static constexpr int QF = 0, QE = 1, KF = 2, KE = KF + kStages, VF = KE + kStages,
                       VE = VF + kStages, SF = VE + kStages, PF = SF + 2, OF = PF + 2,
                       DONE = OF + 2, kNumBars = DONE + 1;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS = 0, kColO = 256;
};

// Two fp32 -> two e4m3 codes (round to nearest even, saturating), low code first.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t x;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(x) : "f"(hi), "f"(lo));
  return x;
}
// acc + both values of an e4m3 pair (exact: e4m3 -> f16 -> f32 is exact).
__device__ __forceinline__ float add_e4m3x2(float acc, uint32_t pair16) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(pair16)));
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %0, hi, %0;\n\t}"
      : "+f"(acc) : "r"(h2));
  return acc;
}

__device__ __forceinline__ void mma_ss_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                          uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
               ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_ts_f8(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                          uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(acc) : "memory");
}

// ---------------------------------------------------------------- softmax
// One K/V tile of the online softmax for this thread's row: p' = 2^(c s - m + 4)
// rounded to e4m3 (four per column) over the first 32 columns of S; O is
// rescaled when the running max grew by more than 2^4.
__device__ __forceinline__ void softmax_step8(uint32_t tS, uint32_t tO, int lo, int limit,
                                              float cl, bool scale_pos, bool first,
                                              RowState& st) {
  uint32_t r[128];
  ptx::tmem_ld_x128(tS, r);
  float cle = cl;
  if (!scale_pos) {
#pragma unroll
    for (int c = 0; c < 128; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * cl);
    cle = 1.0f;
  }
  if (limit < 127 || lo > 0) {
#pragma unroll
    for (int c = 0; c < 128; ++c)
      if (c > limit || c < lo) r[c] = __float_as_uint(-INFINITY);
  }
  float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
  for (int c = 0; c < 128; c += 8) {
    mx0 = ptx::max3(mx0, __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
    mx1 = ptx::max3(mx1, __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
    mx2 = ptx::max3(mx2, __uint_as_float(r[c + 4]), __uint_as_float(r[c + 5]));
    mx3 = ptx::max3(mx3, __uint_as_float(r[c + 6]), __uint_as_float(r[c + 7]));
  }
  const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * cle;
  const float m_new = fmaxf(st.m, m_tile);
  const bool rescale = m_new > st.m + kRescaleLog2F8;
  const float m_use = rescale ? m_new : st.m;
  const float m_safe = (m_use == -INFINITY) ? 0.0f : m_use;
  const float alpha = rescale ? ptx::ex2(st.m - m_safe) : 1.0f;
  st.m = m_use;

  const uint64_t cl2 = ptx::f2(cle, cle);
  const uint64_t nm2 = ptx::f2(kOffsetLog2 - m_safe, kOffsetLog2 - m_safe);  // p' = 2^4 p
  uint64_t lx0 = ptx::f2(0.f, 0.f), lx1 = lx0;
  float lp0 = 0.f, lp1 = 0.f;
  uint32_t pk[32];
#pragma unroll
  for (int c = 0; c < 128; c += 4) {
    float x0, x1, x2, x3;
    ptx::f2_split(ptx::f2_fma(ptx::f2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), cl2,
                              nm2), x0, x1);
    ptx::f2_split(ptx::f2_fma(ptx::f2(__uint_as_float(r[c + 2]), __uint_as_float(r[c + 3])),
                              cl2, nm2), x2, x3);
    const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1), p2 = ptx::ex2(x2), p3 = ptx::ex2(x3);
    lx0 = ptx::f2_add(lx0, ptx::f2(p0, p1));
    lx1 = ptx::f2_add(lx1, ptx::f2(p2, p3));
    const uint32_t a = pack_e4m3x2(p0, p1), b = pack_e4m3x2(p2, p3);
    pk[c / 4] = a | (b << 16);
    lp0 = add_e4m3x2(lp0, a);
    lp1 = add_e4m3x2(lp1, b);
  }
  ptx::tmem_st_x32(tS, pk);
  float a0, a1, b0, b1;
  ptx::f2_split(lx0, a0, a1);
  ptx::f2_split(lx1, b0, b1);
  st.l_x = st.l_x * alpha + ((a0 + a1) + (b0 + b1));
  st.l_p = st.l_p * alpha + (lp0 + lp1);

  if (!first && __any_sync(0xffffffffu, rescale)) {
    const uint64_t al2 = ptx::f2(alpha, alpha);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t o[32];
      ptx::tmem_ld_x32(tO + c0, o);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float x, y;
        ptx::f2_split(
            ptx::f2_mul(ptx::f2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), al2), x, y);
        o[i] = __float_as_uint(x);
        o[i + 1] = __float_as_uint(y);
      }
      ptx::tmem_st_x32(tO + c0, o);
    }
  }
  ptx::tmem_wait_st();
}

template <bool BF16OUT>
__device__ void softmax_role8(const Fp8Params& q8, int t, uint32_t tmem, uint32_t bars,
                              const Ctl& ctl) {
  using L = Layout8;
  const FwdParams& p = q8.f;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + lane_bits + L::kColS + t * 128;
  const uint32_t tO = tmem + lane_bits + L::kColO + t * D;
  const uint32_t bar_s = bars + 8 * (L::SF + t);
  const uint32_t bar_p = bars + 8 * (L::PF + t);
  const uint32_t bar_o = bars + 8 * (L::OF + t);
  uint32_t s_cnt = 0, o_cnt = 0;
  uint16_t* const O = static_cast<uint16_t*>(p.o);

  Cursor cur;
  init_cursor<kUnitRows, false>(p, cur, false);
  Unit w;
  for (int k = 0; decode_unit<false>(p, slot_unit(p, k), cur, w, false); ++k) {
    if (!(t == 0 ? w.valid[0] : w.valid[1])) continue;
    const int q0 = w.q0 + t * kBM;
    const int qrow = q0 + row;
    const bool row_ok = qrow >= 0 && qrow < w.Lq;
    const int n = t == 0 ? w.n[0] : w.n[1];
    const long long orow = (static_cast<long long>(w.q_start) + qrow) * p.H + w.h;
    const long long lidx = (static_cast<long long>(w.b) * p.H + w.h) * p.Sq + qrow;
    RowState rs{-INFINITY, 0.0f, 0.0f};
    if (n > 0) {
      int key_lo, key_hi;
      row_keys(p, w, qrow, key_lo, key_hi);
      for (int j = 0, kb = w.j0 * kBN; j < n; ++j, kb += kBN) {
        if (!wait_bar_warp(bar_s, s_cnt & 1u, ctl)) return;
        ++s_cnt;
        ptx::tc_fence_after();
        softmax_step8(tS, tO, key_lo - kb, min(kBN - 1, key_hi - kb), p.scale_log2,
                      p.scale_pos != 0, j == 0, rs);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_p);
      }
      if (!wait_bar_warp(bar_o, o_cnt & 1u, ctl)) return;
      ++o_cnt;
      ptx::tc_fence_after();
      const float g = rs.l_p > 0.0f ? q8.o_mul / rs.l_p : 0.0f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        ptx::tmem_ld_x32(tO + c0, o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = ptx::pack2<BF16OUT>(__uint_as_float(o[2 * i]) * g,
                                      __uint_as_float(o[2 * i + 1]) * g);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(O + orow * D + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
    } else if (row_ok) {
      uint4* dst = reinterpret_cast<uint4*>(O + orow * D);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (row_ok) {  // l_x sums p' = 2^4 p: LSE = (m - 4 + log2 l_x) ln 2
      p.lse[lidx] = rs.l_x > 0.0f
                        ? (rs.m - kOffsetLog2 + ptx::lg2(rs.l_x)) * 0.69314718055994531f
                        : -INFINITY;
    }
  }
}

// -------------------------------------------------------------------- MMA
static __device__ void mma_loop8(const FwdParams& p, uint32_t smem, uint32_t tmem, uint32_t bars,
                          const Ctl& ctl) {
  using L = Layout8;
  constexpr uint32_t kId = ptx::idesc_f16_f32acc(false, kBM, kBN, false);  // e4m3 x e4m3, N = 128
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t kv_it = 0, q_it = 0, p_cnt[kTiles] = {0, 0};
  const uint64_t dq[kTiles] = {ptx::desc_sw128(smem + L::kQOff, 16, 1024),
                               ptx::desc_sw128(smem + L::kQOff + L::kTile, 16, 1024)};
  const uint64_t dk0 = ptx::desc_sw128(smem + L::kKOff, 16, 1024);
  const uint64_t dv0 = ptx::desc_sw128(smem + L::kVOff, 16, 1024);
  Cursor cur;
  init_cursor<kUnitRows, false>(p, cur, false);
  Unit w;
  for (int k = 0; decode_unit<false>(p, slot_unit(p, k), cur, w, false); ++k) {
    const int nmax = max(w.n[0], w.n[1]);
    if (nmax == 0) continue;
    if (!wait_bar(bar(L::QF), q_it & 1u, ctl)) return;
    ptx::tc_fence_after();
    for (int j = 0; j <= nmax; ++j) {
      bool k_ready = false, v_ready = false;
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        const uint32_t tS = tmem + L::kColS + t * 128;
        const uint32_t tO = tmem + L::kColO + t * D;
        if (j >= 1 && j - 1 < w.n[t]) {  // O_t += P_t(j-1) V(j-1): B = V^T tile, K-major
          if (!wait_bar(bar(L::PF + t), p_cnt[t] & 1u, ctl)) return;
          ++p_cnt[t];
          const uint32_t it = kv_it + j - 1;
          const uint32_t st = it % kStages;
          if (!v_ready) {
            if (!wait_bar(bar(L::VF + st), (it / kStages) & 1u, ctl)) return;
            v_ready = true;
          }
          ptx::tc_fence_after();
          const uint64_t dv = dv0 + ((st * L::kTile) >> 4);
#pragma unroll
          for (int ks = 0; ks < kBN / 32; ++ks)  // 32 keys = 32 B of a V^T row, 8 P columns
            mma_ts_f8(tO, tS + ks * 8, dv + ((ks * 32) >> 4), kId, (j - 1 > 0 || ks > 0) ? 1u : 0u);
          if (t == 1 || j - 1 >= w.n[1]) ptx::mma_commit(bar(L::VE + st));
          if (j - 1 == w.n[t] - 1) ptx::mma_commit(bar(L::OF + t));
        }
        if (j < w.n[t]) {  // S_t(j) = Q_t K(j)^T
          const uint32_t it = kv_it + j;
          const uint32_t st = it % kStages;
          if (!k_ready) {
            if (!wait_bar(bar(L::KF + st), (it / kStages) & 1u, ctl)) return;
            k_ready = true;
            ptx::tc_fence_after();
          }
          const uint64_t dk = dk0 + ((st * L::kTile) >> 4);
#pragma unroll
          for (int ks = 0; ks < D / 32; ++ks)
            mma_ss_f8(tS, dq[t] + ((ks * 32) >> 4), dk + ((ks * 32) >> 4), kId, ks > 0 ? 1u : 0u);
          ptx::mma_commit(bar(L::SF + t));
          if (t == 1 || j >= w.n[1]) ptx::mma_commit(bar(L::KE + st));
        }
      }
      if (j == nmax - 1) ptx::mma_commit(bar(L::QE));
    }
    kv_it += nmax;
    ++q_it;
  }
}

// ------------------------------------------------------------------- load
struct LoadLog8 {
  FillLog<1> q;
  FillLog<kStages> k, v;
};

// Every issued fill is recorded in `f` (see FillLog).
static __device__ void load_loop8(const Fp8Params& q8, uint32_t smem, uint32_t bars, const Ctl& ctl,
                                  LoadLog8& f) {
  using L = Layout8;
  const FwdParams& p = q8.f;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t kv_it = 0, q_it = 0;
  Cursor cur;
  init_cursor<kUnitRows, false>(p, cur, true);
  Unit w;
  for (int k = 0; decode_unit<false>(p, slot_unit(p, k), cur, w, true); ++k) {
    const int nmax = max(w.n[0], w.n[1]);
    if (nmax == 0) continue;
    if (q_it > 0 && !wait_bar(bar(L::QE), (q_it - 1) & 1u, ctl)) return;
    ptx::mbar_arrive_expect_tx(bar(L::QF), kTiles * L::kTile);
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
      ptx::tma_load_3d(smem + L::kQOff + t * L::kTile, &p.tm_q, bar(L::QF), 0, w.h,
                       w.q_start + w.q0 + t * kBM);
    f.q.last[0] = static_cast<int>(q_it);
    ++q_it;
    for (int j = 0; j < nmax; ++j) {
      const uint32_t it = kv_it + j;
      const uint32_t st = it % kStages;
      const int kt = w.j0 + j;
      if (it >= kStages && !wait_bar(bar(L::KE + st), (it / kStages - 1) & 1u, ctl)) return;
      ptx::mbar_arrive_expect_tx(bar(L::KF + st), L::kTile);
      ptx::tma_load_3d(smem + L::kKOff + st * L::kTile, &p.tm_k, bar(L::KF + st), 0, w.h,
                       w.k_start + kt * kBN);
      f.k.last[st] = static_cast<int>(it);
      if (it >= kStages && !wait_bar(bar(L::VE + st), (it / kStages - 1) & 1u, ctl)) return;
      ptx::mbar_arrive_expect_tx(bar(L::VF + st), L::kTile);
      // V^T [H, D, B * sk_pad]: x = key (16-byte aligned: sk_pad and 128 kt are), y = dim
      ptx::tma_load_3d(smem + L::kVOff + st * L::kTile, &p.tm_v, bar(L::VF + st),
                       w.b * q8.sk_pad + kt * kBN, 0, w.h);
      f.v.last[st] = static_cast<int>(it);
    }
    kv_it += nmax;
  }
}

template <bool BF16OUT>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_fp8_kernel(const __grid_constant__ Fp8Params q8) {
  using L = Layout8;
  const FwdParams& p = q8.f;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t smem = (raw + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (smem - raw);
  const uint32_t bars = smem + L::kBarOff;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(base + L::kMiscOff);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(base + L::kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i)
      ptx::mbar_init(bars + 8u * i, (i == L::PF || i == L::PF + 1) ? kBM : 1u);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    ptx::tma_prefetch_desc(&p.tm_q);
    ptx::tma_prefetch_desc(&p.tm_k);
    ptx::tma_prefetch_desc(&p.tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  if (warp < kMmaWarp) {
    softmax_role8<BF16OUT>(q8, warp >> 2, tmem, bars, ctl);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      mma_loop8(p, smem, tmem, bars, ctl);
      const uint32_t done = bars + 8u * L::DONE;
      ptx::mma_commit(done);
      wait_bar(done, 0, ctl, false);
    }
  } else if (lane == 0) {
    LoadLog8 f;
    f.q.clear();
    f.k.clear();
    f.v.clear();
    load_loop8(q8, smem, bars, ctl, f);
    // no TMA write may land after the CTA exits
    drain_fills(bars, L::QF, f.q, ctl);
    drain_fills(bars, L::KF, f.k, ctl);
    drain_fills(bars, L::VF, f.v, ctl);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// V [B, Sk, H, D] e4m3 -> V^T [H, D, B * sk_pad] (keys innermost, zero past Sk).
// One CTA per (b, h, 64-key block): read 64 rows of 128 B, write 128 rows of 64 B.
static __global__ void __launch_bounds__(256) attn_fp8_transpose_v(const uint8_t* __restrict__ v,
                                                            uint8_t* __restrict__ vt, int B,
                                                            int H, int Sk, int sk_pad) {
  __shared__ uint8_t tile[64][D + 4];
  const int nblk = (sk_pad + 63) / 64;
  const int blk = blockIdx.x % nblk;
  const int bh = blockIdx.x / nblk;
  const int h = bh % H, b = bh / H;
  const int k0 = blk * 64;
  for (int i = threadIdx.x; i < 64 * (D / 4); i += 256) {  // 4 bytes per thread-step
    const int kr = i / (D / 4), c4 = i % (D / 4);
    const int key = k0 + kr;
    uint32_t x = 0;
    if (key < Sk)
      x = *reinterpret_cast<const uint32_t*>(
          v + ((static_cast<long long>(b) * Sk + key) * H + h) * D + 4 * c4);
    tile[kr][4 * c4] = x & 0xff;
    tile[kr][4 * c4 + 1] = (x >> 8) & 0xff;
    tile[kr][4 * c4 + 2] = (x >> 16) & 0xff;
    tile[kr][4 * c4 + 3] = x >> 24;
  }
  __syncthreads();
  const int kmax = min(64, sk_pad - k0);
  for (int i = threadIdx.x; i < D * 16; i += 256) {  // D rows x 64 keys, 4 keys per step
    const int d = i / 16, k4 = i % 16;
    if (4 * k4 >= kmax) continue;
    const uint32_t x = tile[4 * k4][d] | (tile[4 * k4 + 1][d] << 8) |
                       (tile[4 * k4 + 2][d] << 16) | (static_cast<uint32_t>(tile[4 * k4 + 3][d]) << 24);
    *reinterpret_cast<uint32_t*>(
        vt + (static_cast<long long>(h) * D + d) * (static_cast<long long>(B) * sk_pad) +
        static_cast<long long>(b) * sk_pad + k0 + 4 * k4) = x;
  }
}

template <bool BF16OUT>
cudaError_t launch_fwd_fp8(const Fp8Params& q8, const uint8_t* v, uint8_t* vt, int grid,
                           cudaStream_t stream) {
  const FwdParams& p = q8.f;
  const int nblk = (q8.sk_pad + 63) / 64;
  attn_fp8_transpose_v<<<static_cast<unsigned>(p.B * p.H * nblk), 256, 0, stream>>>(
      v, vt, p.B, p.H, p.Sk, q8.sk_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const void* fn = reinterpret_cast<const void*>(&attn_fwd_fp8_kernel<BF16OUT>);
  static std::atomic<unsigned long long> opted{0};
  e = smem_opt_in(fn, Layout8::kAlloc, opted);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<Fp8Params*>(&q8)};
  return cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, Layout8::kAlloc, stream);
}

}  // namespace fp8
}  // namespace attn
