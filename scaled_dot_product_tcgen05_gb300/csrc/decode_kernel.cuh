// Attention decode against a KV cache (Sq <= 16 new queries per sequence),
// split over the keys, and the merge of partial results.
//
// What it computes, per sequence b, head h and new query t (at position
// L_b - Sq + t of a sequence whose cache holds L_b keys):
//   O = softmax(scale * q K^T) V over the visible cached keys (all L_b keys, or
//   keys 0 .. L_b - Sq + t when causal), LSE = ln sum exp(scale * q . k).
// The cache layout and the decode step follow page "长文本处理性能断层真相",
// §2.2 (the KV cache that grows with the sequence); the split of the keys
// into chunks whose partial (O, LSE) are merged afterwards is the combine
// step of the ring attention on the same page, §1, applied inside one GPU.
//
// GB300 mapping.  With Sq <= 16 queries per head every cached K/V byte feeds
// at most 16 dot products, so the work is bound by HBM bandwidth, not by the
// tensor cores; the kernel streams the cache once at full bandwidth:
//   * persistent grid, one CTA per SM, work unit = (sequence, head, chunk of
//     the keys); units are dealt round-robin, so every SM streams about the
//     same number of bytes;
//   * warp 4 (one lane) moves 64-key K and V tiles with 3-D TMA into a
//     kStages-deep ring of 128-byte-swizzled shared memory;
//   * warps 0-3 compute: warps 0/1 take keys 0-31 / 32-63 of the even tiles
//     of a unit, warps 2/3 those of the odd tiles.  For q.k one lane owns one
//     key (the swizzle makes the 8 lanes of each shared-memory phase hit
//     different banks); for P.V one lane owns 4 (D=128) or 2 (D=64) output
//     dims and the probabilities come by warp shuffle;
//   * each warp keeps its own online-softmax state (max, sum, O) per query;
//     the four states are merged at the end of the unit through shared memory.
// Every wait is bounded (same error word and abort flag as the forward kernel).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fwd_kernel.cuh"

namespace attn {
namespace dec {

constexpr int kKeys = 64;        // keys per K/V tile (TMA box rows)
constexpr int kCompWarps = 4;
constexpr int kProdWarp = kCompWarps;
constexpr int kThreads = (kCompWarps + 1) * 32;
constexpr int kStages = 4;
constexpr int kMaxSq = 16;

struct DecParams {
  CUtensorMap tm_k;          // [B * Sk, H, D] 16-bit, box 64 x 1 x 64 rows, 128-B swizzle
  CUtensorMap tm_v;
  const uint16_t* q;         // [B, Sq, H, D]
  void* o;                   // [B, Sq, H, D]
  float* lse;                // [B, H, Sq]
  const int32_t* seqlens;    // [B] valid cache rows, or null (= Sk)
  float* ws_o;               // [splits, B, Sq, H, D] partial O (normalised), splits > 1
  float* ws_lse;             // [splits, B, H, Sq]
  int* err;
  int B, H, Sq, Sk;
  int splits, chunk;         // keys per split: a multiple of kKeys
  int causal;
  float scale_log2;          // scale * log2(e)
  long long timeout_ns;
  int inject;                // fault injection for tests: 1 = block 0 skips its first fill
};

template <int D>
struct DLayout {
  static constexpr int kBlk = kKeys * 128;            // 64 rows x 128 B
  static constexpr int kTile = (D / 64) * kBlk;       // one K or V tile
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kStages * kTile;
  static constexpr int kQOff = 2 * kStages * kTile;   // fp32 [kMaxSq][D], scaled by scale*log2e
  static constexpr int kXOff = kQOff + kMaxSq * D * 4;  // per warp: O [kMaxSq][D], m, l [kMaxSq]
  static constexpr int kXWarp = kMaxSq * (D + 2);       // floats per warp
  static constexpr int kBarOff = kXOff + kCompWarps * kXWarp * 4;
  static constexpr int F = 0, E = kStages, kNumBars = 2 * kStages;  // tile full / empty
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;             // abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

// Unit u = ((b * H) + h) * splits + s  ->  its keys [k0, k1) of sequence b.
struct DUnit {
  int b, h, s, L, k0, ntiles;
};

__device__ __forceinline__ bool dec_unit(const DecParams& p, int u, DUnit& w, bool report) {
  if (u >= p.B * p.H * p.splits) return false;
  w.s = u % p.splits;
  const int bh = u / p.splits;
  w.h = bh % p.H;
  w.b = bh / p.H;
  int L = p.Sk;
  if (p.seqlens) {
    L = __ldg(p.seqlens + w.b);
    if (L < 0 || L > p.Sk) {
      if (report) atomicOr(p.err, kErrBadSeqlens);
      L = 0;
    }
  }
  w.L = L;
  w.k0 = w.s * p.chunk;
  const int k1 = min(L, w.k0 + p.chunk);
  w.ntiles = k1 > w.k0 ? (k1 - w.k0 + kKeys - 1) / kKeys : 0;
  return true;
}

// 16-bit pairs -> fp32 (bf16: the bits are the top half of an fp32).
template <bool BF16>
__device__ __forceinline__ void cvt2(uint32_t w, float& lo, float& hi) {
  if constexpr (BF16) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  } else {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = f.x;
    hi = f.y;
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---------------------------------------------------------------- compute
template <int D, int SQ, bool BF16>
__device__ void dec_compute(const DecParams& p, uint8_t* base, uint32_t bars, const Ctl& ctl) {
  using L = DLayout<D>;
  constexpr int DPL = D / 32;  // output dims per lane in P.V
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int half = warp & 1;   // keys 32*half .. 32*half+31 of a tile
  const int par = warp >> 1;   // tiles of this parity within the unit
  const int r = 32 * half + lane;  // tile row (key) of this lane in q.k
  float* const qs = reinterpret_cast<float*>(base + L::kQOff);
  float* const xw = reinterpret_cast<float*>(base + L::kXOff);
  uint32_t it_base = 0;
  bool alive = true;

  DUnit w;
  for (int u = blockIdx.x; dec_unit(p, u, w, false); u += gridDim.x) {
    // q of this unit, pre-scaled, into shared memory (the previous unit's
    // readers of qs and xw are done: barrier 1 below is reached only after
    // the merge that ends the previous unit)
    ptx::named_bar_sync(1, kCompWarps * 32);
    for (int i = threadIdx.x; i < SQ * D; i += kCompWarps * 32) {
      const int t = i / D, d = i - t * D;
      float x = 0.0f;
      if (t < p.Sq) {
        const uint16_t raw = p.q[((static_cast<long long>(w.b) * p.Sq + t) * p.H + w.h) * D + d];
        x = BF16 ? __uint_as_float(static_cast<uint32_t>(raw) << 16)
                 : __half2float(__ushort_as_half(raw));
      }
      qs[i] = x * p.scale_log2;
    }
    ptx::named_bar_sync(1, kCompWarps * 32);

    float m[SQ], l[SQ], o[SQ][DPL];
#pragma unroll
    for (int t = 0; t < SQ; ++t) {
      m[t] = -INFINITY;
      l[t] = 0.0f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[t][i] = 0.0f;
    }
    // last visible key of query t: L-1, or L-Sq+t when causal
    const int last0 = p.causal ? w.L - p.Sq : w.L - 1;
    for (int j = par; j < w.ntiles; j += 2) {
      const uint32_t it = it_base + j;
      const uint32_t st = it % kStages;
      alive = alive && wait_bar(bars + 8u * (L::F + st), (it / kStages) & 1u, ctl);
      if (__all_sync(0xffffffffu, alive)) {
        const uint8_t* kt = base + L::kKOff + st * L::kTile;
        const uint8_t* vt = base + L::kVOff + st * L::kTile;
        // ---- s_t = q_t . k_r (scaled, log2 units), one key per lane
        uint64_t acc[SQ];  // (even dims, odd dims) partial sums of q_t . k_r
#pragma unroll
        for (int t = 0; t < SQ; ++t) acc[t] = 0ull;
#pragma unroll
        for (int cc = 0; cc < D / 8; ++cc) {
          const int blk = cc >> 3, c = cc & 7;
          const uint4 kw = *reinterpret_cast<const uint4*>(kt + blk * L::kBlk + r * 128 +
                                                           ((c ^ (r & 7)) << 4));
          float kf[8];
          cvt2<BF16>(kw.x, kf[0], kf[1]);
          cvt2<BF16>(kw.y, kf[2], kf[3]);
          cvt2<BF16>(kw.z, kf[4], kf[5]);
          cvt2<BF16>(kw.w, kf[6], kf[7]);
#pragma unroll
          for (int t = 0; t < SQ; ++t) {
            const float4 qa = *reinterpret_cast<const float4*>(qs + t * D + cc * 8);
            const float4 qb = *reinterpret_cast<const float4*>(qs + t * D + cc * 8 + 4);
            acc[t] = ptx::f2_fma(ptx::f2(kf[0], kf[1]), ptx::f2(qa.x, qa.y), acc[t]);
            acc[t] = ptx::f2_fma(ptx::f2(kf[2], kf[3]), ptx::f2(qa.z, qa.w), acc[t]);
            acc[t] = ptx::f2_fma(ptx::f2(kf[4], kf[5]), ptx::f2(qb.x, qb.y), acc[t]);
            acc[t] = ptx::f2_fma(ptx::f2(kf[6], kf[7]), ptx::f2(qb.z, qb.w), acc[t]);
          }
        }
        // ---- online softmax per query over this warp's 32 keys
        const int key = w.k0 + j * kKeys + r;
        float pr[SQ];
#pragma unroll
        for (int t = 0; t < SQ; ++t) {
          const bool vis = key <= last0 + t && key < w.L;
          float s0, s1;
          ptx::f2_split(acc[t], s0, s1);
          const float sv = vis ? s0 + s1 : -INFINITY;
          const float m_new = fmaxf(m[t], warp_max(sv));
          const float m_use = m_new == -INFINITY ? 0.0f : m_new;
          const float alpha = ptx::ex2(m[t] - m_use);
          pr[t] = ptx::ex2(sv - m_use);
          l[t] = l[t] * alpha + warp_sum(pr[t]);
          m[t] = m_new;
#pragma unroll
          for (int i = 0; i < DPL; i += 2) {
            float a0, a1;
            ptx::f2_split(ptx::f2_mul(ptx::f2(o[t][i], o[t][i + 1]), ptx::f2(alpha, alpha)), a0, a1);
            o[t][i] = a0;
            o[t][i + 1] = a1;
          }
        }
        // ---- O_t += p_t V over the 32 keys; lane owns DPL output dims
#pragma unroll 4
        for (int kk = 0; kk < 32; ++kk) {
          const int rr = 32 * half + kk;
          float vf[DPL];
          if constexpr (DPL == 4) {
            const int blk = lane >> 4, c = (lane & 15) >> 1;
            const uint2 vw = *reinterpret_cast<const uint2*>(
                vt + blk * L::kBlk + rr * 128 + ((c ^ (rr & 7)) << 4) + ((lane & 1) << 3));
            cvt2<BF16>(vw.x, vf[0], vf[1]);
            cvt2<BF16>(vw.y, vf[2], vf[3]);
          } else {
            const int c = lane >> 2;
            const uint32_t vw = *reinterpret_cast<const uint32_t*>(
                vt + rr * 128 + ((c ^ (rr & 7)) << 4) + ((lane & 3) << 2));
            cvt2<BF16>(vw, vf[0], vf[1]);
          }
#pragma unroll
          for (int t = 0; t < SQ; ++t) {
            const float pv = __shfl_sync(0xffffffffu, pr[t], kk);
#pragma unroll
            for (int i = 0; i < DPL; i += 2) {
              float a0, a1;
              ptx::f2_split(ptx::f2_fma(ptx::f2(pv, pv), ptx::f2(vf[i], vf[i + 1]),
                                        ptx::f2(o[t][i], o[t][i + 1])), a0, a1);
              o[t][i] = a0;
              o[t][i + 1] = a1;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bars + 8u * (L::E + st));
    }
    it_base += w.ntiles;

    // ---- merge the four warps' states; write the unit's result
    float* const xo = xw + warp * L::kXWarp;
#pragma unroll
    for (int t = 0; t < SQ; ++t) {
#pragma unroll
      for (int i = 0; i < DPL; ++i) xo[t * D + lane * DPL + i] = o[t][i];
      if (lane == 0) {
        xo[kMaxSq * D + t] = m[t];
        xo[kMaxSq * D + kMaxSq + t] = l[t];
      }
    }
    ptx::named_bar_sync(1, kCompWarps * 32);
    for (int i = threadIdx.x; i < p.Sq * D; i += kCompWarps * 32) {
      const int t = i / D, d = i - t * D;
      float mw[kCompWarps], M = -INFINITY;
#pragma unroll
      for (int q = 0; q < kCompWarps; ++q) {
        mw[q] = xw[q * L::kXWarp + kMaxSq * D + t];
        M = fmaxf(M, mw[q]);
      }
      float lsum = 0.0f, acc = 0.0f;
#pragma unroll
      for (int q = 0; q < kCompWarps; ++q) {
        const float f = mw[q] == -INFINITY ? 0.0f : ptx::ex2(mw[q] - M);
        lsum += f * xw[q * L::kXWarp + kMaxSq * D + kMaxSq + t];
        acc += f * xw[q * L::kXWarp + t * D + d];
      }
      const float ov = lsum > 0.0f ? acc / lsum : 0.0f;
      const float lse = lsum > 0.0f ? (M + ptx::lg2(lsum)) * 0.69314718055994531f : -INFINITY;
      const long long orow = (static_cast<long long>(w.b) * p.Sq + t) * p.H + w.h;
      const long long lrow = (static_cast<long long>(w.b) * p.H + w.h) * p.Sq + t;
      if (p.splits == 1) {
        uint16_t* const O = static_cast<uint16_t*>(p.o);
        O[orow * D + d] = BF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(ov))
                               : __half_as_ushort(__float2half_rn(ov));
        if (d == 0) p.lse[lrow] = lse;
      } else {
        const long long so = static_cast<long long>(w.s) * p.B * p.Sq * p.H;
        p.ws_o[(so + orow) * D + d] = ov;
        if (d == 0) p.ws_lse[static_cast<long long>(w.s) * p.B * p.H * p.Sq + lrow] = lse;
      }
    }
  }
}

// ---------------------------------------------------------------- producer
template <int D>
__device__ void dec_produce(const DecParams& p, uint32_t smem, uint32_t bars, const Ctl& ctl) {
  using L = DLayout<D>;
  FillLog<kStages> f;
  f.clear();
  uint32_t it = 0;
  bool ok = true;
  DUnit w;
  for (int u = blockIdx.x; ok && dec_unit(p, u, w, true); u += gridDim.x) {
    for (int j = 0; j < w.ntiles; ++j, ++it) {
      const uint32_t st = it % kStages;
      if (it >= kStages && !wait_bar(bars + 8u * (L::E + st), (it / kStages - 1) & 1u, ctl)) {
        ok = false;  // leave both loops; the copies already issued are waited for below
        break;
      }
      // injected fault (tests only): this fill never arrives, so the consumers'
      // bounded wait runs out and the call reports ATTN_ERR_DEVICE_TIMEOUT
      if (p.inject == 1 && blockIdx.x == 0 && it == 0) continue;
      const uint32_t full = bars + 8u * (L::F + st);
      ptx::mbar_arrive_expect_tx(full, 2 * L::kTile);
      const int row = w.b * p.Sk + w.k0 + j * kKeys;
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk) {
        ptx::tma_load_3d(smem + L::kKOff + st * L::kTile + blk * L::kBlk, &p.tm_k, full,
                         blk * 64, w.h, row);
        ptx::tma_load_3d(smem + L::kVOff + st * L::kTile + blk * L::kBlk, &p.tm_v, full,
                         blk * 64, w.h, row);
      }
      f.last[st] = static_cast<int>(it);
    }
  }
  // no copy may land after the CTA exits: wait for the last fill of each stage
  drain_fills(bars, L::F, f, ctl);
}

template <int D, int SQ, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) attn_decode_kernel(const __grid_constant__ DecParams p) {
  using L = DLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t smem = (raw + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (smem - raw);
  const uint32_t bars = smem + L::kBarOff;
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(base + L::kMiscOff);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i)
      ptx::mbar_init(bars + 8u * i, i >= L::E ? 2u : 1u);  // empty: the two warps of a parity
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kProdWarp && (threadIdx.x & 31) == 0) {
    ptx::tma_prefetch_desc(&p.tm_k);
    ptx::tma_prefetch_desc(&p.tm_v);
  }
  __syncthreads();
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  if (warp < kCompWarps) {
    dec_compute<D, SQ, BF16>(p, base, bars, ctl);
  } else if ((threadIdx.x & 31) == 0) {
    dec_produce<D>(p, smem, bars, ctl);
  }
}

template <int D, int SQ, bool BF16>
cudaError_t launch_decode(const DecParams& p, int grid, cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(&attn_decode_kernel<D, SQ, BF16>);
  static std::atomic<unsigned long long> opted{0};
  const cudaError_t e = smem_opt_in(fn, DLayout<D>::kAlloc, opted);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<DecParams*>(&p)};
  return cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, DLayout<D>::kAlloc, stream);
}

}  // namespace dec
}  // namespace attn
