// Attention backward for sm_103a: dQ, dK, dV from Q, K, V, dO, the forward's
// LSE and D = rowsum(dO * O).
//
// What it computes (per sequence b, head h; scores S = scale Q K^T with the
// causal mask when asked, P = exp(S - LSE) row by row, so P is the forward's
// softmax recomputed from its saved logsumexp):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,
//   dK = scale dS^T Q.
// Page "Multi-Head Attention的计算本质与性能瓶颈", §3.3 reserves this backward
// interface and states that masked connections carry no gradient; the
// formulas are the chain rule through the forward definition.
//
// GB300 mapping: a persistent kernel, one CTA per SM, work unit = (sequence,
// head, 128-key tile).  Keys are the M dimension of every product the unit
// accumulates, so dK and dV stay in tensor memory for the whole unit:
//   TMEM columns: S^T | dP^T | dV | dK (128, 128, D, D); dQ of a step is
//   written over dP^T once dS^T has been consumed, so S^T of the next query
//   tile can be computed while this step's dS is still being formed.
//   * warp 9 (one lane): TMA for the unit's K and V tiles and, per step
//     (128 queries), Q and dO tiles into a 2-stage ring;
//   * warp 8 (one lane): tcgen05.mma
//       S^T  = K Q^T      (SS, K-major / K-major)
//       dP^T = V dO^T     (SS)
//       dV  += P^T dO     (TS: P^T from TMEM, dO MN-major)
//       dK  += dS^T Q     (TS: dS^T from TMEM, Q MN-major)
//       dQ   = dS K       (SS: dS MN-major from shared memory, K MN-major)
//   * warps 0-3: one thread per key (TMEM lane): P^T = 2^(S^T scale log2e -
//     LSE log2e) written back as 16-bit over S^T, then dS^T = P^T (dP^T - D)
//     written as 16-bit over dP^T and into the dO stage (whose dO the dV and
//     dP^T products have finished reading), as the A operand of dQ;
//   * warps 4-7: one thread per query row: dQ of each step is added with
//     fp32 atomics to a [B, H, Sq, D] accumulator; at the end of the unit they
//     write dK (times scale) and dV.
// Every wait is bounded (same error word and abort flag as the forward).
#pragma once

#include <cuda_fp16.h>

#include "fwd_kernel.cuh"

namespace attn {
namespace bwd {

constexpr int kBM = 128;  // keys per unit
constexpr int kBN = 128;  // queries per step
constexpr int kThreads = 320;
constexpr int kDqWarp0 = 4;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kTmemCols = 512;

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // [B*S, H, D] 16-bit, box 64 x 1 x 128, 128-B swizzle
  const float* lse;                      // [B, H, Sq] natural log
  const float* dvec;                     // [B, H, Sq]: sum_d dO * O
  float* dq_acc;                         // [B, H, Sq, D] fp32, zero on entry
  void* dk;                              // [B, Sk, H, D]
  void* dv;
  int* err;
  int B, H, Sq, Sk, causal;
  float scale, scale_log2;
  long long timeout_ns;
};

template <int D>
struct BLayout {
  static constexpr int kBlk = 16384;             // 128 rows x 128 B swizzle block
  static constexpr int kTile = (D / 64) * kBlk;  // one 128-row tile of K, V, Q or dO
  static constexpr int kDoStage = 2 * kBlk;      // a dO stage also holds dS (128 x 128 16-bit)
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTile;
  static constexpr int kQOff = 2 * kTile;              // 2 stages
  static constexpr int kDoOff = kQOff + 2 * kTile;     // 2 stages of kDoStage
  static constexpr int kStatOff = kDoOff + 2 * kDoStage;  // [2][2][128]: -LSE*log2e, D
  static constexpr int kBarOff = kStatOff + 2 * 2 * kBN * 4;
  enum : int {
    KVF = 0, KVE, QF0, QF1, QE0, QE1, SF, DPF, PR, DVD, DSR, DQF, DQE, OF, AE, ST0, ST1, DONE,
    kNumBars
  };
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;  // tmem base, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
};

// ---------------------------------------------------------------- helpers
__host__ __device__ constexpr uint32_t idesc_ab(bool bf16, int M, int N, bool a_mn, bool b_mn) {
  return ptx::idesc_f16_f32acc(bf16, M, N, b_mn) | ((a_mn ? 1u : 0u) << 15);
}

// generic-proxy shared-memory writes -> later tensor-core (async proxy) reads
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {"
      "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16"
      "};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// dst[0..3] += v (fp32, relaxed, no return value: the warp does not wait)
__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};"
               ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

template <bool BF16>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
  if constexpr (BF16) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  } else {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = f.x;
    hi = f.y;
  }
}

// Work unit u -> (b, h, key tile kt); units of one head are consecutive, key
// tiles in increasing order (under causal the first key tiles see the most
// query tiles).  Steps: query tiles i0 .. nq-1.
struct BUnit {
  int b, h, kt, i0, n;
};

__device__ __forceinline__ bool bwd_unit(const BwdParams& p, int k, BUnit& w) {
  const int nk = (p.Sk + kBM - 1) / kBM;
  const int u = unit_of(k);
  if (u >= p.B * p.H * nk) return false;
  const int bh = u / nk;
  w.kt = u - bh * nk;
  w.b = bh / p.H;
  w.h = bh - w.b * p.H;
  const int nq = (p.Sq + kBN - 1) / kBN;
  // causal (top-left): query tile i has a row >= every key of tile kt from i = kt on
  w.i0 = p.causal ? w.kt : 0;
  w.n = max(0, nq - w.i0);
  return true;
}

// Steps of this CTA in order, across its units (units without steps skipped).
struct StepIter {
  int k;     // unit counter of this CTA
  BUnit w;
  int j;     // step within the unit
  bool ok;
  __device__ __forceinline__ void start(const BwdParams& p) {
    k = 0;
    j = 0;
    ok = bwd_unit(p, k, w);
    while (ok && w.n == 0) ok = bwd_unit(p, ++k, w);
  }
  __device__ __forceinline__ void next(const BwdParams& p) {
    if (++j < w.n) return;
    j = 0;
    do ok = bwd_unit(p, ++k, w);
    while (ok && w.n == 0);
  }
};

// ------------------------------------------------------------- P and dS
template <int D, bool BF16>
__device__ void ds_role(const BwdParams& p, uint32_t tmem, uint32_t smem, uint8_t* base,
                        uint32_t bars, const Ctl& ctl) {
  using L = BLayout<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = warp * 32 + lane;  // key row of this thread = TMEM lane
  const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tS = tmem + lane_bits + L::kColS;
  const uint32_t tDP = tmem + lane_bits + L::kColDP;
  auto bar = [&](int i) { return bars + 8u * i; };
  float* const stats = reinterpret_cast<float*>(base + L::kStatOff);
  const float log2e = 1.4426950408889634f;

  StepIter cur;
  cur.start(p);
  // statistics of the first step (each thread: column r of the query tile)
  float nl_next = 0.0f, dv_next = 0.0f;
  auto fetch = [&](const StepIter& it) {
    const int q = (it.w.i0 + it.j) * kBN + r;
    nl_next = 0.0f;
    dv_next = 0.0f;
    if (q < p.Sq) {
      const long long idx = (static_cast<long long>(it.w.b) * p.H + it.w.h) * p.Sq + q;
      const float l = __ldg(p.lse + idx);
      nl_next = l == -INFINITY ? -INFINITY : -l * log2e;
      dv_next = __ldg(p.dvec + idx);
    }
  };
  if (cur.ok) fetch(cur);
  for (uint32_t g = 0; cur.ok; ++g) {
    const BUnit w = cur.w;
    const int i = w.i0 + cur.j;
    // ---- publish this step's statistics, prefetch the next step's
    float* const st = stats + (g & 1u) * 2 * kBN;
    st[r] = nl_next;
    st[kBN + r] = dv_next;
    StepIter nxt = cur;
    nxt.next(p);
    if (nxt.ok) fetch(nxt);
    ptx::mbar_arrive(bar(L::ST0 + (g & 1u)));
    if (!wait_bar_warp(bar(L::ST0 + (g & 1u)), (g >> 1) & 1u, ctl)) return;

    const int key = w.kt * kBM + r;
    const int qb = i * kBN;
    // columns c (query qb + c) visible to this key: c >= cmin and qb + c < Sq
    const int cmin = p.causal ? key - qb : 0;
    const int cmax = p.Sq - qb - 1;
    const bool row_ok = key < p.Sk;
    const bool full = row_ok && cmin <= 0 && cmax >= kBN - 1;

    // ---- P^T = 2^(S^T * scale * log2e - LSE * log2e), 16-bit, over S^T
    if (!wait_bar_warp(bar(L::SF), g & 1u, ctl)) return;
    ptx::tc_fence_after();
    uint32_t pk[64];
#pragma unroll
    for (int c0 = 0; c0 < kBN; c0 += 32) {
      uint32_t s[32];
      ptx::tmem_ld_x32(tS + c0, s);
      const float2* nl = reinterpret_cast<const float2*>(st + c0);
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const float2 n2 = nl[c / 2];
        float x0, x1;
        ptx::f2_split(ptx::f2_fma(ptx::f2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])),
                                  ptx::f2(p.scale_log2, p.scale_log2), ptx::f2(n2.x, n2.y)),
                      x0, x1);
        float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
        if (!full) {
          const int cc = c0 + c;
          if (!row_ok || cc < cmin || cc > cmax) p0 = 0.0f;
          if (!row_ok || cc + 1 < cmin || cc + 1 > cmax) p1 = 0.0f;
        }
        pk[(c0 + c) / 2] = ptx::pack2<BF16>(p0, p1);
      }
      uint32_t chunk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) chunk[c] = pk[c0 / 2 + c];
      tmem_st_x16(tS + c0 / 2, chunk);
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(L::PR));

    // ---- dS^T = P^T (dP^T - D), 16-bit, over dP^T and into the dO stage
    if (!wait_bar_warp(bar(L::DPF), g & 1u, ctl)) return;
    if (!wait_bar_warp(bar(L::DVD), g & 1u, ctl)) return;  // dO of this stage consumed
    ptx::tc_fence_after();
    uint8_t* const ds_tile = base + L::kDoOff + (g & 1u) * L::kDoStage;
#pragma unroll
    for (int c0 = 0; c0 < kBN; c0 += 32) {
      uint32_t dp[32];
      ptx::tmem_ld_x32(tDP + c0, dp);
      const float2* dd = reinterpret_cast<const float2*>(st + kBN + c0);
      uint32_t dk[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float p0, p1;
        unpack2<BF16>(pk[(c0 + c) / 2], p0, p1);
        const float2 d2 = dd[c / 2];
        float a, b;
        ptx::f2_split(ptx::f2_mul(ptx::f2(p0, p1),
                                  ptx::f2_add(ptx::f2(__uint_as_float(dp[c]),
                                                      __uint_as_float(dp[c + 1])),
                                              ptx::f2(-d2.x, -d2.y))),
                      a, b);
        dk[c / 2] = ptx::pack2<BF16>(a, b);
      }
      tmem_st_x16(tDP + c0 / 2, dk);
      // shared memory: row r (key), queries c0 .. c0+31 = 4 chunks of 16 B in the
      // 128-B swizzled block of queries 64 * (c0 / 64) .. +63
      uint8_t* const row = ds_tile + (c0 >> 6) * L::kBlk + r * 128;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int chunk = ((c0 & 63) >> 3) + q4;
        *reinterpret_cast<uint4*>(row + ((chunk ^ (r & 7)) << 4)) =
            make_uint4(dk[4 * q4], dk[4 * q4 + 1], dk[4 * q4 + 2], dk[4 * q4 + 3]);
      }
    }
    ptx::tmem_wait_st();
    fence_proxy_async_smem();
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(L::DSR));
    cur = nxt;
  }
  (void)smem;
}

// -------------------------------------------------- dQ and the dK/dV epilogue
template <int D, bool BF16>
__device__ void dq_role(const BwdParams& p, uint32_t tmem, uint32_t bars, const Ctl& ctl) {
  using L = BLayout<D>;
  const int warp = threadIdx.x >> 5;
  const int quarter = warp & 3;
  const int lane = threadIdx.x & 31;
  const int r = quarter * 32 + lane;  // query row (dQ) / key row (dK, dV) = TMEM lane
  const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint16_t* const DK = static_cast<uint16_t*>(p.dk);
  uint16_t* const DV = static_cast<uint16_t*>(p.dv);
  uint32_t g = 0, u_cnt = 0;
  BUnit w;
  for (int k = 0; bwd_unit(p, k, w); ++k) {
    const int key = w.kt * kBM + r;
    const bool key_ok = key < p.Sk;
    const long long krow = (static_cast<long long>(w.b) * p.Sk + key) * p.H + w.h;
    if (w.n == 0) {  // no query sees these keys: dK = dV = 0
      if (key_ok) {
        uint4* a = reinterpret_cast<uint4*>(DK + krow * D);
        uint4* b = reinterpret_cast<uint4*>(DV + krow * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) a[c] = b[c] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    for (int j = 0; j < w.n; ++j, ++g) {
      if (!wait_bar_warp(bar(L::DQF), g & 1u, ctl)) return;
      ptx::tc_fence_after();
      uint32_t v[D];
      if constexpr (D == 128) {
        ptx::tmem_ld_x128(tmem + lane_bits + L::kColDP, v);
      } else {
        ptx::tmem_ld_x64(tmem + lane_bits + L::kColDP, v);
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::DQE));
      const int q = (w.i0 + j) * kBN + r;
      if (q < p.Sq) {
        float* dst = p.dq_acc + ((static_cast<long long>(w.b) * p.H + w.h) * p.Sq + q) * D;
#pragma unroll
        for (int c = 0; c < D / 4; ++c)
          red_add_v4(dst + 4 * c, __uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                     __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
      }
    }
    // ---- dK (times scale) and dV of this key tile
    if (!wait_bar_warp(bar(L::OF), u_cnt & 1u, ctl)) return;
    ++u_cnt;
    ptx::tc_fence_after();
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t col = which == 0 ? L::kColDK : L::kColDV;
      const float mul = which == 0 ? p.scale : 1.0f;
      uint16_t* const out = which == 0 ? DK : DV;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        ptx::tmem_ld_x32(tmem + lane_bits + col + c0, v);
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = ptx::pack2<BF16>(__uint_as_float(v[2 * c]) * mul,
                                   __uint_as_float(v[2 * c + 1]) * mul);
        if (key_ok) {
          uint4* dst = reinterpret_cast<uint4*>(out + krow * D + c0);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
      }
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(L::AE));
  }
}

// -------------------------------------------------------------------- MMA
template <int D, bool BF16>
__device__ void mma_loop(const BwdParams& p, uint32_t smem, uint32_t tmem, uint32_t bars,
                         const Ctl& ctl) {
  using L = BLayout<D>;
  constexpr uint32_t kIdS = idesc_ab(BF16, kBM, kBN, false, false);   // S^T, dP^T
  constexpr uint32_t kIdAcc = idesc_ab(BF16, kBM, D, false, true);    // dV, dK (A from TMEM)
  constexpr uint32_t kIdDq = idesc_ab(BF16, kBN, D, true, true);      // dQ
  auto bar = [&](int i) { return bars + 8u * i; };
  const uint64_t dK_kmaj = ptx::desc_sw128(smem + L::kKOff, 16, 1024);
  const uint64_t dV_kmaj = ptx::desc_sw128(smem + L::kVOff, 16, 1024);
  const uint64_t dK_mn = ptx::desc_sw128(smem + L::kKOff, L::kBlk, 1024);
  const uint32_t tS = tmem + L::kColS, tDP = tmem + L::kColDP;
  const uint32_t tDV = tmem + L::kColDV, tDK = tmem + L::kColDK;
  uint32_t g = 0, kv_cnt = 0, u_cnt = 0;
  // S^T(g) = K Q_g^T into the S^T columns (Q_g of ring stage g % 2)
  auto issue_s = [&](uint32_t gg) -> bool {
    const uint32_t st = gg & 1u;
    if (!wait_bar(bar(L::QF0 + st), (gg >> 1) & 1u, ctl)) return false;
    ptx::tc_fence_after();
    const uint64_t dQ_kmaj = ptx::desc_sw128(smem + L::kQOff + st * L::kTile, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint32_t off = ((ks >> 2) * L::kBlk + (ks & 3) * 32) >> 4;
      ptx::mma_ss(tS, dK_kmaj + off, dQ_kmaj + off, kIdS, ks > 0 ? 1u : 0u);
    }
    ptx::mma_commit(bar(L::SF));
    return true;
  };
  // Order per step g (one issuing thread, so tensor memory reuse follows
  // issue order): S^T(g) [issued during step g-1 when in the same unit],
  // dP^T(g) once dQ(g-1) has been read out of the dP^T columns, dV(g) once P(g)
  // is in TMEM, S^T(g+1) (P(g) is consumed by dV(g) before it), then dK(g) and
  // dQ(g) = dS K into the dP^T columns once dS(g) is ready.
  BUnit w;
  for (int k = 0; bwd_unit(p, k, w); ++k) {
    if (w.n == 0) continue;
    if (!wait_bar(bar(L::KVF), kv_cnt & 1u, ctl)) return;
    ++kv_cnt;
    ptx::tc_fence_after();
    if (!issue_s(g)) return;
    for (int j = 0; j < w.n; ++j, ++g) {
      const uint32_t st = g & 1u;
      const uint32_t qbase = smem + L::kQOff + st * L::kTile;
      const uint32_t dobase = smem + L::kDoOff + st * L::kDoStage;
      if (g > 0 && !wait_bar(bar(L::DQE), (g - 1) & 1u, ctl)) return;  // dP^T columns free
      ptx::tc_fence_after();
      const uint64_t dDo_kmaj = ptx::desc_sw128(dobase, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {  // dP^T = V dO^T
        const uint32_t off = ((ks >> 2) * L::kBlk + (ks & 3) * 32) >> 4;
        ptx::mma_ss(tDP, dV_kmaj + off, dDo_kmaj + off, kIdS, ks > 0 ? 1u : 0u);
      }
      ptx::mma_commit(bar(L::DPF));
      if (!wait_bar(bar(L::PR), g & 1u, ctl)) return;
      if (j == 0 && u_cnt > 0 && !wait_bar(bar(L::AE), (u_cnt - 1) & 1u, ctl)) return;
      ptx::tc_fence_after();
      const uint64_t dDo_mn = ptx::desc_sw128(dobase, L::kBlk, 1024);
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks)  // dV += P^T dO
        ptx::mma_ts(tDV, tS + ks * 8, dDo_mn + ((ks * 2048) >> 4), kIdAcc,
                    (j > 0 || ks > 0) ? 1u : 0u);
      ptx::mma_commit(bar(L::DVD));
      if (j + 1 < w.n && !issue_s(g + 1)) return;  // next query tile of this unit
      if (!wait_bar(bar(L::DSR), g & 1u, ctl)) return;
      ptx::tc_fence_after();
      const uint64_t dQ_mn = ptx::desc_sw128(qbase, L::kBlk, 1024);
      const uint64_t dDs_mn = ptx::desc_sw128(dobase, L::kBlk, 1024);
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks)  // dK += dS^T Q
        ptx::mma_ts(tDK, tDP + ks * 8, dQ_mn + ((ks * 2048) >> 4), kIdAcc,
                    (j > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < kBM / 16; ++ks)  // dQ = dS K (over this tile's keys)
        ptx::mma_ss(tDP, dDs_mn + ((ks * 2048) >> 4), dK_mn + ((ks * 2048) >> 4), kIdDq,
                    ks > 0 ? 1u : 0u);
      ptx::mma_commit(bar(L::DQF));
      ptx::mma_commit(bar(L::QE0 + st));
      if (j == w.n - 1) {
        ptx::mma_commit(bar(L::OF));
        ptx::mma_commit(bar(L::KVE));
      }
    }
    ++u_cnt;
  }
}

// ------------------------------------------------------------------- load
template <int D>
__device__ void load_loop(const BwdParams& p, uint32_t smem, uint32_t bars, const Ctl& ctl,
                          uint32_t& g, uint32_t& kv_cnt) {
  using L = BLayout<D>;
  auto bar = [&](int i) { return bars + 8u * i; };
  BUnit w;
  for (int k = 0; bwd_unit(p, k, w); ++k) {
    if (w.n == 0) continue;
    if (kv_cnt > 0 && !wait_bar(bar(L::KVE), (kv_cnt - 1) & 1u, ctl)) return;
    ptx::mbar_arrive_expect_tx(bar(L::KVF), 2 * L::kTile);
    const int krow = w.b * p.Sk + w.kt * kBM;
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk) {
      ptx::tma_load_3d(smem + L::kKOff + blk * L::kBlk, &p.tm_k, bar(L::KVF), blk * 64, w.h, krow);
      ptx::tma_load_3d(smem + L::kVOff + blk * L::kBlk, &p.tm_v, bar(L::KVF), blk * 64, w.h, krow);
    }
    ++kv_cnt;
    for (int j = 0; j < w.n; ++j, ++g) {
      const uint32_t st = g & 1u;
      if (g >= 2 && !wait_bar(bar(L::QE0 + st), ((g >> 1) - 1) & 1u, ctl)) return;
      ptx::mbar_arrive_expect_tx(bar(L::QF0 + st), 2 * L::kTile);
      const int qrow = w.b * p.Sq + (w.i0 + j) * kBN;
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk) {
        ptx::tma_load_3d(smem + L::kQOff + st * L::kTile + blk * L::kBlk, &p.tm_q,
                         bar(L::QF0 + st), blk * 64, w.h, qrow);
        ptx::tma_load_3d(smem + L::kDoOff + st * L::kDoStage + blk * L::kBlk, &p.tm_do,
                         bar(L::QF0 + st), blk * 64, w.h, qrow);
      }
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
  using L = BLayout<D>;
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
    for (int i = 0; i < L::kNumBars; ++i) {
      const bool many = i == L::PR || i == L::DSR || i == L::DQE || i == L::AE ||
                        i == L::ST0 || i == L::ST1;
      ptx::mbar_init(bars + 8u * i, many ? 128u : 1u);
    }
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
    ptx::tma_prefetch_desc(&p.tm_do);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};

  if (warp < kDqWarp0) {
    ds_role<D, BF16>(p, tmem, smem, base, bars, ctl);
  } else if (warp < kMmaWarp) {
    dq_role<D, BF16>(p, tmem, bars, ctl);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      mma_loop<D, BF16>(p, smem, tmem, bars, ctl);
      const uint32_t done = bars + 8u * L::DONE;
      ptx::mma_commit(done);
      wait_bar(done, 0, ctl, false);
    }
  } else if (lane == 0) {
    uint32_t g = 0, kv_cnt = 0;
    load_loop<D>(p, smem, bars, ctl, g, kv_cnt);
    // no TMA write may land after the CTA exits
    if (kv_cnt > 0) wait_bar(bars + 8u * L::KVF, (kv_cnt - 1) & 1u, ctl, false);
    for (uint32_t st = 0; st < 2 && st < g; ++st) {
      const uint32_t last = st + ((g - 1 - st) / 2) * 2;
      wait_bar(bars + 8u * (L::QF0 + st), (last >> 1) & 1u, ctl, false);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------ pre- and post-processing
// D[b, h, q] = sum_d dO[b, q, h, d] * O[b, q, h, d] (fp32), one warp per row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                           const uint16_t* __restrict__ dout,
                                                           float* __restrict__ dvec, int B, int H,
                                                           int Sq) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(B) * Sq * H) return;
  const int lane = threadIdx.x & 31;
  const int h = static_cast<int>(row % H);
  const long long bq = row / H;
  const int q = static_cast<int>(bq % Sq);
  const int b = static_cast<int>(bq / Sq);
  constexpr int PER = D / 32;  // 2 or 4 elements per lane
  float acc = 0.0f;
  const uint16_t* a = o + row * D + lane * PER;
  const uint16_t* c = dout + row * D + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2) {
    float x0, x1, y0, y1;
    unpack2<BF16>(*reinterpret_cast<const uint32_t*>(a + i), x0, x1);
    unpack2<BF16>(*reinterpret_cast<const uint32_t*>(c + i), y0, y1);
    acc = fmaf(x0, y0, fmaf(x1, y1, acc));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) dvec[(static_cast<long long>(b) * H + h) * Sq + q] = acc;
}

// dQ[b, q, h, :] = scale * acc[b, h, q, :] in the input dtype.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const float* __restrict__ acc,
                                                            uint16_t* __restrict__ dq, int B,
                                                            int H, int Sq, float scale) {
  const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;  // pair index
  const long long n = static_cast<long long>(B) * H * Sq * (D / 2);
  if (i >= n) return;
  const int d2 = static_cast<int>(i % (D / 2));
  const long long row = i / (D / 2);  // (b * H + h) * Sq + q
  const int q = static_cast<int>(row % Sq);
  const long long bh = row / Sq;
  const int h = static_cast<int>(bh % H);
  const int b = static_cast<int>(bh / H);
  const float2 v = reinterpret_cast<const float2*>(acc)[i];
  const uint32_t pk = ptx::pack2<BF16>(v.x * scale, v.y * scale);
  reinterpret_cast<uint32_t*>(dq)[((static_cast<long long>(b) * Sq + q) * H + h) * (D / 2) + d2] =
      pk;
}

template <int D, bool BF16>
cudaError_t launch_bwd(const BwdParams& p, const uint16_t* o, const uint16_t* dout,
                       float* dvec, uint16_t* dq, int grid, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.B) * p.Sq * p.H;
  cudaError_t e = cudaMemsetAsync(p.dq_acc, 0, static_cast<size_t>(rows) * D * sizeof(float),
                                  stream);
  if (e != cudaSuccess) return e;
  attn_bwd_pre_kernel<D, BF16><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      o, dout, dvec, p.B, p.H, p.Sq);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const void* fn = reinterpret_cast<const void*>(&attn_bwd_kernel<D, BF16>);
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, BLayout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<BwdParams*>(&p)};
  e = cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, BLayout<D>::kAlloc, stream);
  if (e != cudaSuccess) return e;
  const long long pairs = rows * (D / 2);
  attn_bwd_post_kernel<D, BF16><<<static_cast<unsigned>((pairs + 255) / 256), 256, 0, stream>>>(
      p.dq_acc, dq, p.B, p.H, p.Sq, p.scale);
  return cudaGetLastError();
}

}  // namespace bwd
}  // namespace attn
