// Fused attention forward on CTA pairs (clusters of 2) with 2-SM tcgen05 MMAs
// and a triple-buffered score tile; head dim D = 64 or 128.
//
// Same computation as attn_fwd_kernel (see fwd_kernel.cuh for the definition
// and its sources).  What changes is how the tensor cores are fed:
//   * One M = 256 tcgen05.mma (cta_group::2), issued by the even CTA of the
//     pair, covers 128 query rows of each CTA.  Each CTA reads only half of
//     every K/V tile from shared memory (K: 64 of the 128 keys; V: D/2 of the
//     D head-dim columns) and loads only that half with TMA.
//   * Each CTA owns one 128-row query tile and three S buffers in tensor
//     memory, so S(G+1) and S(G+2) = Q K^T are ready while the softmax works
//     on S(G): the only ordering left is P(G) -> O += P(G) V(G) -> S(G+3)
//     (P(G) is written over S(G), so S(G+3) reuses that buffer once P(G) has
//     been consumed).  With two buffers the softmax waited for that chain.
//   * TMEM per CTA: S buffers 0, 1, 2 (128 columns each) | O (D columns).
//   * Two threads of the even CTA issue the MMAs: one the S = Q K^T products,
//     one the O += P V products.  A single issuing thread was the bottleneck
//     (each barrier poll and each 2-SM MMA issue costs it tens to hundreds of
//     cycles), and the two streams only meet at "PV done": S(G) may overwrite
//     the buffer of P(G-3) once O += P(G-3) V(G-3) has completed.
// Steps are numbered globally per pair (G = steps of earlier units + j), so
// buffer G % 3 and the phase of every per-step barrier carry across units.
// Work unit = (sequence, head, 256 query rows): CTA r of the pair holds rows
// 256u + 128r .. +127.  Both CTAs' softmax warps run every K/V step of the pair
// (masking what their own rows cannot see) and signal the even CTA, whose two
// MMA threads issue all MMAs.  Barriers: Q/K/V "full" and "P ready"
// live in the even CTA (the odd CTA's copies complete their bytes there, its
// softmax warps arrive there); "S ready", "PV done", "O ready" and the "empty"
// barriers are multicast to both CTAs.
#pragma once

#include "fwd_kernel.cuh"

namespace attn {
namespace pair {

constexpr int kUR = 2 * kBM;    // query rows per pair unit
constexpr int kNBuf = 3;        // S buffers in tensor memory
constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quarter: column halves 0 and 1
constexpr int kEpiWarps = 4;    // one per TMEM lane quarter: O -> global memory
constexpr int kWarps = kSoftmaxWarps + 3 + kEpiWarps;  // + S-MMA, load, PV-MMA, epilogue
constexpr int kPairThreads = kWarps * 32;
constexpr int kPMma = 8;        // issues S = Q K^T; allocates tensor memory
constexpr int kPLoad = 9;
constexpr int kPPv = 10;        // issues O += P V
constexpr int kPEpi = 11;       // first epilogue warp (11..14 cover the four lane quarters)

template <int D>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kStages = D == 128 ? 5 : 8;  // K/V ring depth (half tiles)
  static constexpr int kBlk = 16384;                // 128 rows x 128 B swizzle block
  static constexpr int kQTile = (D / 64) * kBlk;    // 128 rows x D
  static constexpr int kKBlk = 8192;                // 64 keys x 64 dims
  static constexpr int kKHalf = (D / 64) * kKBlk;   // 64 keys x D
  // 128 keys x D/2 dims: one 128-byte-swizzled block (D = 128) or rows of 64 B
  // in 64-byte swizzle atoms (D = 64)
  static constexpr int kVHalf = 128 * D;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQTile;
  static constexpr int kVOff = kKOff + kStages * kKHalf;
  static constexpr int kBarOff = kVOff + kStages * kVHalf;
  static constexpr int QF = 0, QE = 1, KF = 2, KE = KF + kStages, VF = KE + kStages,
                       VE = VF + kStages, SF = VE + kStages, PF = SF + kNBuf,
                       PVD = PF + kNBuf, OF = PVD + kNBuf, DONE = OF + 1, LDONE = DONE + 1,
                       LR = LDONE + 1, LF = LR + 1, OFREE = LF + 1, DR = OFREE + 1,
                       kNumBars = DR + 2;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
  // the odd CTA's loader record (last Q fill, last K / V fill per stage),
  // written into the even CTA before it arrives on LDONE
  static constexpr int kFillOff = kMiscOff + 16;
  static constexpr int kFillWords = 1 + 2 * kStages;
  // softmax exchange between the two warps of a row: per-step partial maxima
  // (two step parities x two halves x 128 rows) and the final row sums
  static constexpr int kXMaxOff = kFillOff + (kFillWords * 4 + 15) / 16 * 16;
  static constexpr int kXSumOff = kXMaxOff + 2 * 2 * 128 * 4;
  // 1 / l of each row of the last finished unit, for the epilogue warps
  static constexpr int kInvLOff = kXSumOff + 2 * 128 * 2 * 4;
  // Two unit descriptors for the softmax warps (unit k in slot k % 2), written
  // one unit ahead by the epilogue warps: a header and each row's visible keys.
  static constexpr int kDescOff = kInvLOff + 128 * 4;
  static constexpr int kDescBytes = 32 + 2 * 128 * 4;
  static constexpr int kBytes = kDescOff + 2 * kDescBytes;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS = 0, kColO = kNBuf * 128;  // O: D columns
  // Per-step barriers come in threes indexed by G % 3; barrier G % 3 completes
  // its phase G / 3 for step G.  No barrier can run two phases ahead of a
  // waiter:
  //   S ready (SF):  S(G+3) needs O += P(G) V(G), which needs the softmax to
  //                  have consumed S(G);
  //   P ready (PF):  a softmax warp can be two steps ahead of the others
  //                  (S(G+1), S(G+2) may be computed), never three (S(G+3)
  //                  needs every warp's P(G));
  //   PV done (PVD): PV(G+3) needs S(G+3), which the S thread issues only after
  //                  waiting for PV(G); the softmax waits for PV(G-1) before
  //                  giving P(G), which PV(G+2) needs.
  static constexpr uint32_t kPArrivals = 2 * kSoftmaxWarps;  // every softmax warp, both CTAs
  static constexpr uint32_t kDoneArrivals = 2;   // both MMA threads
  // End of a unit: the softmax warps of column half 0 publish 1 / l (LR, one
  // arrival per warp); the epilogue warps, having read it, free the slot (LF)
  // and, having read O out of tensor memory, let the next unit's first
  // O += P V overwrite it (OFREE, in the even CTA: both CTAs' epilogue warps).
  static constexpr uint32_t kLrArrivals = kSoftmaxWarps / 2;
  static constexpr uint32_t kLfArrivals = kEpiWarps;
  static constexpr uint32_t kOFreeArrivals = 2 * kEpiWarps;
  // Descriptor k is complete (DR + k % 2, phase k / 2 % 2) when every epilogue
  // warp has written its rows.  The slot of unit k is written again for unit
  // k + 2 only in the epilogue's iteration k + 1, which follows its wait for
  // LR of unit k; the softmax warps read descriptor k at the start of unit k,
  // before they publish LR of unit k.  So no slot or phase is overwritten
  // before it is read.
  static constexpr uint32_t kDrArrivals = kEpiWarps;
};

// Same as wait_bar, but with cluster-scope acquire (used where the peer CTA arrives).
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, const Ctl& c,
                                                 bool honor_abort = true) {
  if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (honor_abort && *c.abort_flag) return false;
      if (static_cast<long long>(ptx::global_timer_ns() - t0) > c.timeout_ns) {
        *c.abort_flag = 1;
        atomicOr(c.err, kErrTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ int q0_of(const Unit& w, int r) { return w.q0 + r * kBM; }

// Decodes the k-th unit of this pair; n = K/V steps of the pair (max over the
// two CTAs' query tiles).
__device__ __forceinline__ bool decode_pair(const FwdParams& p, int k, Cursor& c, Unit& w,
                                            int& n, bool report) {
  const int g = static_cast<int>(gridDim.x) / 2;
  const int cl = static_cast<int>(blockIdx.x) / 2;
  if (!decode_rows<kUR>(p, slot_unit(p, k, g, cl), c, w, report)) return false;
  int lo0, hi0, lo1, hi1;
  tile_keys(p, w, q0_of(w, 0), lo0, hi0);
  tile_keys(p, w, q0_of(w, 1), lo1, hi1);
  // the pair shares every K/V tile: from the first to the last that either CTA's rows need
  int j0 = 0x7fffffff, j1 = 0;
  if (hi0 > lo0) {
    j0 = lo0;
    j1 = hi0;
  }
  if (hi1 > lo1) {
    j0 = min(j0, lo1);
    j1 = max(j1, hi1);
  }
  w.j0 = j1 > 0 ? j0 : 0;
  n = max(0, j1 - w.j0);
  return true;
}

// ---------------------------------------------------------------- softmax
// One K/V step of the online softmax for half of a query row: this thread owns
// keys [64h, 64h+64) of S (the other half sits with the thread of the same lane
// in warp w ^ 4, on the same SM sub-partition and TMEM lane quarter).  The two
// halves exchange their partial maxima through shared memory at a named
// barrier, so both take the same running max and rescale decisions; each
// writes its 32 columns of P and rescales its 64 columns of O.  Masking: keys
// c of this half with c < lo or c > limit are invisible (both already local to
// the half).  Returns false if the wait before a rescale of O gave up (after
// the step's named barrier).
template <int D, bool BF16>
__device__ __forceinline__ bool softmax_half_step(uint32_t tS, uint32_t tP, uint32_t tO, int lo,
                                                  int limit,
                                                  float cl, bool scale_pos, bool first,
                                                  RowState& st, float* x_mine,
                                                  const float* x_other, uint32_t bar_id,
                                                  uint32_t pvd_bar, uint32_t pvd_parity,
                                                  const Ctl& ctl) {
  uint32_t r[64];
  ptx::tmem_ld_x64(tS, r);
  float cle = cl;
  if (!scale_pos) {  // scale <= 0: scale first so that "max" stays a max
#pragma unroll
    for (int c = 0; c < 64; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * cl);
    cle = 1.0f;
  }
  if (limit < 63 || lo > 0) {
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (c > limit || c < lo) r[c] = __float_as_uint(-INFINITY);
  }
  float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
  for (int c = 0; c < 64; c += 8) {
    mx0 = ptx::max3(mx0, __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
    mx1 = ptx::max3(mx1, __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
    mx2 = ptx::max3(mx2, __uint_as_float(r[c + 4]), __uint_as_float(r[c + 5]));
    mx3 = ptx::max3(mx3, __uint_as_float(r[c + 6]), __uint_as_float(r[c + 7]));
  }
  const float r_max = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));  // this half's largest score
  const float m_part = r_max * cle;
  *x_mine = m_part;
  // Both halves have read their S columns (tcgen05.ld waited) before either
  // overwrites the first 64 columns of the buffer with P.
  ptx::tc_fence_before();
  ptx::named_bar_sync(bar_id, 64);
  ptx::tc_fence_after();
  const float m_tile = fmaxf(m_part, *x_other);
  const float m_new = fmaxf(st.m, m_tile);
  const bool rescale = m_new > st.m + kRescaleLog2;  // always true on the first tile
  const float m_use = rescale ? m_new : st.m;
  const float m_safe = (m_use == -INFINITY) ? 0.0f : m_use;
  const float alpha = rescale ? ptx::ex2(st.m - m_safe) : 1.0f;
  st.m = m_use;

  const float nm = -m_safe;
  float la = 0.f, lb = 0.f, lc = 0.f, ld = 0.f;
  uint32_t pk[32];
#pragma unroll
  for (int c = 0; c < 64; c += 4) {
    const float x0 = fmaf(__uint_as_float(r[c]), cle, nm);
    const float x1 = fmaf(__uint_as_float(r[c + 1]), cle, nm);
    const float x2 = fmaf(__uint_as_float(r[c + 2]), cle, nm);
    const float x3 = fmaf(__uint_as_float(r[c + 3]), cle, nm);
    const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1), p2 = ptx::ex2(x2), p3 = ptx::ex2(x3);
    la += p0;
    lb += p1;
    lc += p2;
    ld += p3;
    pk[c / 2] = ptx::pack2<BF16>(p0, p1);
    pk[c / 2 + 1] = ptx::pack2<BF16>(p2, p3);
  }
  ptx::tmem_st_x32(tP, pk);
  // O is normalised by the exact sum plus the rounding error of this half's
  // largest value (computed exactly as in the loop, so the correction cancels
  // that value's rounding in P.V): the largest values are the ones whose
  // rounding would otherwise show in a peaked row, and the per-element loop
  // keeps a single sum.
  const float p_big = ptx::ex2(fmaf(r_max, cle, nm));
  const float sum = (la + lb) + (lc + ld);
  st.l_x = st.l_x * alpha + sum;
  st.l_p = st.l_p * alpha + (sum + (round16<BF16>(p_big) - p_big));

  if (!first && __any_sync(0xffffffffu, rescale)) {
    if (!wait_bar_warp(pvd_bar, pvd_parity, ctl)) {
      ptx::tmem_wait_st();  // no tensor-memory store of this warp left in flight
      return false;
    }
    ptx::tc_fence_after();
    const uint64_t al2 = ptx::f2(alpha, alpha);
#pragma unroll
    for (int c0 = 0; c0 < D / 2; c0 += 32) {  // this half's D/2 columns of O
      uint32_t o[32];
      ptx::tmem_ld_x32(tO + c0, o);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float a, b;
        ptx::f2_split(
            ptx::f2_mul(ptx::f2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), al2), a, b);
        o[i] = __float_as_uint(a);
        o[i + 1] = __float_as_uint(b);
      }
      ptx::tmem_st_x32(tO + c0, o);
    }
  }
  ptx::tmem_wait_st();
  return true;
}

// What the softmax warps need of unit k, published by the epilogue warps one
// unit ahead (they decode every unit anyway), so that the softmax warps spend
// nothing on decoding between units.  Followed in the slot by int lo[128],
// hi[128]: the visible keys (inclusive, within the sequence) of each row of
// this CTA's tile (row_keys), for units with n > 0.
struct UnitDesc {
  int valid;       // 0: the walk has ended (no unit k)
  int n;           // K/V steps of the pair
  int j0;          // first K/V tile
  int q0;          // first query row of this CTA's tile (may be < 0)
  int Lq;          // query rows of the sequence
  int pad;
  long long lse0;  // LSE index of row 0 of the sequence and head (row q adds q)
};
static_assert(sizeof(UnitDesc) == 32, "descriptor header");

// Epilogue warp of lane quarter `quarter`: writes its 32 rows of descriptor k
// (and, for quarter 0, the header), then arrives on DR + k % 2.
template <int D>
__device__ __forceinline__ void publish_desc(const FwdParams& p, uint32_t rank, uint8_t* base,
                                             uint32_t bars, int k, bool valid, const Unit& w,
                                             int n, int quarter, int lane) {
  using L = Layout<D>;
  uint8_t* const slot = base + L::kDescOff + (k & 1) * L::kDescBytes;
  int* const lo = reinterpret_cast<int*>(slot + sizeof(UnitDesc));
  const int row = quarter * 32 + lane;
  const int q0 = valid ? q0_of(w, static_cast<int>(rank)) : 0;
  if (valid && n > 0) {
    int key_lo, key_hi;
    row_keys(p, w, q0 + row, key_lo, key_hi);
    lo[row] = key_lo;
    lo[128 + row] = key_hi;
  }
  if (quarter == 0 && lane == 0) {
    UnitDesc d;
    d.valid = valid ? 1 : 0;
    d.n = valid ? n : 0;
    d.j0 = valid ? w.j0 : 0;
    d.q0 = q0;
    d.Lq = valid ? w.Lq : 0;
    d.pad = 0;
    d.lse0 = !valid ? 0
             : p.varlen ? static_cast<long long>(w.h) * p.Sq + w.q_start
                        : (static_cast<long long>(w.b) * p.H + w.h) * p.Sq;
    *reinterpret_cast<UnitDesc*>(slot) = d;
  }
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(bars + 8u * (L::DR + (k & 1)));
}

// After a wait of a softmax warp gave up: the warp's remaining arrivals at its
// named barrier -- `pending` of the current unit, then n + 1 for every unit
// from k_first on with n > 0 steps (one per step and the closing exchange of
// the row sums).  The two warps of a row walk the same units and steps (the
// units of the descriptors, which come from the same decode), so the partner
// warp, which may have passed the same wait, never stays at that barrier.
static __device__ __noinline__ void finish_row_barriers(const FwdParams& p, int k_first,
                                                        int pending, uint32_t xbar) {
  for (int i = 0; i < pending; ++i) ptx::named_bar_sync(xbar, 64);
  Cursor cur;
  init_cursor<kUR>(p, cur, false);
  Unit w;
  int n = 0;
  for (int k = 0; decode_pair(p, k, cur, w, n, false); ++k)
    for (int i = 0; k >= k_first && n > 0 && i <= n; ++i) ptx::named_bar_sync(xbar, 64);
}

template <int D, bool BF16>
__device__ void softmax_role(const FwdParams& p, uint32_t rank, uint32_t tmem, uint32_t bars,
                             uint8_t* base, const Ctl& ctl) {
  using L = Layout<D>;
  const int warp = threadIdx.x >> 5;  // 0..7
  const int lane = threadIdx.x & 31;
  const int quarter = warp & 3;       // TMEM lane quarter (= SM sub-partition)
  const int half = warp >> 2;         // S columns [64 half, +64), O columns [D/2 half, +D/2)
  const int row = quarter * 32 + lane;
  const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tO = tmem + lane_bits + L::kColO + half * (D / 2);
  const uint32_t bar_p_lead = ptx::mapa(bars + 8 * L::PF, 0);  // + 8 * (G % 3)
  const uint32_t bar_lr = bars + 8 * L::LR, bar_lf = bars + 8 * L::LF;
  const uint32_t xbar = 1 + quarter;  // named barrier of the two warps of these rows
  float* const xmax = reinterpret_cast<float*>(base + L::kXMaxOff);  // [parity][half][row]
  float* const xsum = reinterpret_cast<float*>(base + L::kXSumOff);  // [half][row][2]
  float* const inv_l_slot = reinterpret_cast<float*>(base + L::kInvLOff);
  uint32_t lr_cnt = 0, g_base = 0;

  for (int k = 0;; ++k) {
    if (!wait_bar_warp(bars + 8u * (L::DR + (k & 1)), (static_cast<uint32_t>(k) >> 1) & 1u,
                       ctl)) {
      finish_row_barriers(p, k, 0, xbar);
      return;
    }
    const uint8_t* const slot = base + L::kDescOff + (k & 1) * L::kDescBytes;
    const UnitDesc d = *reinterpret_cast<const UnitDesc*>(slot);
    if (!d.valid) break;
    const int n = d.n;
    const int qrow = d.q0 + row;
    const bool row_ok = qrow >= 0 && qrow < d.Lq;
    const long long lidx = d.lse0 + qrow;
    RowState rs{-INFINITY, 0.0f, 0.0f};
    if (n > 0) {
      // visible keys of this row, shifted to this half's columns
      const int* const keys = reinterpret_cast<const int*>(slot + sizeof(UnitDesc));
      const int key_lo = keys[row] - 64 * half;
      const int key_hi = keys[128 + row] - 64 * half;
      for (int j = 0, kb = d.j0 * kBN; j < n; ++j, kb += kBN) {
        const uint32_t G = g_base + j;
        const uint32_t b = G % kNBuf;
        if (!wait_bar_warp(bars + 8 * (L::SF + b), (G / kNBuf) & 1u, ctl)) {
          finish_row_barriers(p, k + 1, n - j + 1, xbar);
          return;
        }
        ptx::tc_fence_after();
        const int lo = key_lo - kb;
        const int limit = min(63, key_hi - kb);
        // O += P(G-1) V(G-1) may still be running: a rescale of O waits for it.
        const uint32_t gp = G - 1;
        float* const xm = xmax + (G & 1u) * 256;
        const uint32_t tSb = tmem + lane_bits + L::kColS + b * 128;
        if (!softmax_half_step<D, BF16>(tSb + 64 * half, tSb + 32 * half, tO, lo, limit, p.scale_log2,
                                     p.scale_pos != 0, j == 0, rs, xm + half * 128 + row,
                                     xm + (1 - half) * 128 + row, xbar,
                                     bars + 8 * (L::PVD + gp % kNBuf), (gp / kNBuf) & 1u, ctl)) {
          finish_row_barriers(p, k + 1, n - j, xbar);
          return;
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster_relaxed(bar_p_lead + 8u * b);
      }
      g_base += n;
      // both halves' sums are relative to the same running max: add them
      xsum[(half * 128 + row) * 2 + 0] = rs.l_p;
      xsum[(half * 128 + row) * 2 + 1] = rs.l_x;
      ptx::named_bar_sync(xbar, 64);
      rs.l_p += xsum[((1 - half) * 128 + row) * 2 + 0];
      rs.l_x += xsum[((1 - half) * 128 + row) * 2 + 1];
    }
    // Hand 1 / l to the epilogue warps once they have read the last one.  Every
    // unit does this, even one without steps: the epilogue waits for it before
    // writing the unit's rows, which keeps it at most one descriptor ahead.
    if (half == 0) {
      if (lr_cnt > 0 && !wait_bar_warp(bar_lf, (lr_cnt - 1) & 1u, ctl)) {
        finish_row_barriers(p, k + 1, 0, xbar);
        return;
      }
      inv_l_slot[row] = rs.l_p > 0.0f ? 1.0f / rs.l_p : 0.0f;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_lr);
      ++lr_cnt;
    }
    // rows without any visible key (n = 0) get LSE = -inf; their O = 0 is
    // written by the epilogue warps.  Both halves hold the same sums and max
    // after the exchange; half 1 writes the LSE while half 0 hands over 1 / l.
    if (row_ok && half == 1) {
      p.lse[lidx] = rs.l_x > 0.0f ? (rs.m + ptx::lg2(rs.l_x)) * 0.69314718055994531f : -INFINITY;
    }
  }
}

// Epilogue warps (one per TMEM lane quarter, thread = query row): per unit,
// publish the descriptor of the next unit for the softmax warps, wait for
// 1 / l and for the unit's last O += P V, read O (all D columns) out of
// tensor memory, release it to the next unit's products, then scale, round
// and store the row.  The softmax warps meanwhile start the next unit.
template <int D, bool BF16>
__device__ void epilogue_role(const FwdParams& p, uint32_t rank, uint32_t tmem, uint32_t bars,
                              uint8_t* base, const Ctl& ctl) {
  using L = Layout<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // TMEM lane quarter this warp may access
  const int row = quarter * 32 + lane;
  const uint32_t tO = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + L::kColO;
  const uint32_t bar_lr = bars + 8 * L::LR, bar_lf = bars + 8 * L::LF, bar_of = bars + 8 * L::OF;
  const uint32_t bar_free_lead = ptx::mapa(bars + 8 * L::OFREE, 0);
  const float* const inv_l_slot = reinterpret_cast<const float*>(base + L::kInvLOff);
  uint16_t* const O = static_cast<uint16_t*>(p.o);
  // rows are D * 2 bytes apart: 32-byte stores whenever O itself is 32-byte aligned
  const bool o32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
  uint32_t lr_cnt = 0, of_cnt = 0;

  Cursor cur;
  init_cursor<kUR>(p, cur, false);
  Unit w_next;
  int n_next = 0;
  bool more = decode_pair(p, 0, cur, w_next, n_next, false);
  publish_desc<D>(p, rank, base, bars, 0, more, w_next, n_next, quarter, lane);
  for (int k = 0; more; ++k) {
    const Unit w = w_next;
    const int n = n_next;
    more = decode_pair(p, k + 1, cur, w_next, n_next, false);
    publish_desc<D>(p, rank, base, bars, k + 1, more, w_next, n_next, quarter, lane);
    const int qrow = q0_of(w, static_cast<int>(rank)) + row;
    const bool row_ok = qrow >= 0 && qrow < w.Lq;
    const long long orow = (static_cast<long long>(w.q_start) + qrow) * p.H + w.h;
    if (!wait_bar_warp(bar_lr, lr_cnt & 1u, ctl)) return;
    ++lr_cnt;
    const float inv_l = inv_l_slot[row];
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar_lf);
    if (n == 0) {  // no visible key: O = 0
      if (row_ok) {
        uint4* const dst = reinterpret_cast<uint4*>(O + orow * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    if (!wait_bar_warp(bar_of, of_cnt & 1u, ctl)) return;
    ++of_cnt;
    ptx::tc_fence_after();
    uint4* const dst = reinterpret_cast<uint4*>(O + (row_ok ? orow : 0) * D);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 64) {
      uint32_t o[64];
      ptx::tmem_ld_x64(tO + c0, o);
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        pk[i] = ptx::pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l,
                                 __uint_as_float(o[2 * i + 1]) * inv_l);
      if (row_ok) {
        if (o32) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            ptx::st_global_v8(dst + c0 / 8 + 2 * i, pk[8 * i], pk[8 * i + 1], pk[8 * i + 2],
                              pk[8 * i + 3], pk[8 * i + 4], pk[8 * i + 5], pk[8 * i + 6],
                              pk[8 * i + 7]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[c0 / 8 + i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
    }
    // every load of O has completed (tcgen05.ld waits): the next unit may overwrite it
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster_relaxed(bar_free_lead);
  }
}

// -------------------------------------------------------------------- MMA
// S thread: lane 0 of warp kPMma of the even CTA.
template <int D, bool BF16>
__device__ void s_loop(const FwdParams& p, uint32_t smem, uint32_t tmem, uint32_t bars,
                       const Ctl& ctl) {
  using L = Layout<D>;
  constexpr int NS = L::kStages;
  constexpr uint32_t kIdS = ptx::idesc_f16_f32acc(BF16, 2 * kBM, kBN, false);
  constexpr uint16_t kBoth = 3;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t g_base = 0, q_it = 0;
  const uint64_t dq = ptx::desc_sw128(smem + L::kQOff, 16, 1024);
  const uint64_t dk0 = ptx::desc_sw128(smem + L::kKOff, 16, 1024);
  Cursor cur;
  init_cursor<kUR>(p, cur, false);
  Unit w;
  int n = 0;
  for (int k = 0; decode_pair(p, k, cur, w, n, false); ++k) {
    if (n == 0) continue;
    if (!wait_bar(bar(L::QF), q_it & 1u, ctl)) return;
    ptx::tc_fence_after();
    for (int j = 0; j < n; ++j) {
      const uint32_t G = g_base + j;
      if (G >= kNBuf) {  // buffer G % 3 holds P(G-3) until O += P(G-3) V(G-3) is done
        const uint32_t gp = G - kNBuf;
        if (!wait_bar(bar(L::PVD + gp % kNBuf), (gp / kNBuf) & 1u, ctl)) return;
      }
      const uint32_t st = G % NS;
      if (!wait_bar(bar(L::KF + st), (G / NS) & 1u, ctl)) return;
      ptx::tc_fence_after();
      const uint64_t dk = dk0 + ((st * L::kKHalf) >> 4);
      const uint32_t tS = tmem + L::kColS + (G % kNBuf) * 128;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t qoff = ((ks >> 2) * L::kBlk + (ks & 3) * 32) >> 4;
        const uint32_t koff = ((ks >> 2) * L::kKBlk + (ks & 3) * 32) >> 4;
        ptx::mma_ss_pair(tS, dq + qoff, dk + koff, kIdS, ks > 0 ? 1u : 0u);
      }
      ptx::mma_commit_pair(bar(L::SF + G % kNBuf), kBoth);
      ptx::mma_commit_pair(bar(L::KE + st), kBoth);
      if (j == n - 1) ptx::mma_commit_pair(bar(L::QE), kBoth);  // Q no longer read
    }
    g_base += n;
    ++q_it;
  }
}

// PV thread: lane 0 of warp kPPv of the even CTA.
template <int D, bool BF16>
__device__ void pv_loop(const FwdParams& p, uint32_t smem, uint32_t tmem, uint32_t bars,
                        const Ctl& ctl) {
  using L = Layout<D>;
  constexpr int NS = L::kStages;
  constexpr uint32_t kIdPV = ptx::idesc_f16_f32acc(BF16, 2 * kBM, D, true);
  constexpr uint16_t kBoth = 3;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t g_base = 0;
  // V half, MN-major (D/2 dims contiguous per key): one 128-byte swizzle atom
  // column (D = 128) or one 64-byte one (D = 64); the next 8 keys follow at
  // 8 rows x D bytes
  const uint64_t dv0 = D == 128 ? ptx::desc_sw128(smem + L::kVOff, L::kBlk, 1024)
                                : ptx::desc_sw64(smem + L::kVOff, L::kBlk, 512);
  const uint32_t tO = tmem + L::kColO;
  uint32_t u_cnt = 0;  // units with steps so far
  Cursor cur;
  init_cursor<kUR>(p, cur, false);
  Unit w;
  int n = 0;
  for (int k = 0; decode_pair(p, k, cur, w, n, false); ++k) {
    if (n == 0) continue;
    for (int j = 0; j < n; ++j) {
      const uint32_t G = g_base + j;
      // O += P(G) V(G): P(G) in buffer G % 3 of both CTAs
      if (!wait_bar_cluster(bar(L::PF + G % kNBuf), (G / kNBuf) & 1u, ctl)) return;
      // the unit's first product overwrites O: the previous unit's O must have been read
      if (j == 0 && u_cnt > 0 &&
          !wait_bar_cluster(bar(L::OFREE), (u_cnt - 1) & 1u, ctl))
        return;
      const uint32_t st = G % NS;
      if (!wait_bar(bar(L::VF + st), (G / NS) & 1u, ctl)) return;
      ptx::tc_fence_after();
      const uint64_t dv = dv0 + ((st * L::kVHalf) >> 4);
      const uint32_t tP = tmem + L::kColS + (G % kNBuf) * 128;
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks)  // 16 keys = 2 atoms of 8 key rows x D bytes
        ptx::mma_ts_pair(tO, tP + ks * 8, dv + ((ks * 16 * D) >> 4), kIdPV,
                         (j > 0 || ks > 0) ? 1u : 0u);
      ptx::mma_commit_pair(bar(L::VE + st), kBoth);
      ptx::mma_commit_pair(bar(L::PVD + G % kNBuf), kBoth);
      if (j == n - 1) ptx::mma_commit_pair(bar(L::OF), kBoth);
    }
    g_base += n;
    ++u_cnt;
  }
}

// Each MMA thread makes sure its own tcgen05 operations retired before TMEM is
// freed, also when its loop was abandoned.
template <int D>
__device__ __forceinline__ void mma_drain(uint32_t bars, const Ctl& ctl) {
  const uint32_t done = bars + 8u * Layout<D>::DONE;
  ptx::mma_commit_pair(done, 1);
  wait_bar(done, 0, ctl, false);
}

// ------------------------------------------------------------------- load
template <int NS>
struct PairLoadLog {
  FillLog<1> q;
  FillLog<NS> k, v;
};

// Runs on lane 0 of the load warp of both CTAs; each loads its own Q tile and
// its half of every K/V tile, counting the bytes on the even CTA's barriers
// (the even CTA arms each phase for both halves).  Every issued fill is
// recorded in `f`.
template <int D>
static __device__ void load_loop(const FwdParams& p, uint32_t smem, uint32_t bars, uint32_t rank,
                                 const Ctl& ctl, PairLoadLog<Layout<D>::kStages>& f) {
  using L = Layout<D>;
  constexpr int NS = L::kStages;
  const bool lead = rank == 0;
  auto bar = [&](int i) { return bars + 8u * i; };
  auto lbar = [&](int i) { return ptx::mapa(bars + 8u * i, 0); };
  uint32_t kv_it = 0, q_it = 0;
  Cursor cur;
  init_cursor<kUR>(p, cur, true);
  Unit w;
  int n = 0;
  for (int k = 0; decode_pair(p, k, cur, w, n, lead); ++k) {
    if (n == 0) continue;
    if (q_it > 0 && !wait_bar(bar(L::QE), (q_it - 1) & 1u, ctl)) return;
    if (lead) ptx::mbar_arrive_expect_tx(bar(L::QF), 2 * L::kQTile);
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk)
      ptx::tma_load_3d_pair(smem + L::kQOff + blk * L::kBlk, &p.tm_q, lbar(L::QF), blk * 64, w.h,
                            w.q_start + q0_of(w, static_cast<int>(rank)));
    f.q.last[0] = static_cast<int>(q_it);
    ++q_it;
    for (int j = 0; j < n; ++j) {
      const uint32_t it = kv_it + j;
      const uint32_t st = it % NS;
      const int krow = w.k_start + (w.j0 + j) * kBN;
      if (it >= NS && !wait_bar(bar(L::KE + st), (it / NS - 1) & 1u, ctl)) return;
      // injected fault (tests only): the even CTA of pair 0 neither arms nor
      // loads its first K half, so the S thread's bounded wait runs out
      if (!(p.inject == 1 && lead && blockIdx.x == 0 && it == 0)) {
        if (lead) ptx::mbar_arrive_expect_tx(bar(L::KF + st), 2 * L::kKHalf);
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk)
          ptx::tma_load_3d_pair(smem + L::kKOff + st * L::kKHalf + blk * L::kKBlk, &p.tm_kh,
                                lbar(L::KF + st), blk * 64, w.h,
                                krow + 64 * static_cast<int>(rank));
        f.k.last[st] = static_cast<int>(it);
      }
      if (it >= NS && !wait_bar(bar(L::VE + st), (it / NS - 1) & 1u, ctl)) return;
      if (lead) ptx::mbar_arrive_expect_tx(bar(L::VF + st), 2 * L::kVHalf);
      ptx::tma_load_3d_pair(smem + L::kVOff + st * L::kVHalf, &p.tm_vh, lbar(L::VF + st),
                            (D / 2) * static_cast<int>(rank), w.h, krow);
      f.v.last[st] = static_cast<int>(it);
    }
    kv_it += n;
  }
}

// Settles the open phase of one "full" barrier of the even CTA after both
// loaders have stopped and waits (bounded) for it.  `mine` / `peer` are the
// last fills the even / odd CTA issued into this buffer: only the later one
// can still be open (a buffer is refilled only after its previous fill
// completed).  A fill the even CTA issued was armed for both halves; if the
// odd CTA never sent its half, those bytes are counted here.  A fill only the
// odd CTA issued was never armed; it is armed here for the odd half alone.
// Such a repaired phase must not release a consumer: the caller repairs only
// after the MMA threads have finished.
__device__ __forceinline__ void settle_fill(uint32_t bar, int mine, int peer, int ring,
                                            uint32_t half_bytes, const Ctl& ctl) {
  const int last = max(mine, peer);
  if (last < 0) return;
  if (mine < last)
    ptx::mbar_arrive_expect_tx(bar, half_bytes);
  else if (peer < last)
    ptx::mbar_complete_tx(bar, half_bytes);
  wait_bar(bar, (static_cast<uint32_t>(last) / ring) & 1u, ctl, false);
}

template <int D>
static __device__ void load_role(const FwdParams& p, uint32_t smem, uint8_t* base, uint32_t bars,
                                 uint32_t rank, const Ctl& ctl) {
  using L = Layout<D>;
  constexpr int kStages = L::kStages;
  PairLoadLog<kStages> f;
  f.q.clear();
  f.k.clear();
  f.v.clear();
  load_loop<D>(p, smem, bars, rank, ctl, f);
  const uint32_t rec = smem + L::kFillOff;
  if (rank != 0) {
    // hand this CTA's record to the even CTA, whose barriers count our copies
    const uint32_t dst = ptx::mapa(rec, 0);
    ptx::st_shared_cluster(dst, static_cast<uint32_t>(f.q.last[0]));
#pragma unroll
    for (int st = 0; st < kStages; ++st) {
      ptx::st_shared_cluster(dst + 4u * (1 + st), static_cast<uint32_t>(f.k.last[st]));
      ptx::st_shared_cluster(dst + 4u * (1 + kStages + st), static_cast<uint32_t>(f.v.last[st]));
    }
    ptx::mbar_arrive_cluster(ptx::mapa(bars + 8u * L::LDONE, 0));  // release: stores first
    return;
  }
  // Even CTA: no copy of the pair may land after either CTA exits (the odd one
  // leaves only after the closing cluster barrier, which this thread reaches
  // after the waits below).
  PairLoadLog<kStages> o = f;
  if (wait_bar_cluster(bars + 8u * L::LDONE, 0, Ctl{ctl.abort_flag, ctl.err, ctl.timeout_ns},
                       false)) {
    const int* r = reinterpret_cast<const int*>(base + L::kFillOff);
    o.q.last[0] = r[0];
#pragma unroll
    for (int st = 0; st < kStages; ++st) {
      o.k.last[st] = r[1 + st];
      o.v.last[st] = r[1 + kStages + st];
    }
  }
  // The records differ only if a loader stopped early or a fill was skipped:
  // then the MMA threads may still be waiting for the phases about to be
  // repaired, so wait (bounded) until both have finished (they always do,
  // every one of their waits being bounded) before repairing any.
  bool differ = f.q.last[0] != o.q.last[0];
  for (int st = 0; st < kStages; ++st)
    differ = differ || f.k.last[st] != o.k.last[st] || f.v.last[st] != o.v.last[st];
  if (differ) wait_bar(bars + 8u * L::DONE, 0, ctl, false);
  settle_fill(bars + 8u * L::QF, f.q.last[0], o.q.last[0], 1, L::kQTile, ctl);
#pragma unroll 1
  for (int st = 0; st < kStages; ++st) {
    settle_fill(bars + 8u * (L::KF + st), f.k.last[st], o.k.last[st], kStages, L::kKHalf, ctl);
    settle_fill(bars + 8u * (L::VF + st), f.v.last[st], o.v.last[st], kStages, L::kVHalf, ctl);
  }
}

// ------------------------------------------------------------------ kernel
template <int D, bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    attn_fwd_kernel_2sm(const __grid_constant__ FwdParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t smem = (raw + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (smem - raw);
  const uint32_t bars = smem + L::kBarOff;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(base + L::kMiscOff);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(base + L::kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_rank();

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i)
      ptx::mbar_init(bars + 8u * i, (i >= L::PF && i < L::PF + kNBuf) ? L::kPArrivals
                                    : i == L::DONE                  ? L::kDoneArrivals
                                    : i == L::LR                    ? L::kLrArrivals
                                    : i == L::LF                    ? L::kLfArrivals
                                    : i == L::OFREE                 ? L::kOFreeArrivals
                                    : i >= L::DR                    ? L::kDrArrivals
                                                                    : 1u);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA use
  build_seq_order(p);
  if (warp == kPMma) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  if (warp == kPLoad && lane == 0) {
    ptx::tma_prefetch_desc(&p.tm_q);
    ptx::tma_prefetch_desc(&p.tm_kh);
    ptx::tma_prefetch_desc(&p.tm_vh);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};

  if (warp < kSoftmaxWarps) {
    softmax_role<D, BF16>(p, rank, tmem, bars, base, ctl);
  } else if (warp == kPMma) {
    if (lane == 0 && rank == 0) {
      s_loop<D, BF16>(p, smem, tmem, bars, ctl);
      mma_drain<D>(bars, ctl);
    }
  } else if (warp == kPPv) {
    if (lane == 0 && rank == 0) {
      pv_loop<D, BF16>(p, smem, tmem, bars, ctl);
      mma_drain<D>(bars, ctl);
    }
  } else if (warp == kPLoad) {
    if (lane == 0) load_role<D>(p, smem, base, bars, rank, ctl);
  } else {
    epilogue_role<D, BF16>(p, rank, tmem, bars, base, ctl);
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the even CTA's MMAs (reading both CTAs) are all retired
  ptx::tc_fence_after();
  if (warp == kPMma) ptx::tmem_dealloc_pair(tmem, kTmemCols);
}

template <int D>
inline int fwd_2sm_smem_bytes(const FwdParams& p) {
  return Layout<D>::kAlloc + (seq_ordered(p) ? kOrderBytes : 0);
}

template <int D, bool BF16>
cudaError_t launch_fwd_2sm(const FwdParams& params, int grid, cudaStream_t stream) {
  FwdParams p = params;
  p.order_off = Layout<D>::kBytes;  // the packed-sequence order follows the layout
  const void* fn = reinterpret_cast<const void*>(&attn_fwd_kernel_2sm<D, BF16>);
  static std::atomic<unsigned long long> opted{0};
  const cudaError_t e = smem_opt_in(fn, Layout<D>::kAlloc + kOrderBytes, opted);
  if (e != cudaSuccess) return e;
  void* args[] = {&p};
  return cudaLaunchKernel(fn, dim3(grid), dim3(kPairThreads), args, fwd_2sm_smem_bytes<D>(p),
                          stream);
}

}  // namespace pair
}  // namespace attn
