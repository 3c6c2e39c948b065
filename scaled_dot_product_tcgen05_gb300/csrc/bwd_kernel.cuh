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
// Sequences are either dense (B of Sq queries and Sk keys) or packed
// (cu_seqlens, as the forward); every index below is within the sequence.
//
// GB300 mapping: a persistent kernel, one CTA per SM, work unit = (sequence,
// head, 128-key tile).  Keys are the M dimension of every product the unit
// accumulates, so dK and dV stay in tensor memory for the whole unit:
//   TMEM columns: S^T | dP^T | dV | dK (128, 128, D, D); dQ of a step is
//   written over dP^T once dS^T has been consumed, so S^T of the next query
//   tile can be computed while this step's dS is still being formed.
//   * warp 13 (one lane): TMA for the unit's K and V tiles and, per step
//     (128 queries), Q and dO tiles into a 2-stage ring;
//   * warp 12 (one lane): tcgen05.mma
//       S^T  = K Q^T      (SS, K-major / K-major)
//       dP^T = V dO^T     (SS)
//       dV  += P^T dO     (TS: P^T from TMEM, dO MN-major)
//       dK  += dS^T Q     (TS: dS^T from TMEM, Q MN-major)
//       dQ   = dS K       (SS: dS MN-major from shared memory, K MN-major)
//   * the per-query terms -LSE/scale and -D enter the products themselves: one
//     extra K = 16 step multiplies a ones column (in shared memory) by a
//     three-part bf16 split of each term (16 bytes per query row, written by
//     the pre-pass), so S^T arrives as S^T - LSE/scale and dP^T as dP^T - D
//     and the per-element loops below need no per-column loads;
//   * warps 0-7: two threads per key (TMEM lane; warps w and w + 4 share lane
//     quarter w), each for 64 of the step's 128 queries: P^T = 2^(scale log2e
//     S'^T) written back as 16-bit into its own half's columns of S^T, then
//     dS^T = P^T dP'^T into its half's columns of dP^T and into the dO stage
//     (whose dO the dV and dP^T products have finished reading), as the A
//     operand of dQ.  Half h writes only columns 64h .. 64h + 31, which it has
//     already read, so the halves never wait for each other;
//   * warps 8-11: one thread per query row: dQ of each step is staged in the
//     step's dO ring stage (free once dQ is computed; 128-byte swizzled, so
//     the row-per-thread writes hit distinct banks; 64 columns at a time) and
//     added to an fp32 [H, rows, D] accumulator by TMA tensor reduce-adds,
//     after which the dO stage goes back to the loader.  The Q stage has its
//     own barriers and returns to the loader as soon as dQ is computed, so the
//     next Q tile is not held up by the reduce-adds.  At the end of the unit
//     these warps write dK (times scale) and dV.
// Every wait is bounded (same error word and abort flag as the forward).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fwd_kernel.cuh"

namespace attn {
namespace bwd {

constexpr int kBM = 128;  // keys per unit
constexpr int kBN = 128;  // queries per step
constexpr int kThreads = 448;  // 14 warps: at most 4 per SM sub-partition, so <= 128 registers
constexpr int kDsWarps = 8;
constexpr int kDqWarp0 = 8;
constexpr int kMmaWarp = 12;
constexpr int kLoadWarp = 13;
constexpr int kTmemCols = 512;
// A 128 x 16 16-bit operand without swizzle: 8 x 8 core matrices of 8 rows x
// 16 B; row r, element k at (r / 8) * 256 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2.
constexpr int kBiasBytes = 4096;
constexpr int kBiasParts = 3;  // a term is the sum of three bf16 values

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // [rows, H, D] 16-bit, box 64 x 1 x 128, 128-B swizzle
  // dq_acc, fp32, box 32 x 128 x 1, 128-B swizzle: dense [B*H, Sq, D], packed [H, Tq, D]
  CUtensorMap tm_dq;
  // per 128-query tile t of (sequence b, head h): [2][kBiasBytes] (-LSE/scale,
  // -D), t = tile0(b) * H + h * nq(b) + i, tile0(b) = the tiles of sequences
  // before b (dense: b * nq)
  const uint8_t* bias;
  const int32_t* tiles;                  // packed: tile0(0..B) and a valid-bounds flag
  float* dq_acc;                         // zero on entry
  void* dk;                              // [key rows, H, D]
  void* dv;
  const int32_t* cu_q;                   // packed sequences only
  const int32_t* cu_k;
  int* err;
  int B, H, Sq, Sk;  // dense: per-sequence lengths; packed: total rows
  int Tq;            // query rows in all: B * Sq dense, Sq packed
  int varlen, causal;
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
  static constexpr int kOnesOff = kDoOff + 2 * kDoStage;  // 128 x 16 ones column (bf16)
  static constexpr int kBiasOff = kOnesOff + kBiasBytes;   // 2 stages x (S bias, D bias)
  static constexpr int kBarOff = kBiasOff + 2 * 2 * kBiasBytes;
  // QF/QE: Q tile + S bias of a ring stage; DOF/DOE: dO tile + D bias (and
  // later dS, then the dQ staging) of a ring stage.
  enum : int {
    KVF = 0, KVE, QF0, QF1, QE0, QE1, DOF0, DOF1, DOE0, DOE1, SF, DPF, PR, DVD, DSR, DQF, DQE,
    OF, AE, STG, STF, DONE, kNumBars
  };
  // dQ staging: fp32, 128 rows x 32 columns = one 16 KiB swizzled box; two
  // boxes (64 columns) at a time in the step's dO stage.
  static constexpr int kDqBox = 16384;
  __host__ __device__ static constexpr int dq_box_off(int st, int pos) {
    return kDoOff + st * kDoStage + pos * kDqBox;
  }
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;  // tmem base, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
};

// ---------------------------------------------------------------- helpers
__host__ __device__ constexpr uint32_t idesc_ab(bool bf16, int M, int N, bool a_mn, bool b_mn) {
  return ptx::idesc_f16_f32acc(bf16, M, N, b_mn) | ((a_mn ? 1u : 0u) << 15);
}

// Descriptor of a K-major operand without swizzle (layout above): leading
// byte offset 128 (next core matrix along K), stride byte offset 256 (next 8
// rows), version bit 46, swizzle mode 0.
__device__ __forceinline__ uint64_t desc_noswz(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 16;
  d |= static_cast<uint64_t>(256 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar) : "memory");
}

// TMA tensor reduce-add of one box from shared memory into global fp32.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int c0,
                                                  int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%1, %2, %3}], [%4];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {  // sources of all committed groups read
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {   // all committed groups complete
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__host__ __device__ constexpr int bias_offset(int r, int k) {
  return (r / 8) * 256 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2;
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
// query tiles).  Steps: query tiles i0 .. nq-1 of the sequence.
struct BUnit {
  int b, h, kt, i0, n;
  int q_start, Lq, k_start, Lk;  // the sequence's first rows and lengths
  int tile0;                     // bias tiles of the sequences before b, per head
  int base, units;               // packed: first unit of sequence b and its unit count
};

// Packed sequences: sequence w.b's rows, lengths and unit count into w.
__device__ __forceinline__ void bwd_load_seq(const BwdParams& p, BUnit& w, bool report) {
  w.units = 0;
  w.q_start = w.Lq = w.k_start = w.Lk = 0;
  if (w.b >= p.B) return;
  const int q0 = __ldg(p.cu_q + w.b), q1 = __ldg(p.cu_q + w.b + 1);
  const int k0 = __ldg(p.cu_k + w.b), k1 = __ldg(p.cu_k + w.b + 1);
  const bool ok = 0 <= q0 && q0 <= q1 && q1 <= p.Sq && 0 <= k0 && k0 <= k1 && k1 <= p.Sk;
  if (!ok) {  // the sequence is skipped and the call reports ATTN_ERR_BAD_SEQLENS
    if (report) atomicOr(p.err, kErrBadSeqlens);
    return;
  }
  w.q_start = q0;
  w.Lq = q1 - q0;
  w.k_start = k0;
  w.Lk = k1 - k0;
  w.tile0 = __ldg(p.tiles + w.b);
  w.units = p.H * ((w.Lk + kBM - 1) / kBM);
}

// Before the first bwd_unit call of a role.
template <bool VARLEN>
__device__ __forceinline__ void bwd_walk(const BwdParams& p, BUnit& w, bool report) {
  w.b = 0;
  w.base = 0;
  if constexpr (VARLEN) {
    if (__ldg(p.tiles + p.B + 1) == 0) {  // malformed bounds somewhere: no work at all
      w.b = p.B;
      w.units = 0;
      return;
    }
    bwd_load_seq(p, w, report);
  }
}

// The k-th unit of this CTA (dealt as the forward deals its units); packed
// sequences are walked forward, so k must increase from call to call.
template <bool VARLEN>
__device__ __forceinline__ bool bwd_unit(const BwdParams& p, int k, BUnit& w,
                                         bool report = false) {
  const int u = unit_of(k);
  if constexpr (!VARLEN) {
    const int nk = (p.Sk + kBM - 1) / kBM;
    if (u >= p.B * p.H * nk) return false;
    const int bh = u / nk;
    w.kt = u - bh * nk;
    w.b = bh / p.H;
    w.h = bh - w.b * p.H;
    w.q_start = w.b * p.Sq;
    w.Lq = p.Sq;
    w.k_start = w.b * p.Sk;
    w.Lk = p.Sk;
    w.tile0 = w.b * ((p.Sq + kBN - 1) / kBN);
  } else {
    while (true) {
      if (w.b >= p.B) return false;
      if (u < w.base + w.units) break;
      w.base += w.units;
      w.b += 1;
      bwd_load_seq(p, w, report);
    }
    const int rem = u - w.base;
    const int nk = w.units / p.H;
    w.h = rem / nk;
    w.kt = rem - w.h * nk;
  }
  const int nq = (w.Lq + kBN - 1) / kBN;
  // causal (top-left): query tile i has a row >= every key of tile kt from i = kt on
  w.i0 = p.causal ? w.kt : 0;
  w.n = max(0, nq - w.i0);
  return true;
}

// Steps of this CTA in order, across its units (units without steps skipped).
template <bool VARLEN>
struct StepIter {
  int k;     // unit counter of this CTA
  BUnit w;
  int j;     // step within the unit
  bool ok;
  __device__ __forceinline__ void start(const BwdParams& p) {
    k = 0;
    j = 0;
    bwd_walk<VARLEN>(p, w, false);
    ok = bwd_unit<VARLEN>(p, k, w);
    while (ok && w.n == 0) ok = bwd_unit<VARLEN>(p, ++k, w);
  }
  __device__ __forceinline__ void next(const BwdParams& p) {
    if (++j < w.n) return;
    j = 0;
    do ok = bwd_unit<VARLEN>(p, ++k, w);
    while (ok && w.n == 0);
  }
};

// ------------------------------------------------------------- P and dS
template <int D, bool BF16, bool VARLEN>
__device__ void ds_role(const BwdParams& p, uint32_t tmem, uint8_t* base, uint32_t bars,
                        const Ctl& ctl) {
  using L = BLayout<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int half = warp >> 2;           // queries 64 half .. 64 half + 63 of the step
  const int r = quarter * 32 + lane;    // key row of this thread = TMEM lane
  const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + lane_bits + L::kColS + 64 * half;    // S^T, P^T of this half
  const uint32_t tDP = tmem + lane_bits + L::kColDP + 64 * half;  // dP^T, dS^T of this half
  auto bar = [&](int i) { return bars + 8u * i; };
  const uint64_t c2 = ptx::f2(p.scale_log2, p.scale_log2);

  StepIter<VARLEN> cur;
  cur.start(p);
  for (uint32_t g = 0; cur.ok; ++g) {
    const BUnit& w = cur.w;
    const int i = w.i0 + cur.j;
    const int key = w.kt * kBM + r;
    const int qb = i * kBN + 64 * half;
    // columns c (query qb + c) visible to this key: c >= cmin and qb + c < Sq
    const int cmin = p.causal ? key - qb : 0;
    const int cmax = w.Lq - qb - 1;
    const bool row_ok = key < w.Lk;
    const bool full = row_ok && cmin <= 0 && cmax >= 63;

    // ---- P^T = 2^(scale log2e (S^T - LSE / scale)), 16-bit, over S^T
    if (!wait_bar_warp(bar(L::SF), g & 1u, ctl)) return;
    ptx::tc_fence_after();
    uint32_t pk[32];
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t s[32];
      ptx::tmem_ld_x32(tS + c0, s);
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float x0, x1;
        ptx::f2_split(ptx::f2_mul(ptx::f2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), c2),
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
    uint8_t* const ds_tile = base + L::kDoOff + (g & 1u) * L::kDoStage + half * L::kBlk;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t dp[32];
      ptx::tmem_ld_x32(tDP + c0, dp);
      uint32_t dk[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float p0, p1;
        unpack2<BF16>(pk[(c0 + c) / 2], p0, p1);
        float a, b;
        ptx::f2_split(ptx::f2_mul(ptx::f2(p0, p1), ptx::f2(__uint_as_float(dp[c]),
                                                            __uint_as_float(dp[c + 1]))),
                      a, b);
        dk[c / 2] = ptx::pack2<BF16>(a, b);
      }
      tmem_st_x16(tDP + c0 / 2, dk);
      // shared memory: row r (key), queries 64 half + c0 .. +31 = 4 chunks of
      // 16 B in the 128-B swizzled block of this half's 64 queries
      uint8_t* const row = ds_tile + r * 128;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int chunk = (c0 >> 3) + q4;
        *reinterpret_cast<uint4*>(row + ((chunk ^ (r & 7)) << 4)) =
            make_uint4(dk[4 * q4], dk[4 * q4 + 1], dk[4 * q4 + 2], dk[4 * q4 + 3]);
      }
    }
    ptx::tmem_wait_st();
    fence_proxy_async_smem();
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(L::DSR));
    cur.next(p);
  }
}

// -------------------------------------------------- dQ and the dK/dV epilogue
template <int D, bool BF16, bool VARLEN>
__device__ void dq_role(const BwdParams& p, uint32_t tmem, uint32_t smem, uint8_t* base,
                        uint32_t bars, const Ctl& ctl) {
  using L = BLayout<D>;
  const int warp = threadIdx.x >> 5;
  const int quarter = warp & 3;
  const int lane = threadIdx.x & 31;
  const int r = quarter * 32 + lane;  // query row (dQ) / key row (dK, dV) = TMEM lane
  const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint16_t* const DK = static_cast<uint16_t*>(p.dk);
  uint16_t* const DV = static_cast<uint16_t*>(p.dv);
  uint32_t g = 0, u_cnt = 0, stg_n = 0, stf_n = 0;
  BUnit w;
  bwd_walk<VARLEN>(p, w, false);
  for (int k = 0; bwd_unit<VARLEN>(p, k, w); ++k) {
    const int key = w.kt * kBM + r;
    const bool key_ok = key < w.Lk;
    const long long krow = (static_cast<long long>(w.k_start) + key) * p.H + w.h;
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
      const uint32_t st = g & 1u;
      const bool issuer = threadIdx.x == kDqWarp0 * 32;
      // the tile's first query row and the slice: dense [B*H, Sq, D], packed [H, Tq, D]
      const int q0 = (VARLEN ? w.q_start : 0) + (w.i0 + j) * kBN;
      const int slice = VARLEN ? w.h : w.b * p.H + w.h;
      auto stage_box = [&](int pos, const uint32_t (&v)[32]) {  // row r of a box, swizzled
        uint8_t* const row = base + L::dq_box_off(st, pos) + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
              make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      };
      // the issuer waits until all 128 rows are staged, reduces the two boxes
      // of columns x0 .. x0+63, and waits until they have been read
      auto flush = [&](int x0) -> bool {
        fence_proxy_async_smem();
        ptx::mbar_arrive(bar(L::STG));
        if (issuer) {
          if (!wait_bar(bar(L::STG), stg_n & 1u, ctl)) return false;
          tma_reduce_add_3d(&p.tm_dq, smem + L::dq_box_off(st, 0), x0, q0, slice);
          tma_reduce_add_3d(&p.tm_dq, smem + L::dq_box_off(st, 1), x0 + 32, q0, slice);
          bulk_commit();
          bulk_wait_read();
        }
        ++stg_n;
        return true;
      };
      uint32_t v0[32], v1[32];
      ptx::tmem_ld_x32(tmem + lane_bits + L::kColDP, v0);
      ptx::tmem_ld_x32(tmem + lane_bits + L::kColDP + 32, v1);
      if constexpr (D == 64) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::DQE));  // dQ fully read: the dP^T columns are free
        stage_box(0, v0);
        stage_box(1, v1);
        if (!flush(0)) return;
      } else {
        stage_box(0, v0);
        stage_box(1, v1);
        ptx::tmem_ld_x32(tmem + lane_bits + L::kColDP + 64, v0);
        ptx::tmem_ld_x32(tmem + lane_bits + L::kColDP + 96, v1);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::DQE));  // dQ fully read: the dP^T columns are free
        if (!flush(0)) return;
        if (issuer) ptx::mbar_arrive(bar(L::STF));  // the staging boxes may be reused
        if (!wait_bar_warp(bar(L::STF), stf_n & 1u, ctl)) return;
        ++stf_n;
        stage_box(0, v0);
        stage_box(1, v1);
        if (!flush(64)) return;
      }
      if (issuer) ptx::mbar_arrive(bar(L::DOE0 + st));  // the dO stage goes back to the loader
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
template <int D, bool BF16, bool VARLEN>
__device__ void mma_loop(const BwdParams& p, uint32_t smem, uint32_t tmem, uint32_t bars,
                         const Ctl& ctl) {
  using L = BLayout<D>;
  constexpr uint32_t kIdS = idesc_ab(BF16, kBM, kBN, false, false);   // S^T, dP^T
  constexpr uint32_t kIdAcc = idesc_ab(BF16, kBM, D, false, true);    // dV, dK (A from TMEM)
  constexpr uint32_t kIdDq = idesc_ab(BF16, kBN, D, true, true);      // dQ
  constexpr uint32_t kIdBias = idesc_ab(true, kBM, kBN, false, false); // bf16 ones x bias
  const uint64_t dOnes = desc_noswz(smem + L::kOnesOff);
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
    // + ones x (-LSE / scale): S'^T = S^T - LSE / scale per query column
    ptx::mma_ss(tS, dOnes, desc_noswz(smem + L::kBiasOff + st * 2 * kBiasBytes), kIdBias, 1u);
    ptx::mma_commit(bar(L::SF));
    return true;
  };
  // Order per step g (one issuing thread, so tensor memory reuse follows
  // issue order): S^T(g) [issued during step g-1 when in the same unit],
  // dP^T(g) once dQ(g-1) has been read out of the dP^T columns, dV(g) once P(g)
  // is in TMEM, S^T(g+1) (P(g) is consumed by dV(g) before it), then dK(g) and
  // dQ(g) = dS K into the dP^T columns once dS(g) is ready.
  BUnit w;
  bwd_walk<VARLEN>(p, w, false);
  for (int k = 0; bwd_unit<VARLEN>(p, k, w); ++k) {
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
      if (!wait_bar(bar(L::DOF0 + st), (g >> 1) & 1u, ctl)) return;     // dO and D bias here
      ptx::tc_fence_after();
      const uint64_t dDo_kmaj = ptx::desc_sw128(dobase, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {  // dP^T = V dO^T
        const uint32_t off = ((ks >> 2) * L::kBlk + (ks & 3) * 32) >> 4;
        ptx::mma_ss(tDP, dV_kmaj + off, dDo_kmaj + off, kIdS, ks > 0 ? 1u : 0u);
      }
      // + ones x (-D): dP'^T = dP^T - D per query column
      ptx::mma_ss(tDP, dOnes, desc_noswz(smem + L::kBiasOff + (st * 2 + 1) * kBiasBytes),
                  kIdBias, 1u);
      ptx::mma_commit(bar(L::DPF));
      if (!wait_bar(bar(L::PR), g & 1u, ctl)) return;
      if (j == 0 && u_cnt > 0 && !wait_bar(bar(L::AE), (u_cnt - 1) & 1u, ctl)) return;
      ptx::tc_fence_after();
      const uint64_t dDo_mn = ptx::desc_sw128(dobase, L::kBlk, 1024);
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks)  // dV += P^T dO (P^T of half h at 64 h)
        ptx::mma_ts(tDV, tS + (ks >> 2) * 64 + (ks & 3) * 8, dDo_mn + ((ks * 2048) >> 4), kIdAcc,
                    (j > 0 || ks > 0) ? 1u : 0u);
      ptx::mma_commit(bar(L::DVD));
      if (j + 1 < w.n && !issue_s(g + 1)) return;  // next query tile of this unit
      if (!wait_bar(bar(L::DSR), g & 1u, ctl)) return;
      ptx::tc_fence_after();
      const uint64_t dQ_mn = ptx::desc_sw128(qbase, L::kBlk, 1024);
      const uint64_t dDs_mn = ptx::desc_sw128(dobase, L::kBlk, 1024);
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks)  // dK += dS^T Q (dS^T of half h at 64 h)
        ptx::mma_ts(tDK, tDP + (ks >> 2) * 64 + (ks & 3) * 8, dQ_mn + ((ks * 2048) >> 4),
                    kIdAcc, (j > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < kBM / 16; ++ks)  // dQ = dS K (over this tile's keys)
        ptx::mma_ss(tDP, dDs_mn + ((ks * 2048) >> 4), dK_mn + ((ks * 2048) >> 4), kIdDq,
                    ks > 0 ? 1u : 0u);
      ptx::mma_commit(bar(L::DQF));
      ptx::mma_commit(bar(L::QE0 + st));  // Q and the S bias no longer read
      if (j == w.n - 1) {
        ptx::mma_commit(bar(L::OF));
        ptx::mma_commit(bar(L::KVE));
      }
    }
    ++u_cnt;
  }
}

// ------------------------------------------------------------------- load
struct BwdLoadLog {
  FillLog<1> kv;
  FillLog<2> q, dout;
};

// Every issued fill is recorded in `f` (see FillLog).
template <int D, bool VARLEN>
__device__ void load_loop(const BwdParams& p, uint32_t smem, uint32_t bars, const Ctl& ctl,
                          BwdLoadLog& f) {
  using L = BLayout<D>;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t g = 0, kv_cnt = 0;
  BUnit w;
  bwd_walk<VARLEN>(p, w, true);
  for (int k = 0; bwd_unit<VARLEN>(p, k, w, true); ++k) {
    if (w.n == 0) continue;
    if (kv_cnt > 0 && !wait_bar(bar(L::KVE), (kv_cnt - 1) & 1u, ctl)) return;
    ptx::mbar_arrive_expect_tx(bar(L::KVF), 2 * L::kTile);
    const int krow = w.k_start + w.kt * kBM;
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk) {
      ptx::tma_load_3d(smem + L::kKOff + blk * L::kBlk, &p.tm_k, bar(L::KVF), blk * 64, w.h, krow);
      ptx::tma_load_3d(smem + L::kVOff + blk * L::kBlk, &p.tm_v, bar(L::KVF), blk * 64, w.h, krow);
    }
    f.kv.last[0] = static_cast<int>(kv_cnt);
    ++kv_cnt;
    for (int j = 0; j < w.n; ++j, ++g) {
      const uint32_t st = g & 1u;
      const int qrow = w.q_start + (w.i0 + j) * kBN;
      const long long tile = static_cast<long long>(w.tile0) * p.H +
                             static_cast<long long>(w.h) * ((w.Lq + kBN - 1) / kBN) + w.i0 + j;
      // Q tile and S bias
      if (g >= 2 && !wait_bar(bar(L::QE0 + st), ((g >> 1) - 1) & 1u, ctl)) return;
      ptx::mbar_arrive_expect_tx(bar(L::QF0 + st), L::kTile + kBiasBytes);
      bulk_load(smem + L::kBiasOff + st * 2 * kBiasBytes, p.bias + tile * 2 * kBiasBytes,
                kBiasBytes, bar(L::QF0 + st));
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        ptx::tma_load_3d(smem + L::kQOff + st * L::kTile + blk * L::kBlk, &p.tm_q,
                         bar(L::QF0 + st), blk * 64, w.h, qrow);
      f.q.last[st] = static_cast<int>(g);
      // dO tile and D bias
      if (g >= 2 && !wait_bar(bar(L::DOE0 + st), ((g >> 1) - 1) & 1u, ctl)) return;
      ptx::mbar_arrive_expect_tx(bar(L::DOF0 + st), L::kTile + kBiasBytes);
      bulk_load(smem + L::kBiasOff + (st * 2 + 1) * kBiasBytes,
                p.bias + tile * 2 * kBiasBytes + kBiasBytes, kBiasBytes, bar(L::DOF0 + st));
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        ptx::tma_load_3d(smem + L::kDoOff + st * L::kDoStage + blk * L::kBlk, &p.tm_do,
                         bar(L::DOF0 + st), blk * 64, w.h, qrow);
      f.dout.last[st] = static_cast<int>(g);
    }
  }
}

template <int D, bool BF16, bool VARLEN>
__global__ void __maxnreg__(128) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
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
      const uint32_t count = (i == L::PR || i == L::DSR) ? 32u * kDsWarps
                             : (i == L::DQE || i == L::AE || i == L::STG) ? 128u
                                                                            : 1u;
      ptx::mbar_init(bars + 8u * i, count);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (threadIdx.x < kBM) {  // the ones column of the bias products: k = 0, 1, 2 are 1.0 (bf16)
    uint8_t* const ones = base + L::kOnesOff;
    const int r = threadIdx.x;
    *reinterpret_cast<uint4*>(ones + bias_offset(r, 0)) =
        make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u);
    *reinterpret_cast<uint4*>(ones + bias_offset(r, 8)) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
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

  if (warp < kDsWarps) {
    ds_role<D, BF16, VARLEN>(p, tmem, base, bars, ctl);
  } else if (warp < kMmaWarp) {
    dq_role<D, BF16, VARLEN>(p, tmem, smem, base, bars, ctl);
    if (threadIdx.x == kDqWarp0 * 32) bulk_wait_all();  // every reduce-add landed
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      mma_loop<D, BF16, VARLEN>(p, smem, tmem, bars, ctl);
      const uint32_t done = bars + 8u * L::DONE;
      ptx::mma_commit(done);
      wait_bar(done, 0, ctl, false);
    }
  } else if (lane == 0) {
    BwdLoadLog f;
    f.kv.clear();
    f.q.clear();
    f.dout.clear();
    load_loop<D, VARLEN>(p, smem, bars, ctl, f);
    // no TMA or bulk copy may land after the CTA exits
    drain_fills(bars, L::KVF, f.kv, ctl);
    drain_fills(bars, L::QF0, f.q, ctl);
    drain_fills(bars, L::DOF0, f.dout, ctl);
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------ pre- and post-processing
// v = hi + mid + lo in bf16 (the residual of three parts is about 2^-27 |v|).
__device__ __forceinline__ void split3_bf16(float v, uint16_t (&out)[kBiasParts]) {
  float rest = v;
#pragma unroll
  for (int i = 0; i < kBiasParts; ++i) {
    const __nv_bfloat16 b = __float2bfloat16_rn(rest);
    out[i] = __bfloat16_as_ushort(b);
    rest -= __bfloat162float(b);
  }
}

// One warp, one query row: row r of the bias tile t, the two per-query terms
// -LSE/scale (S^T) and -D with D = sum_d dO * O (dP^T), each split in three
// bf16 parts at k = 0, 1, 2 of the row (k = 3..15 zero).  orow < 0: a padding
// row past the sequence, all zero.  A row without keys (LSE = -inf) is seen by
// no work unit; its terms are written as zero.
template <int D, bool BF16>
__device__ __forceinline__ void bias_row(const uint16_t* __restrict__ o,
                                         const uint16_t* __restrict__ dout, long long orow,
                                         const float* lse_elem, float scale, uint8_t* t, int r) {
  const int lane = threadIdx.x & 31;
  float dsum = 0.0f, nls = 0.0f;
  if (orow >= 0) {
    constexpr int PER = D / 32;  // 2 or 4 elements per lane
    const uint16_t* a = o + orow * D + lane * PER;
    const uint16_t* c = dout + orow * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; i += 2) {
      float x0, x1, y0, y1;
      unpack2<BF16>(*reinterpret_cast<const uint32_t*>(a + i), x0, x1);
      unpack2<BF16>(*reinterpret_cast<const uint32_t*>(c + i), y0, y1);
      dsum = fmaf(x0, y0, fmaf(x1, y1, dsum));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
    const float l = *lse_elem;
    nls = isfinite(l) ? -l / scale : 0.0f;
  }
  if (lane == 0) {
    uint16_t sp[kBiasParts], dp[kBiasParts];
    split3_bf16(nls, sp);
    split3_bf16(-dsum, dp);
    *reinterpret_cast<uint4*>(t + bias_offset(r, 0)) =
        make_uint4(sp[0] | (static_cast<uint32_t>(sp[1]) << 16), sp[2], 0u, 0u);
    *reinterpret_cast<uint4*>(t + bias_offset(r, 8)) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(t + kBiasBytes + bias_offset(r, 0)) =
        make_uint4(dp[0] | (static_cast<uint32_t>(dp[1]) << 16), dp[2], 0u, 0u);
    *reinterpret_cast<uint4*>(t + kBiasBytes + bias_offset(r, 8)) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Dense sequences: every row (b, h, q) of every query tile, q < Sq padded to
// whole tiles; tile (b * H + h) * nq + q / 128.  One warp per row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(const uint16_t* __restrict__ o,
                                                           const uint16_t* __restrict__ dout,
                                                           const float* __restrict__ lse,
                                                           uint8_t* __restrict__ bias, int B,
                                                           int H, int Sq, float scale) {
  const int nq = (Sq + kBN - 1) / kBN;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(B) * H * nq * kBN) return;  // row = (b*H + h) * nq*128 + q
  const int q = static_cast<int>(row % (static_cast<long long>(nq) * kBN));
  const long long bh = row / (static_cast<long long>(nq) * kBN);
  const int h = static_cast<int>(bh % H);
  const int b = static_cast<int>(bh / H);
  const bool real = q < Sq;
  bias_row<D, BF16>(o, dout, real ? (static_cast<long long>(b) * Sq + q) * H + h : -1,
                    real ? lse + bh * Sq + q : nullptr, scale,
                    bias + (bh * nq + q / kBN) * 2 * kBiasBytes, q % kBN);
}

// Packed sequences, one block of 1024 threads: tiles[b] = the 128-query tiles
// of sequences 0 .. b-1 (b = 0..B) and tiles[B + 1] = 1 when every sequence's
// bounds are well formed (0 <= cu_q[b] <= cu_q[b+1] <= Sq, the same for cu_k),
// else 0 and the error word reports ATTN_ERR_BAD_SEQLENS.  Well-formed bounds
// tile at most Sq rows, so tiles[B] <= (Sq + 127 B) / 128.
static __global__ void __launch_bounds__(1024)
    attn_bwd_tiles_kernel(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k,
                          int B, int Sq, int Sk, int32_t* __restrict__ tiles, int* err) {
  __shared__ int part[1024];
  __shared__ int bad;
  const int t = threadIdx.x;
  if (t == 0) bad = 0;
  __syncthreads();
  auto count = [&](int b, bool& ok) {
    const int q0 = __ldg(cu_q + b), q1 = __ldg(cu_q + b + 1);
    const int k0 = __ldg(cu_k + b), k1 = __ldg(cu_k + b + 1);
    ok = 0 <= q0 && q0 <= q1 && q1 <= Sq && 0 <= k0 && k0 <= k1 && k1 <= Sk;
    return ok ? (q1 - q0 + kBN - 1) / kBN : 0;
  };
  const int per = (B + 1023) / 1024;
  const int b0 = min(B, t * per), b1 = min(B, b0 + per);
  int sum = 0;
  bool any_bad = false;
  for (int b = b0; b < b1; ++b) {
    bool ok;
    sum += count(b, ok);
    any_bad |= !ok;
  }
  if (any_bad) atomicOr(&bad, 1);
  part[t] = sum;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan of part[]
    const int v = t >= off ? part[t - off] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  int run = part[t] - sum;
  for (int b = b0; b < b1; ++b) {
    tiles[b] = run;
    bool ok;
    run += count(b, ok);
  }
  if (t == 1023) {
    tiles[B] = part[1023];
    tiles[B + 1] = bad ? 0 : 1;
    if (bad) atomicOr(err, kErrBadSeqlens);
  }
}

// Packed sequences: every row of every query tile (tiles[B] * H tiles of 128
// rows); tile t = tiles[b] * H + h * nq(b) + i belongs to the largest b with
// tiles[b] * H <= t.  Rows past the sequence are zero.  One warp per row;
// nothing when the bounds were malformed.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_pre_varlen_kernel(
    const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
    const float* __restrict__ lse, uint8_t* __restrict__ bias, const int32_t* __restrict__ tiles,
    const int32_t* __restrict__ cu_q, int B, int H, int Tq, float scale) {
  if (__ldg(tiles + B + 1) == 0) return;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= static_cast<long long>(__ldg(tiles + B)) * H * kBN) return;
  const long long t = row / kBN;
  const int r = static_cast<int>(row - t * kBN);
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<long long>(__ldg(tiles + mid)) * H <= t) lo = mid;
    else hi = mid - 1;
  }
  const int tb = __ldg(tiles + lo);
  const int nq = __ldg(tiles + lo + 1) - tb;  // > 0: tile t lies in sequence lo's range
  const long long rem = t - static_cast<long long>(tb) * H;
  const int h = static_cast<int>(rem / nq);
  const int i = static_cast<int>(rem - static_cast<long long>(h) * nq);
  const int q0 = __ldg(cu_q + lo), lq = __ldg(cu_q + lo + 1) - q0;
  const int pos = i * kBN + r;
  const bool real = pos < lq;
  const long long q = static_cast<long long>(q0) + pos;
  bias_row<D, BF16>(o, dout, real ? q * H + h : -1,
                    real ? lse + static_cast<long long>(h) * Tq + q : nullptr, scale,
                    bias + t * 2 * kBiasBytes, r);
}

// dQ[b, q, h, :] = scale * acc[b, h, q, :] in the input dtype; packed
// sequences are one batch of Tq rows (B = 1, Sq = Tq; rows of no sequence: 0).
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const float* __restrict__ acc,
                                                            uint16_t* __restrict__ dq, int B,
                                                            int H, int Sq, float scale) {
  const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;  // pair index
  const long long n = static_cast<long long>(B) * H * Sq * (D / 2);
  if (i >= n) return;
  const int d2 = static_cast<int>(i % (D / 2));
  const long long row = i / (D / 2);  // dense (b * H + h) * Sq + q; packed h * Sq + q
  const int q = static_cast<int>(row % Sq);
  const long long bh = row / Sq;
  const int h = static_cast<int>(bh % H);
  const int b = static_cast<int>(bh / H);
  const float2 v = reinterpret_cast<const float2*>(acc)[i];
  const uint32_t pk = ptx::pack2<BF16>(v.x * scale, v.y * scale);
  reinterpret_cast<uint32_t*>(dq)[((static_cast<long long>(b) * Sq + q) * H + h) * (D / 2) + d2] =
      pk;
}

// The four launches of one backward.  Dense: bias holds B*H*nq tiles.  Packed
// (p.varlen): bias holds tiles_bound*H tiles, p.tiles B + 2 ints, and the
// accumulator is [H, Tq, D] (Tq = p.Sq rows).
template <int D, bool BF16>
cudaError_t launch_bwd(const BwdParams& p, const uint16_t* o, const uint16_t* dout,
                       const float* lse, uint8_t* bias, int32_t* tiles, long long tiles_bound,
                       uint16_t* dq, int grid, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.Tq) * p.H;
  cudaError_t e = cudaMemsetAsync(p.dq_acc, 0, static_cast<size_t>(rows) * D * sizeof(float),
                                  stream);
  if (e != cudaSuccess) return e;
  if (p.varlen) {
    attn_bwd_tiles_kernel<<<1, 1024, 0, stream>>>(p.cu_q, p.cu_k, p.B, p.Sq, p.Sk, tiles, p.err);
    const long long prow = tiles_bound * p.H * kBN;
    attn_bwd_pre_varlen_kernel<D, BF16><<<static_cast<unsigned>((prow + 7) / 8), 256, 0, stream>>>(
        o, dout, lse, bias, tiles, p.cu_q, p.B, p.H, p.Tq, p.scale);
  } else {
    const long long prow = static_cast<long long>(p.B) * p.H * ((p.Sq + kBN - 1) / kBN) * kBN;
    attn_bwd_pre_kernel<D, BF16><<<static_cast<unsigned>((prow + 7) / 8), 256, 0, stream>>>(
        o, dout, lse, bias, p.B, p.H, p.Sq, p.scale);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // packed sequences walk their bounds; the dense instantiation has no walk
  const void* fn = p.varlen ? reinterpret_cast<const void*>(&attn_bwd_kernel<D, BF16, true>)
                            : reinterpret_cast<const void*>(&attn_bwd_kernel<D, BF16, false>);
  static std::atomic<unsigned long long> opted[2] = {{0}, {0}};
  e = smem_opt_in(fn, BLayout<D>::kAlloc, opted[p.varlen ? 1 : 0]);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<BwdParams*>(&p)};
  e = cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, BLayout<D>::kAlloc, stream);
  if (e != cudaSuccess) return e;
  const long long pairs = rows * (D / 2);
  attn_bwd_post_kernel<D, BF16><<<static_cast<unsigned>((pairs + 255) / 256), 256, 0, stream>>>(
      p.dq_acc, dq, p.varlen ? 1 : p.B, p.H, p.varlen ? p.Tq : p.Sq, p.scale);
  return cudaGetLastError();
}

}  // namespace bwd
}  // namespace attn
