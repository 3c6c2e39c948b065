// Fused attention forward for sm_103a: one persistent, warp-specialised kernel.
//
// What it computes (per sequence b, head h, query row i):
//   O_i   = sum_j softmax_j(scale * q_i . k_j) v_j   over the visible keys j
//   LSE_i = ln sum_j exp(scale * q_i . k_j)
// Definition: page "Multi-Head Attention的计算本质与性能瓶颈", §1/§2.1; causal
// rule (key j visible iff j <= i) from §3.1 of the same page; varlen packing
// from page "长文本处理性能断层真相", §1.  The scores are consumed tile by tile
// with the online softmax of page "深度学习算子优化：从TFLOPS幻觉到
// FlashAttention实战", §3 (running row max m_i, running exp-sum l_i, rescale of
// the accumulator, one final normalisation), so S never reaches global memory.
//
// GB300 mapping (the pages' A100 sketches are prior art only):
//   * work unit = (sequence, head, 256 query rows) = two 128-row query tiles
//     that share every K/V tile; persistent grid, units dealt in snake order,
//     head-major with the heaviest causal units of each head first;
//   * warp 9 (one lane) streams Q, K, V with 3-D TMA into 128-byte-swizzled
//     shared memory, K and V each in a ring of kStages buffers;
//   * warp 8 (one lane) issues tcgen05.mma: S_t = Q_t K^T (both operands in
//     shared memory) and O_t += P_t V (P read from tensor memory);
//   * warps 0-3 / 4-7 run the softmax of query tile 0 / 1, one thread per
//     query row (= one TMEM lane), so row max and row sum need no shuffles;
//     they write P (16-bit) over the S columns in TMEM and rescale O in TMEM
//     only when the running max grows by more than 2^8;
//   * TMEM: S0 | S1 | O0 | O1 columns; P_t aliases the first 64 columns of S_t.
// Every pipeline wait is bounded: on expiry the kernel records an error in a
// device word, tells the other roles through a shared flag and winds down.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace attn {

constexpr int kBM = 128;                 // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;                 // keys per K/V tile
constexpr int kTiles = 2;                // query tiles per work unit
constexpr int kUnitRows = kBM * kTiles;  // query rows per work unit
constexpr int kThreads = 320;            // 8 softmax warps + MMA warp + load warp
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kTileSoftmaxWarps = 8;     // warps 0-3: query tile 0, warps 4-7: query tile 1
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;     // rescale O only if max grows by > 2^8
constexpr int kUnbounded = 1 << 30;      // window side without a bound

enum : int { kErrTimeout = 1, kErrBadSeqlens = 2 };

struct FwdParams {
  CUtensorMap tm_q;          // [rows_q, H, D] 16-bit, box 128 x 1 x 64
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_kh;         // K with a 64-row box (pair kernel: each CTA loads half a tile)
  CUtensorMap tm_vh;         // V halves of the pair kernel: box D/2 x 1 x 128, D-byte swizzle
  void* o;
  float* lse;
  const int32_t* cu_q;       // varlen only
  const int32_t* cu_k;
  int* err;                  // device error word (bit flags above)
  int B, H, Sq, Sk;          // dense: per-batch lengths; varlen: total packed rows
  int varlen, causal;
  // Visibility of key j to query i (indices within the sequence): rows
  // i >= global_q see keys i - win_left <= j <= i + win_right; rows
  // i < global_q see every key (j <= i when causal).  An unbounded side is
  // kUnbounded; causal sets win_right = 0.
  int win_left, win_right, global_q;
  float scale_log2;          // scale * log2(e)
  int scale_pos;             // scale > 0: fold the scale into the exp2 argument
  long long timeout_ns;      // limit for any single pipeline wait
  // Schedule items pair the row blocks i and nU-1-i of one (sequence, head)
  // (see decode_rows); set by the host when the units far outnumber the workers.
  int pair_blocks = 0;
  // Dense calls only: units ordered row block first, (batch, head) second
  // (see decode_rows); set by the host when every head's K and V fit in L2
  // together, so that no head needs its CTAs to run side by side.
  int block_major = 0;
  // Offset (from the 1024-aligned origin of the dynamic shared memory) of the
  // packed-sequence walk order, past every other buffer of the kernel; set by
  // the host, which adds kOrderBytes to the launch when the order is used.
  int order_off = 0;
  // Fault injection for the failure-detection tests (0 in normal use): 1 makes
  // the loader of CTA 0 skip its first K tile, so a bounded wait runs out.
  int inject = 0;
};

constexpr int kDescSlots = 4;     // unit descriptors in flight (single-CTA kernel)

template <int D>
struct Layout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kBlk = 16384;                  // 128 rows x 128 B swizzle block
  static constexpr int kTileBytes = (D / 64) * kBlk;  // one 128-row tile, all of D
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTiles * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  // barrier indices
  static constexpr int QF = 0, QE = 1, KF = 2, KE = KF + kStages, VF = KE + kStages,
                       VE = VF + kStages, SF = VE + kStages, PF = SF + 2, OF = PF + 2,
                       DONE = OF + 2, DRY = DONE + 1, DFR = DRY + kDescSlots,
                       kNumBars = DFR + kDescSlots;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;  // tmem base, abort flag
  // Ring of unit descriptors the loader publishes for the softmax warps (unit
  // k in slot k % kDescSlots: "ready" DRY + slot, "free" DFR + slot).
  static constexpr int kDescOff = kMiscOff + 16;
  static constexpr int kBytes = kDescOff + kDescSlots * 48;
  static constexpr int kAlloc = kBytes + 1024;             // slack for 1024-B alignment
  // TMEM columns
  static constexpr uint32_t kColS = 0, kColO = 256;
};

// ------------------------------------------------------------ bounded waits
struct Ctl {
  volatile int* abort_flag;  // shared memory
  int* err;
  long long timeout_ns;
};

// Polls `bar` for the phase of the given parity.  Gives up (returning false)
// when another role has raised the abort flag, or after c.timeout_ns, in which
// case it raises the flag and records kErrTimeout.  With honor_abort == false
// only the time limit applies (used to drain work already in flight).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c,
                                         bool honor_abort = true) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
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

// Index of the last copy issued into each buffer of a ring (-1: none).  A
// loader records every fill when it issues it; after its loop ends, also when
// it was abandoned half-way through a unit, it waits for exactly the fills
// that may still be in flight (one per buffer: a buffer is refilled only after
// its previous fill has landed and been consumed).
template <int N>
struct FillLog {
  int last[N];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < N; ++i) last[i] = -1;
  }
};

// Bounded waits, ignoring the abort flag, for the last fill of each buffer of
// a ring whose "full" barriers are full0, full0 + 1, ... (fill i completes
// phase i / N of barrier i % N).
template <int N>
__device__ __forceinline__ void drain_fills(uint32_t bars, int full0, const FillLog<N>& f,
                                            const Ctl& ctl) {
#pragma unroll 1
  for (int st = 0; st < N; ++st)
    if (f.last[st] >= 0)
      wait_bar(bars + 8u * (full0 + st), (static_cast<uint32_t>(f.last[st]) / N) & 1u, ctl,
               false);
}

// All 32 lanes wait; the warp proceeds only if every lane saw the phase.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Ctl& c) {
  const bool ok = wait_bar(bar, parity, c);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------- work units
struct Unit {
  int b, h;                   // sequence, head
  int q0;                     // first query row of the unit within the sequence (may be < 0)
  int q_start, Lq, k_start, Lk;
  int j0;                     // first K/V tile visited (step j reads tile j0 + j)
  int n[kTiles];              // K/V tiles visited by each query tile
  bool valid[kTiles];         // tile holds at least one real query row
};

struct Cursor {               // forward-only walk over varlen sequences
  int b, base, units;         // b: position in the walk order
  int seq;                    // the sequence at position b
  int q_start, Lq, k_start, Lk;
  const int* order;           // walk order in shared memory, or null (given order)
};

// Packed sequences are walked longest first (by Lq * Lk) when there are at
// most kMaxOrderedSeqs of them, so that the last items dealt to the workers
// are the cheapest ones and the loads end close together; every CTA ranks the
// sequences itself at its start (build_seq_order).  Larger batches keep their
// given order.  The order and the ranking keys live in dynamic shared memory
// at FwdParams::order_off (static shared memory is avoided: on GB300 even
// 1 KB of it slowed these kernels by 3-4 %).
constexpr int kMaxOrderedSeqs = 256;
constexpr int kOrderBytes = kMaxOrderedSeqs * (4 + 8);

__host__ __device__ __forceinline__ bool seq_ordered(const FwdParams& p) {
  return p.varlen && p.B <= kMaxOrderedSeqs;
}

// 1024-aligned origin of the dynamic shared memory (the kernels' layouts start here).
__device__ __forceinline__ uint8_t* smem_origin() {
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t raw = ptx::smem_u32(smem_dyn);
  return smem_dyn + (((raw + 1023u) & ~1023u) - raw);
}

// Called by every thread of the CTA before the barrier that ends the kernel's
// prologue.  Sequence b gets position #{b' : key(b') > key(b), or key(b') ==
// key(b) and b' < b} (a permutation, also for malformed offsets, which
// load_seq reports when the walk gets there).  Its own barrier is reached by
// every launch, ordered or not: a barrier under a condition made the compiler
// treat the whole kernel's control flow more conservatively (3-6 % slower,
// measured).
__device__ __forceinline__ void build_seq_order(const FwdParams& p) {
  const bool ordered = seq_ordered(p);
  int* const order = reinterpret_cast<int*>(smem_origin() + p.order_off);
  long long* const key = reinterpret_cast<long long*>(order + kMaxOrderedSeqs);
  for (int b = threadIdx.x; ordered && b < p.B; b += blockDim.x) {
    const long long lq = __ldg(p.cu_q + b + 1) - __ldg(p.cu_q + b);
    const long long lk = __ldg(p.cu_k + b + 1) - __ldg(p.cu_k + b);
    key[b] = lq * lk;
  }
  __syncthreads();
  for (int b = threadIdx.x; ordered && b < p.B; b += blockDim.x) {
    const long long kb = key[b];
    int r = 0;
    for (int x = 0; x < p.B; ++x) {
      const long long kx = key[x];
      r += (kx > kb || (kx == kb && x < b)) ? 1 : 0;
    }
    order[r] = b;
  }
}

template <int UR>
__device__ __forceinline__ void load_seq(const FwdParams& p, Cursor& c, bool report) {
  c.units = 0;
  c.q_start = c.Lq = c.k_start = c.Lk = 0;
  if (c.b >= p.B) return;
  c.seq = c.order ? c.order[c.b] : c.b;
  const int q0 = __ldg(p.cu_q + c.seq), q1 = __ldg(p.cu_q + c.seq + 1);
  const int k0 = __ldg(p.cu_k + c.seq), k1 = __ldg(p.cu_k + c.seq + 1);
  const bool ok = 0 <= q0 && q0 <= q1 && q1 <= p.Sq && 0 <= k0 && k0 <= k1 && k1 <= p.Sk;
  if (!ok) {
    if (report) atomicOr(p.err, kErrBadSeqlens);
    return;
  }
  c.q_start = q0;
  c.Lq = q1 - q0;
  c.k_start = k0;
  c.Lk = k1 - k0;
  const int nU = (c.Lq + UR - 1) / UR;
  c.units = p.H * (p.pair_blocks ? (nU + 1) / 2 : nU);  // schedule items of this sequence
}

// VL = false compiles the walk for dense batches only (p.varlen must be 0).
template <int UR, bool VL = true>
__device__ __forceinline__ void init_cursor(const FwdParams& p, Cursor& c, bool report) {
  c.b = 0;
  c.base = 0;
  c.seq = 0;
  c.order = VL && seq_ordered(p) ? reinterpret_cast<const int*>(smem_origin() + p.order_off)
                                  : nullptr;
  if (VL && p.varlen) load_seq<UR>(p, c, report);
}

// Row block `blk` of a sequence, or no rows at all (empty).  Under a causal
// mask the blocks are aligned to the end of the sequence (block nU-1 ends at
// the last row), so a partial block holds the first rows, which see the fewest
// keys; its rows before row 0 are computed as fully masked rows and never
// written.  Without a causal mask blocks start at row 0.
template <int UR>
__device__ __forceinline__ void set_block(const FwdParams& p, Unit& w, int nU, int blk,
                                          bool empty) {
  const int off = p.causal ? w.Lq - nU * UR : 0;
  w.q0 = empty ? w.Lq : off + blk * UR;
}

// Decodes unit u (units are visited in increasing order by each worker) into
// its sequence, head and block of UR query rows.
// Order: (sequence, head) outer, row blocks inner.  Keeping one head's blocks
// together keeps the K/V tiles that the concurrently running workers stream
// within L2 (one head of a 64K-token sequence is 32 MB).  A dense call whose
// K and V fit in L2 as a whole (p.block_major) orders row blocks outer and
// (batch, head) inner instead: the blocks then come heaviest first across all
// heads, so the snake deal ends level even with few units per worker.  Without
// p.pair_blocks, u enumerates the blocks of a (sequence, head), heaviest
// causal block first.  With p.pair_blocks, u = 2 s + part: schedule item s
// holds block nU-1-i (part 0, the heaviest under a causal mask) and block i
// (part 1) of one (sequence, head), so that every item of a (sequence, head)
// costs about the same; the middle block of an odd nU stands alone and its
// part 1 is empty.  Items are dealt to the workers in a snake order (see
// slot_unit).
template <int UR, bool VL = true>
__device__ __forceinline__ bool decode_rows(const FwdParams& p, int u, Cursor& c, Unit& w,
                                            bool report) {
  const int s = p.pair_blocks ? (u >> 1) : u;  // schedule item
  int nU, i;
  if (!VL || !p.varlen) {
    nU = (p.Sq + UR - 1) / UR;
    const int per = p.pair_blocks ? (nU + 1) / 2 : nU;
    const int heads = p.B * p.H;
    if (s >= heads * per) return false;
    int bh;
    if (p.block_major) {
      i = s / heads;
      bh = s - i * heads;
    } else {
      bh = s / per;
      i = s - bh * per;
    }
    w.b = bh / p.H;
    w.h = bh - w.b * p.H;
    w.q_start = w.b * p.Sq;
    w.Lq = p.Sq;
    w.k_start = w.b * p.Sk;
    w.Lk = p.Sk;
  } else {
    while (true) {
      if (c.b >= p.B) return false;
      if (s < c.base + c.units) break;
      c.base += c.units;
      c.b += 1;
      load_seq<UR>(p, c, report);
    }
    const int rem = s - c.base;
    const int per = c.units / p.H;
    w.h = rem / per;
    i = rem - w.h * per;
    nU = (c.Lq + UR - 1) / UR;
    w.b = c.seq;
    w.q_start = c.q_start;
    w.Lq = c.Lq;
    w.k_start = c.k_start;
    w.Lk = c.Lk;
  }
  if (p.pair_blocks) {
    const bool second = (u & 1) != 0;
    set_block<UR>(p, w, nU, second ? i : nU - 1 - i, second && i == nU - 1 - i);
  } else {
    set_block<UR>(p, w, nU, p.causal ? nU - 1 - i : i, false);
  }
  return true;
}

// K/V tiles [lo, hi) holding every key that some row of the 128-row query
// tile starting at row q0 (which may be negative: rows before 0 do not exist)
// can see (hi <= lo: none).  Tiles outside the range are never loaded or
// multiplied; keys inside it that a row cannot see are masked in the softmax.
__device__ __forceinline__ void tile_keys(const FwdParams& p, const Unit& w, int q0, int& lo,
                                          int& hi) {
  lo = hi = 0;
  const int r0 = max(q0, 0);
  if (r0 >= w.Lq || q0 + kBM <= 0) return;
  const int q1 = min(q0 + kBM, w.Lq) - 1;
  const int nk = (w.Lk + kBN - 1) / kBN;
  if (r0 < p.global_q) {  // rows that see every key (up to the diagonal when causal)
    hi = p.causal ? min(nk, q1 / kBN + 1) : nk;
    return;
  }
  // rows r0..q1 see keys r0 - win_left .. q1 + win_right
  lo = max(0, r0 - p.win_left) / kBN;
  hi = static_cast<int>(min(static_cast<long long>(nk),
                            (static_cast<long long>(q1) + p.win_right) / kBN + 1));
}

// Keys lo..hi (inclusive, indices within the sequence) that query row qrow
// may see; once per unit.  Step j masks columns c of tile j0 + j outside
// lo - kb .. hi - kb, kb = (j0 + j) * 128.
__device__ __forceinline__ void row_keys(const FwdParams& p, const Unit& w, int qrow, int& lo,
                                         int& hi) {
  hi = w.Lk - 1;
  lo = 0;
  if (qrow >= p.global_q) {  // qrow + win_right and qrow - win_left without overflow
    hi = qrow > hi - p.win_right ? hi : qrow + p.win_right;
    lo = qrow > p.win_left ? qrow - p.win_left : 0;
  } else if (p.causal) {
    hi = min(hi, qrow);
  }
}

template <bool VL = true>
__device__ __forceinline__ bool decode_unit(const FwdParams& p, int u, Cursor& c, Unit& w,
                                            bool report) {
  if (!decode_rows<kUnitRows, VL>(p, u, c, w, report)) return false;
  int lo[kTiles], hi[kTiles];
  w.j0 = -1;
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    const int q0 = w.q0 + t * kBM;
    w.valid[t] = q0 + kBM > 0 && q0 < w.Lq;
    tile_keys(p, w, q0, lo[t], hi[t]);
    if (w.j0 < 0 && w.valid[t]) w.j0 = lo[t];
  }
  // both query tiles walk the K/V tiles from the first one either needs (that
  // of the first tile with rows); each stops at its own last tile
  if (w.j0 < 0) w.j0 = 0;
#pragma unroll
  for (int t = 0; t < kTiles; ++t) w.n[t] = w.valid[t] ? max(0, hi[t] - w.j0) : 0;
  return true;
}

// The k-th unit of worker c out of g: units are dealt in rounds of g, left to
// right in even rounds and right to left in odd rounds, so that the worker
// that got the heaviest unit of one round gets the lightest of the next.
__device__ __forceinline__ int unit_of(int k, int g, int c) {
  return k * g + ((k & 1) ? (g - 1 - c) : c);
}
__device__ __forceinline__ int unit_of(int k) {
  return unit_of(k, static_cast<int>(gridDim.x), static_cast<int>(blockIdx.x));
}

// The unit of the forward kernels' k-th slot of worker c out of g: with paired
// blocks, slots 2m and 2m+1 hold the two blocks of the worker's m-th schedule
// item (items dealt in the snake order of unit_of); otherwise the units
// themselves are dealt that way.
__device__ __forceinline__ int slot_unit(const FwdParams& p, int k, int g, int c) {
  return p.pair_blocks ? 2 * unit_of(k >> 1, g, c) + (k & 1) : unit_of(k, g, c);
}
__device__ __forceinline__ int slot_unit(const FwdParams& p, int k) {
  return slot_unit(p, k, static_cast<int>(gridDim.x), static_cast<int>(blockIdx.x));
}

// ---------------------------------------------------------------- softmax
// x rounded to the 16-bit input type (nearest even) and back to fp32.
template <bool BF16>
__device__ __forceinline__ float round16(float x) {
  const uint32_t pk = ptx::pack2<BF16>(x, 0.0f);  // x in the low half
  float y;
  if constexpr (BF16) {
    y = __uint_as_float(pk << 16);
  } else {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}"
        : "=f"(y) : "r"(pk));
  }
  return y;
}

// Running state of one query row.  l_x sums the unrounded P values (it gives
// the logsumexp).  l_p normalises O: the 16-bit kernels keep the same exact sum
// plus, once per tile, the rounding error of the largest value a thread
// writes (in a peaked row the largest values carry the rounding that shows
// in O; the rounding of the rest averages out); the FP8 kernel sums the
// rounded values themselves.
struct RowState {
  float m;    // running max, log2 units (scale * log2e * s)
  float l_p;
  float l_x;
};

// One K/V tile of the online softmax for the calling thread's query row.
// S is read from TMEM (128 fp32 columns), masked (keys c < lo or c > limit are
// invisible),
// turned into P = 2^(scale*log2e*s - m) rounded to 16 bits and written back over
// the first 64 columns of S.  O is rescaled in TMEM when the running max moved
// by more than 2^kRescaleLog2; otherwise the stale max is kept for P and l,
// which leaves the result exact.
// pvd_bar != 0: before rescaling O, wait (parity pvd_parity) for the MMA that
// accumulates the previous tile into O; returns false if that wait gave up.
template <int D, bool BF16>
__device__ __forceinline__ bool softmax_step_pv(uint32_t tS, uint32_t tO, int lo, int limit,
                                                float cl,
                                                bool scale_pos, bool first, RowState& st,
                                                uint32_t pvd_bar, uint32_t pvd_parity,
                                                const Ctl& ctl) {
  uint32_t r[128];
  ptx::tmem_ld_x128(tS, r);
  float cle = cl;
  if (!scale_pos) {  // scale <= 0: scale first so that "max" stays a max
    const uint64_t c2 = ptx::f2(cl, cl);
#pragma unroll
    for (int c = 0; c < 128; c += 2) {
      float a, b;
      ptx::f2_split(ptx::f2_mul(ptx::f2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), c2),
                    a, b);
      r[c] = __float_as_uint(a);
      r[c + 1] = __float_as_uint(b);
    }
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
  const float r_max = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));  // this row's largest score
  const float m_tile = r_max * cle;
  const float m_new = fmaxf(st.m, m_tile);
  const bool rescale = m_new > st.m + kRescaleLog2;  // always true on the first tile
  const float m_use = rescale ? m_new : st.m;
  const float m_safe = (m_use == -INFINITY) ? 0.0f : m_use;
  const float alpha = rescale ? ptx::ex2(st.m - m_safe) : 1.0f;
  st.m = m_use;

  // the rounding error of the largest value, computed exactly as in the loop:
  // it joins O's denominator
  const float p_big = ptx::ex2(fmaf(r_max, cle, -m_safe));
  const float corr = round16<BF16>(p_big) - p_big;
  const uint64_t cl2 = ptx::f2(cle, cle);
  const uint64_t nm2 = ptx::f2(-m_safe, -m_safe);
  uint64_t lx0 = ptx::f2(0.f, 0.f), lx1 = lx0;
  uint32_t pk[64];
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
    pk[c / 2] = ptx::pack2<BF16>(p0, p1);
    pk[c / 2 + 1] = ptx::pack2<BF16>(p2, p3);
  }
  ptx::tmem_st_x64(tS, pk);
  float a0, a1, b0, b1;
  ptx::f2_split(lx0, a0, a1);
  ptx::f2_split(lx1, b0, b1);
  const float sum = (a0 + a1) + (b0 + b1);
  st.l_x = st.l_x * alpha + sum;
  st.l_p = st.l_p * alpha + (sum + corr);

  if (!first && __any_sync(0xffffffffu, rescale)) {
    if (pvd_bar != 0) {
      if (!wait_bar_warp(pvd_bar, pvd_parity, ctl)) return false;
      ptx::tc_fence_after();
    }
    const uint64_t al2 = ptx::f2(alpha, alpha);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
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

// What the softmax warps need of unit k, published by the loader thread (which
// decodes every unit first anyway), so that the softmax warps spend nothing on
// decoding between units.
struct TileUnitDesc {
  int more;        // 0: the walk has ended (no unit k)
  int n0, n1;      // K/V steps of query tile 0 / 1
  int valid;       // bit t: query tile t holds rows of the sequence
  int q0;          // first query row of tile 0 (may be < 0)
  int Lq, Lk;      // rows and keys of the sequence
  int j0;          // first K/V tile
  long long o0;    // O row index (rows of [rows, H]) of sequence row 0, this head
  long long lse0;  // LSE index of sequence row 0, this head
};
static_assert(sizeof(TileUnitDesc) == 48, "descriptor");

// Loader: writes descriptor k (more = false: the end of the walk) once the
// softmax warps have read descriptor k - kDescSlots from the same slot.
template <int D>
__device__ __forceinline__ bool publish_tile_desc(const FwdParams& p, uint8_t* base,
                                                  uint32_t bars, int k, bool more, const Unit& w,
                                                  const Ctl& ctl) {
  using L = Layout<D>;
  const int slot = k % kDescSlots;
  if (k >= kDescSlots &&
      !wait_bar(bars + 8u * (L::DFR + slot), (static_cast<uint32_t>(k / kDescSlots) - 1u) & 1u,
                ctl))
    return false;
  TileUnitDesc d;
  d.more = more ? 1 : 0;
  d.n0 = more ? w.n[0] : 0;
  d.n1 = more ? w.n[1] : 0;
  d.valid = more ? (w.valid[0] ? 1 : 0) | (w.valid[1] ? 2 : 0) : 0;
  d.q0 = more ? w.q0 : 0;
  d.Lq = more ? w.Lq : 0;
  d.Lk = more ? w.Lk : 0;
  d.j0 = more ? w.j0 : 0;
  d.o0 = more ? static_cast<long long>(w.q_start) * p.H + w.h : 0;
  d.lse0 = !more ? 0
           : p.varlen ? static_cast<long long>(w.h) * p.Sq + w.q_start
                      : (static_cast<long long>(w.b) * p.H + w.h) * p.Sq;
  *reinterpret_cast<TileUnitDesc*>(base + L::kDescOff + slot * 48) = d;
  ptx::mbar_arrive(bars + 8u * (L::DRY + slot));
  return true;
}

template <int D, bool BF16>
__device__ void softmax_role(const FwdParams& p, int t, uint32_t tmem, uint32_t bars,
                             const uint8_t* base, const Ctl& ctl) {
  using L = Layout<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // TMEM lane quarter this warp may access
  const int row = quarter * 32 + lane;
  const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + lane_bits + L::kColS + t * 128;
  const uint32_t tO = tmem + lane_bits + L::kColO + t * D;
  const uint32_t bar_s = bars + 8 * (L::SF + t);
  const uint32_t bar_p = bars + 8 * (L::PF + t);
  const uint32_t bar_o = bars + 8 * (L::OF + t);
  uint32_t s_cnt = 0, o_cnt = 0;
  using out_t = uint16_t;
  out_t* const O = static_cast<out_t*>(p.o);

  for (int k = 0;; ++k) {
    const int slot = k % kDescSlots;
    if (!wait_bar_warp(bars + 8u * (L::DRY + slot), static_cast<uint32_t>(k / kDescSlots) & 1u,
                       ctl))
      return;
    const TileUnitDesc d = *reinterpret_cast<const TileUnitDesc*>(base + L::kDescOff + slot * 48);
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bars + 8u * (L::DFR + slot));
    if (!d.more) break;
    if (((d.valid >> t) & 1) == 0) continue;
    const int q0 = d.q0 + t * kBM;
    const int qrow = q0 + row;
    const bool row_ok = qrow >= 0 && qrow < d.Lq;
    const int n = t == 0 ? d.n0 : d.n1;
    const long long orow = d.o0 + static_cast<long long>(qrow) * p.H;
    const long long lidx = d.lse0 + qrow;
    RowState rs{-INFINITY, 0.0f, 0.0f};
    if (n > 0) {
      int key_lo, key_hi;
      Unit wk;  // row_keys reads the key count only
      wk.Lk = d.Lk;
      row_keys(p, wk, qrow, key_lo, key_hi);
      for (int j = 0, kb = d.j0 * kBN; j < n; ++j, kb += kBN) {
        if (!wait_bar_warp(bar_s, s_cnt & 1u, ctl)) return;
        ++s_cnt;
        ptx::tc_fence_after();
        const int lo = key_lo - kb;
        const int limit = min(kBN - 1, key_hi - kb);
        // the S(j) commit implies O += P(j-1) V(j-1) is done: no extra wait
        softmax_step_pv<D, BF16>(tS, tO, lo, limit, p.scale_log2, p.scale_pos != 0, j == 0, rs, 0u,
                                 0u, ctl);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_p);
      }
      if (!wait_bar_warp(bar_o, o_cnt & 1u, ctl)) return;
      ++o_cnt;
      ptx::tc_fence_after();
      const float inv_l = rs.l_p > 0.0f ? 1.0f / rs.l_p : 0.0f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        ptx::tmem_ld_x32(tO + c0, o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = ptx::pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l,
                                   __uint_as_float(o[2 * i + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(O + orow * D + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
    } else if (row_ok) {  // no visible key at all: O = 0, LSE = -inf
      uint4* dst = reinterpret_cast<uint4*>(O + orow * D);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (row_ok) {
      p.lse[lidx] = rs.l_x > 0.0f ? (rs.m + ptx::lg2(rs.l_x)) * 0.69314718055994531f : -INFINITY;
    }
  }
}

// -------------------------------------------------------------------- MMA
template <int D, bool BF16>
__device__ void mma_loop(const FwdParams& p, uint32_t smem, uint32_t tmem, uint32_t bars,
                         const Ctl& ctl) {
  using L = Layout<D>;
  constexpr int NS = L::kStages;
  constexpr uint32_t kIdS = ptx::idesc_f16_f32acc(BF16, kBM, kBN, false);
  constexpr uint32_t kIdPV = ptx::idesc_f16_f32acc(BF16, kBM, D, true);
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t kv_it = 0, q_it = 0, p_cnt[kTiles] = {0, 0};

  // Descriptor templates: only the 14-bit start-address field (bits 0-13,
  // address >> 4) changes between operands, so per-MMA descriptors are formed
  // by adding (offset >> 4) to a template built from the buffer's base.
  const uint64_t dq[kTiles] = {ptx::desc_sw128(smem + L::kQOff, 16, 1024),
                               ptx::desc_sw128(smem + L::kQOff + L::kTileBytes, 16, 1024)};
  const uint64_t dk0 = ptx::desc_sw128(smem + L::kKOff, 16, 1024);
  const uint64_t dv0 = ptx::desc_sw128(smem + L::kVOff, L::kBlk, 1024);

  Cursor cur;
  init_cursor<kUnitRows>(p, cur, false);
  Unit w;
  for (int k = 0; decode_unit(p, slot_unit(p, k), cur, w, false); ++k) {
    const int nmax = max(w.n[0], w.n[1]);
    if (nmax == 0) continue;
    if (!wait_bar(bar(L::QF), q_it & 1u, ctl)) return;
    ptx::tc_fence_after();
    for (int j = 0; j <= nmax; ++j) {
      // K(j) and V(j-1) are each waited for once per step, by the first user.
      bool k_ready = false, v_ready = false;
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        const uint32_t tS = tmem + L::kColS + t * 128;
        const uint32_t tO = tmem + L::kColO + t * D;
        if (j >= 1 && j - 1 < w.n[t]) {  // O_t += P_t(j-1) V(j-1)
          if (!wait_bar(bar(L::PF + t), p_cnt[t] & 1u, ctl)) return;
          ++p_cnt[t];
          const uint32_t it = kv_it + j - 1;
          const uint32_t st = it % NS;
          if (!v_ready) {
            if (!wait_bar(bar(L::VF + st), (it / NS) & 1u, ctl)) return;
            v_ready = true;
          }
          ptx::tc_fence_after();
          const uint64_t dv = dv0 + ((st * L::kTileBytes) >> 4);
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            // V is MN-major: 16 keys = 2 swizzle atoms of 8 keys x 128 B;
            // LBO = next 64-column block of D, SBO = next 8 keys.
            ptx::mma_ts(tO, tS + ks * 8, dv + ((ks * 2048) >> 4), kIdPV,
                        (j - 1 > 0 || ks > 0) ? 1u : 0u);
          }
          if (t == 1 || j - 1 >= w.n[1]) ptx::mma_commit(bar(L::VE + st));
          if (j - 1 == w.n[t] - 1) ptx::mma_commit(bar(L::OF + t));
        }
        if (j < w.n[t]) {  // S_t(j) = Q_t K(j)^T
          const uint32_t it = kv_it + j;
          const uint32_t st = it % NS;
          if (!k_ready) {
            if (!wait_bar(bar(L::KF + st), (it / NS) & 1u, ctl)) return;
            k_ready = true;
            ptx::tc_fence_after();
          }
          const uint64_t dk = dk0 + ((st * L::kTileBytes) >> 4);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            // K-major, 16 elements = 32 B step inside the 128-B swizzle row.
            const uint32_t off = ((ks >> 2) * L::kBlk + (ks & 3) * 32) >> 4;
            ptx::mma_ss(tS, dq[t] + off, dk + off, kIdS, ks > 0 ? 1u : 0u);
          }
          ptx::mma_commit(bar(L::SF + t));
          if (t == 1 || j >= w.n[1]) ptx::mma_commit(bar(L::KE + st));
        }
      }
      if (j == nmax - 1) ptx::mma_commit(bar(L::QE));
    }
    kv_it += nmax;
    ++q_it;
  }
  // make sure every issued tcgen05 operation retired before TMEM is freed
}

template <int D, bool BF16>
__device__ void mma_role(const FwdParams& p, uint32_t smem, uint32_t tmem, uint32_t bars,
                         const Ctl& ctl) {
  mma_loop<D, BF16>(p, smem, tmem, bars, ctl);
  // Every tcgen05 operation issued so far must retire before TMEM is freed,
  // also when the loop was abandoned.
  const uint32_t done = bars + 8u * Layout<D>::DONE;
  ptx::mma_commit(done);
  wait_bar(done, 0, ctl, false);
}

// ------------------------------------------------------------------- load
template <int D>
struct LoadLog {
  FillLog<1> q;
  FillLog<Layout<D>::kStages> k, v;
};

template <int D>
__device__ void load_loop(const FwdParams& p, uint32_t smem, uint8_t* base, uint32_t bars,
                          const Ctl& ctl, LoadLog<D>& f) {
  using L = Layout<D>;
  constexpr int NS = L::kStages;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t kv_it = 0, q_it = 0;
  Cursor cur;
  init_cursor<kUnitRows>(p, cur, true);
  Unit w;
  int k = 0;
  for (; decode_unit(p, slot_unit(p, k), cur, w, true); ++k) {
    if (!publish_tile_desc<D>(p, base, bars, k, true, w, ctl)) return;
    const int nmax = max(w.n[0], w.n[1]);
    if (nmax == 0) continue;
    if (q_it > 0 && !wait_bar(bar(L::QE), (q_it - 1) & 1u, ctl)) return;
    ptx::mbar_arrive_expect_tx(bar(L::QF), kTiles * L::kTileBytes);
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        ptx::tma_load_3d(smem + L::kQOff + t * L::kTileBytes + blk * L::kBlk, &p.tm_q,
                         bar(L::QF), blk * 64, w.h, w.q_start + w.q0 + t * kBM);
    f.q.last[0] = static_cast<int>(q_it);
    ++q_it;
    for (int j = 0; j < nmax; ++j) {
      const uint32_t it = kv_it + j;
      const uint32_t st = it % NS;
      const int krow = w.k_start + (w.j0 + j) * kBN;
      if (it >= NS && !wait_bar(bar(L::KE + st), (it / NS - 1) & 1u, ctl)) return;
      // injected fault (tests only): this K tile never arrives, so the MMA
      // thread's bounded wait runs out and the call reports a device timeout
      if (!(p.inject == 1 && blockIdx.x == 0 && it == 0)) {
        ptx::mbar_arrive_expect_tx(bar(L::KF + st), L::kTileBytes);
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk)
          ptx::tma_load_3d(smem + L::kKOff + st * L::kTileBytes + blk * L::kBlk, &p.tm_k,
                           bar(L::KF + st), blk * 64, w.h, krow);
        f.k.last[st] = static_cast<int>(it);
      }
      if (it >= NS && !wait_bar(bar(L::VE + st), (it / NS - 1) & 1u, ctl)) return;
      ptx::mbar_arrive_expect_tx(bar(L::VF + st), L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        ptx::tma_load_3d(smem + L::kVOff + st * L::kTileBytes + blk * L::kBlk, &p.tm_v,
                         bar(L::VF + st), blk * 64, w.h, krow);
      f.v.last[st] = static_cast<int>(it);
    }
    kv_it += nmax;
  }
  publish_tile_desc<D>(p, base, bars, k, false, w, ctl);
}

template <int D>
__device__ void load_role(const FwdParams& p, uint32_t smem, uint8_t* base, uint32_t bars,
                          const Ctl& ctl) {
  using L = Layout<D>;
  LoadLog<D> f;
  f.q.clear();
  f.k.clear();
  f.v.clear();
  load_loop<D>(p, smem, base, bars, ctl, f);
  // No TMA write may land after the CTA exits: wait for the last copy issued
  // into each buffer (normally these phases completed long ago).
  drain_fills(bars, L::QF, f.q, ctl);
  drain_fills(bars, L::KF, f.k, ctl);
  drain_fills(bars, L::VF, f.v, ctl);
}

// ------------------------------------------------------------------ kernel
template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i)
      ptx::mbar_init(bars + 8u * i, (i == L::PF || i == L::PF + 1) ? kBM
                                    : (i >= L::DFR)                  ? kTileSoftmaxWarps
                                                                     : 1u);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  build_seq_order(p);
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
    softmax_role<D, BF16>(p, warp >> 2, tmem, bars, base, ctl);
  } else if (warp == kMmaWarp) {
    if (lane == 0) mma_role<D, BF16>(p, smem, tmem, bars, ctl);
  } else if (lane == 0) {
    load_role<D>(p, smem, base, bars, ctl);
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// Opts the kernel `fn` in to `bytes` of dynamic shared memory on the current
// device, once per device: `done` holds one bit per device for that kernel
// (setting the attribute on every launch cost host time on every call).
inline cudaError_t smem_opt_in(const void* fn, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Dynamic shared memory of a launch: the layout, plus the packed-sequence
// order past its end when that is used (FwdParams::order_off = kBytes).
template <int D>
inline int fwd_smem_bytes(const FwdParams& p) {
  return Layout<D>::kAlloc + (seq_ordered(p) ? kOrderBytes : 0);
}

template <int D, bool BF16>
cudaError_t launch_fwd(const FwdParams& params, int grid, cudaStream_t stream) {
  FwdParams p = params;
  p.order_off = Layout<D>::kBytes;
  const void* fn = reinterpret_cast<const void*>(&attn_fwd_kernel<D, BF16>);
  static std::atomic<unsigned long long> opted{0};
  const cudaError_t e = smem_opt_in(fn, Layout<D>::kAlloc + kOrderBytes, opted);
  if (e != cudaSuccess) return e;
  void* args[] = {&p};
  return cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, fwd_smem_bytes<D>(p), stream);
}

}  // namespace attn
