// C ABI of the fused attention forward (declarations and contract in attn.h).
//
// Host side only: argument checks, per-device state (SM count, device error
// word), TMA tensor-map encoding and the launch of the persistent kernel on the
// caller's stream.  No synchronisation happens inside attn_fwd.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "attn.h"
#include "bwd_kernel.cuh"
#include "host_common.h"
#include "decode_kernel.cuh"
#include "fwd_fp8_kernel.cuh"
#include "launch.cuh"
#include "merge_kernel.cuh"

namespace attn {

namespace {

using host::aligned;
using host::encode_rows_heads_dim;
using host::inject_from_env;
using host::kMaxDevices;
using host::on_device;
using host::timeout_ns_from_env;

// Per-device state of the allocating entry points: the SM count and the
// device error word the kernels report into (one per device, shared by every
// stream and every call on that device; allocated on first use, freed by
// attn_release).
struct DeviceState {
  int sms = 0;
  int* err = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

thread_local int t_last_grid = -1;
thread_local int t_last_smem = -1;

// Records the shape of a launch for attn_last_launch; with ATTN_DEBUG=1 in the
// environment also prints one line per launch to stderr (the library is
// silent otherwise).
void note_launch(const char* what, int grid, int smem) {
  t_last_grid = grid;
  t_last_smem = smem;
  const char* dbg = std::getenv("ATTN_DEBUG");
  if (dbg && dbg[0] == '1') std::fprintf(stderr, "attn: %s grid=%d smem=%d\n", what, grid, smem);
}

// The per-device state on first use (an sm_103 device; the error word is
// allocated here).  Returns ATTN_OK or an error.
int device_state(int dev, DeviceState** out) {
  const host::DeviceInfo* info = nullptr;
  const int st = host::device_info(dev, &info);
  if (st != ATTN_OK) return st;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.err) {
    if (cudaMalloc(&s.err, sizeof(int)) != cudaSuccess) {
      s.err = nullptr;
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    if (cudaMemset(s.err, 0, sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
  }
  s.sms = info->sms;
  *out = &s;
  return ATTN_OK;
}

// The backward's fp32 dQ accumulator [slices, rows, D] as a 3-D map {D, rows,
// slices} with 32 x 128 x 1 boxes (128 B inner extent) and 128-byte swizzle:
// the target of the per-step TMA reduce-adds.  Dense: slices = B*H, rows =
// Sq; packed: slices = H, rows = all query rows.
int encode_dq_acc(CUtensorMap* m, float* ptr, int slices, int rows, int D) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(slices)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4,
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(D) * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = host::encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace attn

using namespace attn;

namespace attn {
namespace {

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int Sq, int Sk, int D, float scale, int causal, int window_left, int window_right,
             int global_q, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int dtype,
             void* stream) {
  FwdParams p;
  host::FwdCall call;
  int st = host::check_fwd_args(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, window_left,
                                window_right, global_q, cu_seqlens_q, cu_seqlens_k, dtype, &p,
                                &call);
  if (st != ATTN_OK || call.nothing) return st;
  int dev = 0;
  if ((st = host::current_device(&dev)) != ATTN_OK) return st;
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds)) != ATTN_OK) return st;
  if ((st = host::prepare_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale, cu_seqlens_q,
                              cu_seqlens_k, dev, call, &p)) != ATTN_OK)
    return st;
  p.err = ds->err;
  p.inject = inject_from_env() == 1 ? 1 : 0;
  LaunchInfo info;
  const cudaError_t e = launch_forward(p, D, call.bf16, call.varlen, B, H, call.rows_q, Sq,
                                       ds->sms, static_cast<cudaStream_t>(stream), &info);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  note_launch(window_left != -1 || window_right != -1 || global_q != 0 ? "attn_fwd_window"
                                                                       : "attn_fwd",
              info.grid, info.smem);
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int Sq, int Sk, int D, float scale, int causal,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int dtype,
                        void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, -1, -1, 0, cu_seqlens_q,
                  cu_seqlens_k, dtype, stream);
}

extern "C" int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int H, int Sq, int Sk, int D, float scale, int causal,
                               int window_left, int window_right, int global_q,
                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                               int dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, window_left, window_right,
                  global_q, cu_seqlens_q, cu_seqlens_k, dtype, stream);
}

// ------------------------------------------------------------------ decode
namespace attn {
namespace dec {
#define ATTN_DEC_EXTERN(D)                                                                   \
  extern template cudaError_t launch_decode<D, 1, false>(const DecParams&, int, cudaStream_t); \
  extern template cudaError_t launch_decode<D, 4, false>(const DecParams&, int, cudaStream_t); \
  extern template cudaError_t launch_decode<D, 16, false>(const DecParams&, int, cudaStream_t); \
  extern template cudaError_t launch_decode<D, 1, true>(const DecParams&, int, cudaStream_t);  \
  extern template cudaError_t launch_decode<D, 4, true>(const DecParams&, int, cudaStream_t);  \
  extern template cudaError_t launch_decode<D, 16, true>(const DecParams&, int, cudaStream_t);
ATTN_DEC_EXTERN(64)
ATTN_DEC_EXTERN(128)
#undef ATTN_DEC_EXTERN
extern template cudaError_t launch_merge<float, false>(const float*, const float*, int, int, int,
                                                       int, int, void*, float*, cudaStream_t);
extern template cudaError_t launch_merge<float, true>(const float*, const float*, int, int, int,
                                                      int, int, void*, float*, cudaStream_t);
extern template cudaError_t launch_merge<uint16_t, false>(const uint16_t*, const float*, int, int,
                                                          int, int, int, void*, float*,
                                                          cudaStream_t);
extern template cudaError_t launch_merge<uint16_t, true>(const uint16_t*, const float*, int, int,
                                                         int, int, int, void*, float*,
                                                         cudaStream_t);
}  // namespace dec

namespace {

// Split of the cache keys into chunks of whole 64-key tiles.  Every CTA of the
// persistent grid takes units round-robin, so the step lasts about
// ceil(units / sms) chunks; the split count (from about 8 units per SM up to 4x
// that) is the one whose busiest SM streams the fewest tiles relative to the
// average, with chunks of at least 256 keys (4 tiles) where the cache allows.
void decode_plan(int B, int H, int Sk, int sms, int* splits, int* chunk) {
  const long long tiles = (static_cast<long long>(Sk) + dec::kKeys - 1) / dec::kKeys;
  const long long bh = static_cast<long long>(B) * H;
  long long want = (8LL * sms + bh - 1) / bh;
  if (want > tiles) want = tiles;
  if (want < 1) want = 1;
  const long long min_ct = tiles < 4 ? tiles : 4;
  long long best_ct = 0;
  double best_eff = -1.0;
  for (long long s = want; s <= 4 * want && s <= tiles; ++s) {
    long long ct = (tiles + s - 1) / s;
    if (ct < min_ct) ct = min_ct;
    const long long real = (tiles + ct - 1) / ct;
    const long long units = bh * real;
    const long long waves = (units + sms - 1) / sms;
    const double eff = static_cast<double>(bh * tiles) / (static_cast<double>(sms) * waves * ct);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best_ct = ct;
    }
  }
  if (best_ct < 1) best_ct = tiles < 1 ? 1 : tiles;
  *chunk = static_cast<int>(best_ct * dec::kKeys);
  *splits = static_cast<int>((tiles + best_ct - 1) / best_ct);
}

long long decode_ws_bytes(int B, int H, int Sq, int D, int splits) {
  if (splits <= 1) return 0;
  const long long o = static_cast<long long>(splits) * B * Sq * H * D * 4;
  const long long l = static_cast<long long>(splits) * B * H * Sq * 4;
  return ((o + 255) / 256) * 256 + l;
}

int current_device_state(DeviceState** ds) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  return device_state(dev, ds);
}

}  // namespace
}  // namespace attn

extern "C" int attn_decode_workspace(int B, int H, int Sq, int Sk, int D, size_t* bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  if (B < 0 || H < 1 || Sq < 1 || Sk < 1) return ATTN_ERR_INVALID_ARG;
  if ((D != 64 && D != 128) || Sq > dec::kMaxSq) return ATTN_ERR_UNSUPPORTED;
  if (B == 0) return ATTN_OK;
  DeviceState* ds = nullptr;
  const int st = current_device_state(&ds);
  if (st != ATTN_OK) return st;
  int splits = 1, chunk = 0;
  decode_plan(B, H, Sk, ds->sms, &splits, &chunk);
  *bytes = static_cast<size_t>(decode_ws_bytes(B, H, Sq, D, splits));
  return ATTN_OK;
}

extern "C" int attn_fwd_decode(const void* q, const void* k_cache, const void* v_cache, void* o,
                               float* lse, int B, int H, int Sq, int Sk, int D, float scale,
                               int causal, const int32_t* seqlens_k, void* workspace,
                               size_t workspace_bytes, int dtype, void* stream) {
  // ---- argument checks (no CUDA call before these pass)
  if (B < 0 || H < 1 || Sq < 1 || Sk < 1) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (Sq > dec::kMaxSq) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_DTYPE_FP16 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (B == 0) return ATTN_OK;
  if (!q || !k_cache || !v_cache || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || (seqlens_k && !aligned(seqlens_k, 4)) ||
      (workspace && !aligned(workspace, 256)))
    return ATTN_ERR_MISALIGNED;
  const long long rows_k = static_cast<long long>(B) * Sk;
  if (rows_k > INT_MAX - 2 * dec::kKeys) return ATTN_ERR_INVALID_ARG;

  // ---- device checks
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  if (st != ATTN_OK) return st;
  int splits = 1, chunk = 0;
  decode_plan(B, H, Sk, ds->sms, &splits, &chunk);
  const long long units = static_cast<long long>(B) * H * splits;
  if (units > INT_MAX / 2) return ATTN_ERR_INVALID_ARG;
  const long long need = decode_ws_bytes(B, H, Sq, D, splits);
  if (need > 0 && (!workspace || static_cast<long long>(workspace_bytes) < need))
    return ATTN_ERR_INVALID_ARG;
  if (!on_device(q, dev) || !on_device(k_cache, dev) || !on_device(v_cache, dev) ||
      !on_device(o, dev) || !on_device(lse, dev) || (seqlens_k && !on_device(seqlens_k, dev)) ||
      (need > 0 && !on_device(workspace, dev)))
    return ATTN_ERR_INVALID_ARG;

  // ---- parameters
  dec::DecParams p;
  const bool bf16 = dtype == ATTN_DTYPE_BF16;
  if (encode_rows_heads_dim(&p.tm_k, k_cache, rows_k, H, D, bf16, dec::kKeys) != ATTN_OK ||
      encode_rows_heads_dim(&p.tm_v, v_cache, rows_k, H, D, bf16, dec::kKeys) != ATTN_OK)
    return ATTN_ERR_CUDA;
  p.q = static_cast<const uint16_t*>(q);
  p.o = o;
  p.lse = lse;
  p.seqlens = seqlens_k;
  float* ws = static_cast<float*>(workspace);
  p.ws_o = need > 0 ? ws : nullptr;
  p.ws_lse = need > 0 ? ws + ((static_cast<long long>(splits) * B * Sq * H * D * 4 + 255) / 256) *
                                 64
                      : nullptr;
  p.err = ds->err;
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.splits = splits;
  p.chunk = chunk;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.timeout_ns = timeout_ns_from_env();
  p.inject = inject_from_env();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // injected launch failure (tests only): an empty grid, which the launch rejects
  const int grid = p.inject == 2 ? 0 : static_cast<int>(units < ds->sms ? units : ds->sms);
  cudaError_t e;
#define ATTN_DEC_LAUNCH(DD, BB)                                                   \
  (Sq == 1 ? dec::launch_decode<DD, 1, BB>(p, grid, s)                          \
           : Sq <= 4 ? dec::launch_decode<DD, 4, BB>(p, grid, s)                \
                     : dec::launch_decode<DD, 16, BB>(p, grid, s))
  if (D == 64)
    e = bf16 ? ATTN_DEC_LAUNCH(64, true) : ATTN_DEC_LAUNCH(64, false);
  else
    e = bf16 ? ATTN_DEC_LAUNCH(128, true) : ATTN_DEC_LAUNCH(128, false);
#undef ATTN_DEC_LAUNCH
  if (e == cudaSuccess && splits > 1)
    e = bf16 ? dec::launch_merge<float, true>(p.ws_o, p.ws_lse, splits, B, Sq, H, D, o, lse, s)
             : dec::launch_merge<float, false>(p.ws_o, p.ws_lse, splits, B, Sq, H, D, o, lse, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  note_launch("attn_fwd_decode", grid,
              D == 64 ? dec::DLayout<64>::kAlloc : dec::DLayout<128>::kAlloc);
  return ATTN_OK;
}

extern "C" int attn_merge(const void* o_parts, const float* lse_parts, int n_parts, int B, int S,
                          int H, int D, void* o, float* lse, int dtype, void* stream) {
  if (n_parts < 1 || B < 0 || S < 0 || H < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (D > dec::kMergeMaxD) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_DTYPE_FP16 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || S == 0) return ATTN_OK;
  if (!o_parts || !lse_parts || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned(o_parts, 2) || !aligned(o, 2) || !aligned(lse_parts, 4) || !aligned(lse, 4))
    return ATTN_ERR_MISALIGNED;
  const long long rows = static_cast<long long>(B) * S * H;
  if (rows * D > (1LL << 40) || rows > INT_MAX) return ATTN_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  if (st != ATTN_OK) return st;
  if (!on_device(o_parts, dev) || !on_device(lse_parts, dev) || !on_device(o, dev) ||
      !on_device(lse, dev))
    return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* parts = static_cast<const uint16_t*>(o_parts);
  const cudaError_t e =
      dtype == ATTN_DTYPE_BF16
          ? dec::launch_merge<uint16_t, true>(parts, lse_parts, n_parts, B, S, H, D, o, lse, s)
          : dec::launch_merge<uint16_t, false>(parts, lse_parts, n_parts, B, S, H, D, o, lse, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

// ---------------------------------------------------------------- backward
namespace attn {
namespace bwd {
extern template cudaError_t launch_bwd<64, false>(const BwdParams&, const uint16_t*, const uint16_t*, const float*, uint8_t*, int32_t*, long long, uint16_t*, int, cudaStream_t);
extern template cudaError_t launch_bwd<64, true>(const BwdParams&, const uint16_t*, const uint16_t*, const float*, uint8_t*, int32_t*, long long, uint16_t*, int, cudaStream_t);
extern template cudaError_t launch_bwd<128, false>(const BwdParams&, const uint16_t*, const uint16_t*, const float*, uint8_t*, int32_t*, long long, uint16_t*, int, cudaStream_t);
extern template cudaError_t launch_bwd<128, true>(const BwdParams&, const uint16_t*, const uint16_t*, const float*, uint8_t*, int32_t*, long long, uint16_t*, int, cudaStream_t);
}  // namespace bwd
namespace {
// The backward's workspace: an fp32 dQ accumulator, then the bias tiles of the
// two products (-LSE/scale and -D, 2 x 4 KiB per 128-query tile and head),
// then (packed sequences) the per-sequence tile offsets.  Dense: B*H*ceil(Sq/128)
// tiles; packed (Sq = all query rows): at most floor((Sq + 127 B) / 128) per head.
struct BwdWs {
  long long acc, bias, tiles_bound, tiles, total;
};
BwdWs bwd_ws(int B, int H, int Sq, int D, bool varlen) {
  BwdWs w;
  const long long rows = varlen ? Sq : static_cast<long long>(B) * Sq;
  w.acc = ((rows * H * D * 4 + 255) / 256) * 256;
  w.tiles_bound = varlen ? (static_cast<long long>(Sq) + 127LL * B) / bwd::kBN
                         : static_cast<long long>(B) * ((Sq + bwd::kBN - 1) / bwd::kBN);
  w.bias = w.tiles_bound * H * 2 * bwd::kBiasBytes;
  w.tiles = varlen ? ((static_cast<long long>(B) + 2) * 4 + 255) / 256 * 256 : 0;
  w.total = w.acc + w.bias + w.tiles;
  return w;
}
}  // namespace
}  // namespace attn

extern "C" int attn_bwd_workspace(int B, int H, int Sq, int D, int varlen, size_t* bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  if (B < 0 || H < 1 || Sq < 0) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  *bytes = static_cast<size_t>(bwd_ws(B, H, Sq, D, varlen != 0).total);
  return ATTN_OK;
}

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                        int H, int Sq, int Sk, int D, float scale, int causal,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                        void* workspace, size_t workspace_bytes, int dtype, void* stream) {
  // ---- argument checks (no CUDA call before these pass)
  if (B < 0 || H < 1 || Sq < 0 || Sk < 1) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_DTYPE_FP16 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (scale == 0.0f) return ATTN_ERR_UNSUPPORTED;  // the LSE term is carried as -LSE/scale
  const bool varlen = cu_seqlens_q != nullptr || cu_seqlens_k != nullptr;
  if (varlen && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (B == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256))
    return ATTN_ERR_MISALIGNED;
  if (varlen && (!aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))) return ATTN_ERR_MISALIGNED;
  const long long rows_q = varlen ? Sq : static_cast<long long>(B) * Sq;
  const long long rows_k = varlen ? Sk : static_cast<long long>(B) * Sk;
  if (rows_q > INT_MAX - 2 * bwd::kBN || rows_k > INT_MAX - 2 * bwd::kBM)
    return ATTN_ERR_INVALID_ARG;
  // unit indices are int: B*H*ceil(Sk/128) (dense) or H*(ceil(Sk/128)+B) (packed)
  const long long units = varlen
      ? static_cast<long long>(H) * ((rows_k + bwd::kBM - 1) / bwd::kBM + B)
      : static_cast<long long>(B) * H * ((Sk + bwd::kBM - 1) / bwd::kBM);
  if (units > INT_MAX / 2) return ATTN_ERR_INVALID_ARG;
  const BwdWs wsl = bwd_ws(B, H, Sq, D, varlen);
  if (wsl.tiles_bound * H * bwd::kBN / 8 > INT_MAX) return ATTN_ERR_INVALID_ARG;  // pre-pass grid
  if (rows_q > 0 && static_cast<long long>(workspace_bytes) < wsl.total)
    return ATTN_ERR_INVALID_ARG;

  // ---- device checks
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  if (st != ATTN_OK) return st;
  const void* ptrs[] = {q, k, v, o, dout, lse, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (!on_device(ptr, dev)) return ATTN_ERR_INVALID_ARG;
  if (varlen && (!on_device(cu_seqlens_q, dev) || !on_device(cu_seqlens_k, dev)))
    return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rows_q == 0) {  // no query sees any key: dK = dV = 0
    const size_t bytes = static_cast<size_t>(rows_k) * H * D * 2;
    if (cudaMemsetAsync(dk, 0, bytes, s) != cudaSuccess ||
        cudaMemsetAsync(dv, 0, bytes, s) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
  }

  // ---- parameters
  bwd::BwdParams p;
  const bool bf16 = dtype == ATTN_DTYPE_BF16;
  if (encode_rows_heads_dim(&p.tm_q, q, rows_q, H, D, bf16) != ATTN_OK ||
      encode_rows_heads_dim(&p.tm_do, dout, rows_q, H, D, bf16) != ATTN_OK ||
      encode_rows_heads_dim(&p.tm_k, k, rows_k, H, D, bf16) != ATTN_OK ||
      encode_rows_heads_dim(&p.tm_v, v, rows_k, H, D, bf16) != ATTN_OK)
    return ATTN_ERR_CUDA;
  p.dq_acc = static_cast<float*>(workspace);
  if (encode_dq_acc(&p.tm_dq, p.dq_acc, varlen ? H : B * H, Sq, D) != ATTN_OK)
    return ATTN_ERR_CUDA;
  uint8_t* bias = static_cast<uint8_t*>(workspace) + wsl.acc;
  int32_t* tiles = varlen ? reinterpret_cast<int32_t*>(bias + wsl.bias) : nullptr;
  p.bias = bias;
  p.tiles = tiles;
  p.dk = dk;
  p.dv = dv;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.err = ds->err;
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.Tq = static_cast<int>(rows_q);
  p.varlen = varlen ? 1 : 0;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.timeout_ns = timeout_ns_from_env();
  const int grid = static_cast<int>(units < ds->sms ? (units > 0 ? units : 1) : ds->sms);
  const uint16_t* o16 = static_cast<const uint16_t*>(o);
  const uint16_t* do16 = static_cast<const uint16_t*>(dout);
  uint16_t* dq16 = static_cast<uint16_t*>(dq);
  cudaError_t e;
  if (D == 64)
    e = bf16 ? bwd::launch_bwd<64, true>(p, o16, do16, lse, bias, tiles, wsl.tiles_bound, dq16,
                                         grid, s)
             : bwd::launch_bwd<64, false>(p, o16, do16, lse, bias, tiles, wsl.tiles_bound, dq16,
                                          grid, s);
  else
    e = bf16 ? bwd::launch_bwd<128, true>(p, o16, do16, lse, bias, tiles, wsl.tiles_bound,
                                          dq16, grid, s)
             : bwd::launch_bwd<128, false>(p, o16, do16, lse, bias, tiles, wsl.tiles_bound,
                                           dq16, grid, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  note_launch("attn_bwd", grid, D == 64 ? bwd::BLayout<64>::kAlloc : bwd::BLayout<128>::kAlloc);
  return ATTN_OK;
}

// -------------------------------------------------------------- fp8 (e4m3)
namespace attn {
namespace fp8 {
extern template cudaError_t launch_fwd_fp8<true>(const Fp8Params&, const uint8_t*, uint8_t*, int,
                                                 cudaStream_t);
extern template cudaError_t launch_fwd_fp8<false>(const Fp8Params&, const uint8_t*, uint8_t*,
                                                  int, cudaStream_t);
}  // namespace fp8
namespace {
int fp8_sk_pad(int Sk) { return (Sk + 15) / 16 * 16; }
// [rows, H, 128] e4m3 tensor, box 128 elements (128 B) x 1 head x 128 rows.
int encode_e4m3_rows(CUtensorMap* m, const void* ptr, long long rows, int H) {
  cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(H) * 128};
  cuuint32_t box[3] = {128, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = host::encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}
// V^T [H, 128, keys] e4m3 (keys innermost), box 128 keys x 128 dims x 1 head.
int encode_e4m3_vt(CUtensorMap* m, const void* ptr, long long keys, int H) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(keys), 128, static_cast<cuuint64_t>(H)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(keys), static_cast<cuuint64_t>(keys) * 128};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = host::encoder_slot()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}
}  // namespace
}  // namespace attn

extern "C" int attn_fwd_fp8_workspace(int B, int H, int Sk, int D, size_t* bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  if (B < 0 || H < 1 || Sk < 1) return ATTN_ERR_INVALID_ARG;
  if (D != 128) return ATTN_ERR_UNSUPPORTED;
  *bytes = static_cast<size_t>(H) * 128 * static_cast<size_t>(B) * fp8_sk_pad(Sk);
  return ATTN_OK;
}

extern "C" int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int Sq, int Sk, int D, float scale, float q_scale,
                            float k_scale, float v_scale, int causal, void* workspace,
                            size_t workspace_bytes, int out_dtype, void* stream) {
  // ---- argument checks (no CUDA call before these pass)
  if (B < 0 || H < 1 || Sq < 0 || Sk < 1) return ATTN_ERR_INVALID_ARG;
  if (D != 128) return ATTN_ERR_UNSUPPORTED;
  if (out_dtype != ATTN_DTYPE_FP16 && out_dtype != ATTN_DTYPE_BF16) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !std::isfinite(q_scale) || !std::isfinite(k_scale) ||
      !std::isfinite(v_scale))
    return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256))
    return ATTN_ERR_MISALIGNED;
  const long long rows_q = static_cast<long long>(B) * Sq;
  const long long sk_pad = fp8_sk_pad(Sk);
  const long long keys_t = static_cast<long long>(B) * sk_pad;
  if (rows_q > INT_MAX - 2 * kUnitRows || keys_t > INT_MAX - 2 * kBN) return ATTN_ERR_INVALID_ARG;
  const long long units = static_cast<long long>(B) * H * ((Sq + kUnitRows - 1) / kUnitRows);
  if (units > INT_MAX / 2) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(workspace_bytes) < static_cast<long long>(H) * 128 * keys_t)
    return ATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  if (st != ATTN_OK) return st;
  const void* ptrs[] = {q, k, v, o, lse, workspace};
  for (const void* ptr : ptrs)
    if (!on_device(ptr, dev)) return ATTN_ERR_INVALID_ARG;

  fp8::Fp8Params q8;
  FwdParams& p = q8.f;
  if (encode_e4m3_rows(&p.tm_q, q, rows_q, H) != ATTN_OK ||
      encode_e4m3_rows(&p.tm_k, k, static_cast<long long>(B) * Sk, H) != ATTN_OK ||
      encode_e4m3_vt(&p.tm_v, workspace, keys_t, H) != ATTN_OK)
    return ATTN_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.cu_q = nullptr;
  p.cu_k = nullptr;
  p.err = ds->err;
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.varlen = 0;
  set_mask(p, causal, -1, -1, 0);
  const double c = static_cast<double>(scale) * q_scale * k_scale;
  p.scale_log2 = static_cast<float>(c * 1.4426950408889634);
  p.scale_pos = c > 0.0 ? 1 : 0;
  p.timeout_ns = timeout_ns_from_env();
  q8.sk_pad = static_cast<int>(sk_pad);
  q8.o_mul = v_scale;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = static_cast<int>(units < ds->sms ? units : ds->sms);
  p.pair_blocks = pair_blocks_for(units, grid);
  const uint8_t* v8 = static_cast<const uint8_t*>(v);
  uint8_t* vt = static_cast<uint8_t*>(workspace);
  const cudaError_t e = out_dtype == ATTN_DTYPE_BF16
                            ? fp8::launch_fwd_fp8<true>(q8, v8, vt, grid, s)
                            : fp8::launch_fwd_fp8<false>(q8, v8, vt, grid, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  note_launch("attn_fwd_fp8", grid, fp8::Layout8::kAlloc);
  return ATTN_OK;
}

extern "C" int attn_check(void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  int word = 0;
  if (cudaMemcpy(&word, ds->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(ds->err, 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (word & kErrTimeout) return ATTN_ERR_DEVICE_TIMEOUT;
  if (word & kErrBadSeqlens) return ATTN_ERR_BAD_SEQLENS;
  return ATTN_OK;
}

extern "C" const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
    case ATTN_ERR_BAD_SEQLENS: return "ATTN_ERR_BAD_SEQLENS";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

extern "C" int attn_num_sms(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  return st == ATTN_OK ? ds->sms : st;
}

extern "C" int attn_last_launch(int* grid_ctas, int* smem_bytes) {
  if (t_last_grid < 0) return ATTN_ERR_INVALID_ARG;
  if (grid_ctas) *grid_ctas = t_last_grid;
  if (smem_bytes) *smem_bytes = t_last_smem;
  return ATTN_OK;
}

extern "C" int attn_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int rc = ATTN_OK;
  int cur = 0;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (int d = 0; d < kMaxDevices; ++d) {
    DeviceState& s = g_dev[d];
    if (s.err) {
      if (cudaSetDevice(d) != cudaSuccess || cudaFree(s.err) != cudaSuccess) rc = ATTN_ERR_CUDA;
    }
    s = DeviceState();
  }
  host::clear_pointer_cache();
  if (have_cur) cudaSetDevice(cur);
  cudaGetLastError();
  return rc;
}
