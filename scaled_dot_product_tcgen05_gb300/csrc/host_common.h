// Host-side helpers shared by the C entry points (api.cu, noalloc.cu): device
// capability, pointer and alignment checks, TMA tensor-map encoding, the
// argument rules of the forward, and the environment settings.  Internal to
// the library; the contract of every entry point is in include/attn.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "attn.h"
#include "launch.cuh"

namespace attn {
namespace host {

constexpr int kMaxDevices = 64;

// What the library needs to know about a device: whether it is an sm_103 part
// and its SM count (the persistent grids' size).  Queried once per device.
struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sms = 0;
};

inline std::mutex& info_mutex() {
  static std::mutex mu;
  return mu;
}

inline DeviceInfo* device_table() {
  static DeviceInfo table[kMaxDevices];
  return table;
}

inline PFN_cuTensorMapEncodeTiled_v12000& encoder_slot() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  return fn;
}

// Capability and SM count of `dev` (queried on first use); the tensor-map
// encoder is resolved at the same time.  ATTN_OK, ATTN_ERR_UNSUPPORTED (not an
// sm_103 device) or ATTN_ERR_CUDA.
inline int device_info(int dev, const DeviceInfo** out) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(info_mutex());
  DeviceInfo& s = device_table()[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    if (major == 10 && minor == 3 && !encoder_slot()) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
      }
      encoder_slot() = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    s.supported = (major == 10 && minor == 3);
    s.sms = sms;
    s.ready = true;
  }
  if (!s.supported) return ATTN_ERR_UNSUPPORTED;
  *out = &s;
  return ATTN_OK;
}

inline int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Device pointers this thread has already checked, per device (a small ring):
// a caller that passes the same buffers call after call pays for one
// cudaPointerGetAttributes per buffer, not one per call.  Only positive
// results are kept, and clear_pointer_cache() (attn_release) empties it.
struct PtrCache {
  static constexpr int kSlots = 16;
  const void* ptr[kSlots] = {};
  int dev[kSlots] = {};
  int next = 0;
  unsigned epoch = 0;
};

inline std::atomic<unsigned>& pointer_epoch() {
  static std::atomic<unsigned> e{1};
  return e;
}

inline void clear_pointer_cache() { pointer_epoch().fetch_add(1); }

// The pointer must be device (or managed) memory reachable from `dev`.
inline bool on_device(const void* p, int dev) {
  thread_local PtrCache cache;
  const unsigned epoch = pointer_epoch().load(std::memory_order_relaxed);
  if (cache.epoch != epoch) {
    cache = PtrCache();
    cache.epoch = epoch;
  }
  for (int i = 0; i < PtrCache::kSlots; ++i)
    if (cache.ptr[i] == p && cache.dev[i] == dev && p != nullptr) return true;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const bool ok = a.type == cudaMemoryTypeManaged || (a.type == cudaMemoryTypeDevice &&
                                                      a.device == dev);
  if (ok) {
    cache.ptr[cache.next] = p;
    cache.dev[cache.next] = dev;
    cache.next = (cache.next + 1) % PtrCache::kSlots;
  }
  return ok;
}

// [rows, H, D] 16-bit tensor, box = box_rows rows x 1 head x box_cols elements
// (128 B by default, with 128-byte swizzle; 32 elements = 64 B with 64-byte
// swizzle), zero fill outside the tensor.
inline int encode_rows_heads_dim(CUtensorMap* m, const void* ptr, long long rows, int H, int D,
                                 bool bf16, int box_rows = kBM, int box_cols = 64) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encoder_slot()(
      m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
      const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// The limit of any single device-side wait: ATTN_WAIT_TIMEOUT_MS milliseconds
// (read at every call), 5000 when unset or not positive.
inline long long timeout_ns_from_env() {
  const char* s = std::getenv("ATTN_WAIT_TIMEOUT_MS");
  long long ms = s ? std::atoll(s) : 0;
  if (ms <= 0) ms = 5000;
  return ms * 1000000LL;
}

// Fault injection for the failure-detection tests (ATTN_INJECT_FAULT, unset in
// normal use): 1 makes block 0 of the forward kernels (attn_fwd,
// attn_fwd_window) skip its first K tile and block 0 of the decode kernel its
// first fill, so a bounded wait runs out; 2 makes attn_fwd_decode launch an
// empty grid, which the launch rejects.
inline int inject_from_env() {
  const char* s = std::getenv("ATTN_INJECT_FAULT");
  return s ? std::atoi(s) : 0;
}

// A forward call after its argument checks.
struct FwdCall {
  bool varlen = false;
  bool bf16 = false;
  bool nothing = false;  // B == 0 or Sq == 0: a valid call with nothing to compute
  long long rows_q = 0, rows_k = 0;
};

// The argument rules of attn_fwd / attn_fwd_window / attn_fwd_noalloc, checked
// before any CUDA call (the window fields of p are filled by set_mask).
inline int check_fwd_args(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, int B, int H, int Sq, int Sk, int D, float scale,
                          int causal, int window_left, int window_right, int global_q,
                          const int32_t* cu_q, const int32_t* cu_k, int dtype, FwdParams* p,
                          FwdCall* call) {
  if (B < 0 || H < 1 || Sq < 0 || Sk < 1) return ATTN_ERR_INVALID_ARG;
  if (!set_mask(*p, causal, window_left, window_right, global_q)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_DTYPE_FP16 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  call->varlen = cu_q != nullptr || cu_k != nullptr;
  call->bf16 = dtype == ATTN_DTYPE_BF16;
  if (call->varlen && (cu_q == nullptr || cu_k == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0) {
    call->nothing = true;
    return ATTN_OK;
  }
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return ATTN_ERR_MISALIGNED;
  if (call->varlen && (!aligned(cu_q, 4) || !aligned(cu_k, 4))) return ATTN_ERR_MISALIGNED;
  call->rows_q = call->varlen ? Sq : static_cast<long long>(B) * Sq;
  call->rows_k = call->varlen ? Sk : static_cast<long long>(B) * Sk;
  if (call->rows_q > INT_MAX - 2 * kUnitRows || call->rows_k > INT_MAX - 2 * kBN)
    return ATTN_ERR_INVALID_ARG;
  // unit indices are int: B*H*ceil(Sq/256) (dense) or H*(ceil(Sq/256)+B) (varlen)
  const long long units = call->varlen
      ? static_cast<long long>(H) * ((call->rows_q + kUnitRows - 1) / kUnitRows + B)
      : static_cast<long long>(B) * H * ((Sq + kUnitRows - 1) / kUnitRows);
  if (units > INT_MAX / 2) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Device-side checks of a forward call (pointers reachable from `dev`) and the
// kernel parameters: tensor maps, sizes, scale, wait limit.  The caller sets
// p->err (where the kernel reports device-side errors) and p->inject.
inline int prepare_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int Sq, int Sk, int D, float scale, const int32_t* cu_q,
                       const int32_t* cu_k, int dev, const FwdCall& call, FwdParams* p) {
  if (!on_device(q, dev) || !on_device(k, dev) || !on_device(v, dev) || !on_device(o, dev) ||
      !on_device(lse, dev))
    return ATTN_ERR_INVALID_ARG;
  if (call.varlen && (!on_device(cu_q, dev) || !on_device(cu_k, dev)))
    return ATTN_ERR_INVALID_ARG;
  if (encode_rows_heads_dim(&p->tm_q, q, call.rows_q, H, D, call.bf16) != ATTN_OK ||
      encode_rows_heads_dim(&p->tm_k, k, call.rows_k, H, D, call.bf16) != ATTN_OK ||
      encode_rows_heads_dim(&p->tm_v, v, call.rows_k, H, D, call.bf16) != ATTN_OK ||
      encode_rows_heads_dim(&p->tm_kh, k, call.rows_k, H, D, call.bf16, kBN / 2) != ATTN_OK ||
      encode_rows_heads_dim(&p->tm_vh, v, call.rows_k, H, D, call.bf16, kBN, D / 2) != ATTN_OK)
    return ATTN_ERR_CUDA;
  p->o = o;
  p->lse = lse;
  p->cu_q = cu_q;
  p->cu_k = cu_k;
  p->B = B;
  p->H = H;
  p->Sq = Sq;
  p->Sk = Sk;
  p->varlen = call.varlen ? 1 : 0;
  p->scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p->scale_pos = scale > 0.0f ? 1 : 0;
  p->timeout_ns = timeout_ns_from_env();
  return ATTN_OK;
}

}  // namespace host
}  // namespace attn
