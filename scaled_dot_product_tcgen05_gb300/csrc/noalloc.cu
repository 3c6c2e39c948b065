// attn_fwd_noalloc: the fused attention forward for callers that must not
// allocate device memory.
//
// attn_fwd keeps its one piece of scratch memory -- the device error word the
// kernel reports timeouts and bad cu_seqlens into -- in a buffer that the
// library cudaMalloc's on the first call on each device.  Some callers cannot
// allow that: a framework whose caching allocator has reserved (almost) all of
// the GPU's memory and accounts for every byte, a latency-critical loop where
// cudaMalloc's implicit device-wide synchronisation is not acceptable, or a
// host that simply forbids raw cudaMalloc outside its own allocator.  This
// entry point runs the same kernel with its scratch in a fixed, statically
// sized __device__ array instead, so it calls no cudaMalloc, cudaFree or any
// other allocating routine.
//
// Limits and sharing rules:
//   * the array holds kNoAllocScratchBytes (256) bytes, which every GPU that
//     loads this library keeps until the process exits; the kernel needs one
//     4-byte error word for any problem size, and the call checks that need
//     against the array's size before launching;
//   * every call on a device uses the same array and the array keeps the last
//     call's contents, so the call clears the error word (an asynchronous
//     memset on the caller's stream) before each launch; calls whose kernels
//     overlap on the GPU (for example on two streams) race on that word and
//     may report each other's errors;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture is started on the device.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"
#include "launch.cuh"

namespace attn {

namespace {

constexpr int kNoAllocScratchBytes = 256;
constexpr int kNoAllocMaxDevices = 64;

// Scratch of attn_fwd_noalloc: word 0 is the kernel's error word.
static __device__ __align__(256) int g_noalloc_scratch[kNoAllocScratchBytes / sizeof(int)];

struct NoAllocDevice {
  bool ready = false;
  bool supported = false;
  int sms = 0;
  int* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_na_mu;
NoAllocDevice g_na_dev[kNoAllocMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_na_encode = nullptr;

// Once per device, with that device current: capability, SM count, and the
// device address of the static scratch array.  Allocates nothing.
int noalloc_setup(int dev, NoAllocDevice** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_na_mu);
  NoAllocDevice& s = g_na_dev[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    s.supported = (major == 10 && minor == 3);
    s.sms = sms;
    if (s.supported) {
      if (!g_na_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
          cudaGetLastError();
          return ATTN_ERR_CUDA;
        }
        g_na_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
      }
      s.scratch = static_cast<int*>(ptr);
    }
    s.ready = true;
  }
  if (!s.supported) return ATTN_ERR_UNSUPPORTED;
  *out = &s;
  return ATTN_OK;
}

bool na_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool na_on_device(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

int na_encode(CUtensorMap* m, const void* ptr, long long rows, int H, int D, bool bf16,
              int box_rows = kBM) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_na_encode(
      m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
      const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int Sq, int Sk, int D, float scale, int causal,
                                const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                int dtype, void* stream, int* device_status) {
  if (device_status) *device_status = ATTN_OK;
  // ---- the same argument rules as attn_fwd, checked before any CUDA call
  if (B < 0 || H < 1 || Sq < 0 || Sk < 1) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_DTYPE_FP16 && dtype != ATTN_DTYPE_BF16) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens_q != nullptr || cu_seqlens_k != nullptr;
  if (varlen && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!na_aligned(q, 16) || !na_aligned(k, 16) || !na_aligned(v, 16) || !na_aligned(o, 16) ||
      !na_aligned(lse, 4))
    return ATTN_ERR_MISALIGNED;
  if (varlen && (!na_aligned(cu_seqlens_q, 4) || !na_aligned(cu_seqlens_k, 4)))
    return ATTN_ERR_MISALIGNED;
  const long long rows_q = varlen ? Sq : static_cast<long long>(B) * Sq;
  const long long rows_k = varlen ? Sk : static_cast<long long>(B) * Sk;
  if (rows_q > INT_MAX - 2 * kUnitRows || rows_k > INT_MAX - 2 * kBN) return ATTN_ERR_INVALID_ARG;
  const long long units_bound = varlen
      ? static_cast<long long>(H) * ((rows_q + kUnitRows - 1) / kUnitRows + B)
      : static_cast<long long>(B) * H * ((Sq + kUnitRows - 1) / kUnitRows);
  if (units_bound > INT_MAX / 2) return ATTN_ERR_INVALID_ARG;
  // scratch needed by this call: one error word, whatever the problem size
  const long long scratch_needed = static_cast<long long>(sizeof(int));
  if (scratch_needed > kNoAllocScratchBytes) return ATTN_ERR_INVALID_ARG;

  // ---- device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  NoAllocDevice* ds = nullptr;
  int st = noalloc_setup(dev, &ds);
  if (st != ATTN_OK) return st;
  if (!na_on_device(q, dev) || !na_on_device(k, dev) || !na_on_device(v, dev) ||
      !na_on_device(o, dev) || !na_on_device(lse, dev))
    return ATTN_ERR_INVALID_ARG;
  if (varlen && (!na_on_device(cu_seqlens_q, dev) || !na_on_device(cu_seqlens_k, dev)))
    return ATTN_ERR_INVALID_ARG;

  FwdParams p;
  const bool bf16 = dtype == ATTN_DTYPE_BF16;
  if (na_encode(&p.tm_q, q, rows_q, H, D, bf16) != ATTN_OK ||
      na_encode(&p.tm_k, k, rows_k, H, D, bf16) != ATTN_OK ||
      na_encode(&p.tm_v, v, rows_k, H, D, bf16) != ATTN_OK ||
      na_encode(&p.tm_kh, k, rows_k, H, D, bf16, kBN / 2) != ATTN_OK)
    return ATTN_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.err = ds->scratch;
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.varlen = varlen ? 1 : 0;
  set_mask(p, causal, -1, -1, 0);  // no window: cannot fail
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.scale_pos = scale > 0.0f ? 1 : 0;
  p.timeout_ns = 5000LL * 1000000LL;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the shared error word must start at zero for this call
  if (cudaMemsetAsync(ds->scratch, 0, sizeof(int), s) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  LaunchInfo info;
  const cudaError_t e = launch_forward(p, D, bf16, varlen, B, H, rows_q, Sq, ds->sms, s, &info);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (device_status) {  // optional: wait and report what the kernel recorded
    int word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(&word, ds->scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    *device_status = (word & kErrTimeout)      ? ATTN_ERR_DEVICE_TIMEOUT
                     : (word & kErrBadSeqlens) ? ATTN_ERR_BAD_SEQLENS
                                               : ATTN_OK;
  }
  return ATTN_OK;
}
