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
//   * every device-side wait is bounded as in attn_fwd (ATTN_WAIT_TIMEOUT_MS,
//     read at every call, default 5 s);
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

#include <cstdint>
#include <mutex>

#include "attn.h"
#include "host_common.h"
#include "launch.cuh"

namespace attn {

namespace {

constexpr int kNoAllocScratchBytes = 256;

// Scratch of attn_fwd_noalloc: word 0 is the kernel's error word.
static __device__ __align__(256) int g_noalloc_scratch[kNoAllocScratchBytes / sizeof(int)];

// Device address of g_noalloc_scratch, per device (null until that device's
// first call).  In host code the array's name is only a host-side stand-in,
// so the address is looked up once per device, with that device current.
std::mutex g_na_mu;
int* g_na_scratch[host::kMaxDevices] = {};

int noalloc_scratch(int dev, int** out) {
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_na_scratch[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    g_na_scratch[dev] = static_cast<int*>(ptr);
  }
  *out = g_na_scratch[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int Sq, int Sk, int D, float scale, int causal,
                                const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                int dtype, void* stream, int* device_status) {
  if (device_status) *device_status = ATTN_OK;
  // the argument rules of attn_fwd, checked before any CUDA call
  FwdParams p;
  host::FwdCall call;
  int st = host::check_fwd_args(q, k, v, o, lse, B, H, Sq, Sk, D, scale, causal, -1, -1, 0,
                                cu_seqlens_q, cu_seqlens_k, dtype, &p, &call);
  if (st != ATTN_OK || call.nothing) return st;
  // scratch needed by this call: one error word, whatever the problem size
  const long long scratch_needed = static_cast<long long>(sizeof(int));
  if (scratch_needed > kNoAllocScratchBytes) return ATTN_ERR_INVALID_ARG;

  int dev = 0;
  if ((st = host::current_device(&dev)) != ATTN_OK) return st;
  const host::DeviceInfo* info = nullptr;
  if ((st = host::device_info(dev, &info)) != ATTN_OK) return st;
  int* scratch = nullptr;
  if ((st = noalloc_scratch(dev, &scratch)) != ATTN_OK) return st;
  if ((st = host::prepare_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale, cu_seqlens_q,
                              cu_seqlens_k, dev, call, &p)) != ATTN_OK)
    return st;
  p.err = scratch;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the shared error word must start at zero for this call
  if (cudaMemsetAsync(scratch, 0, sizeof(int), s) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  LaunchInfo linfo;
  const cudaError_t e =
      launch_forward(p, D, call.bf16, call.varlen, B, H, call.rows_q, Sq, info->sms, s, &linfo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (device_status) {  // optional: wait and report what the kernel recorded
    int word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(&word, scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    *device_status = (word & kErrTimeout)      ? ATTN_ERR_DEVICE_TIMEOUT
                     : (word & kErrBadSeqlens) ? ATTN_ERR_BAD_SEQLENS
                                               : ATTN_OK;
  }
  return ATTN_OK;
}
