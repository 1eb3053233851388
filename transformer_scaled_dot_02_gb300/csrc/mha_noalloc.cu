// Multi-head attention for callers that cannot allocate device memory.
//
// mha_forward needs a device workspace for the projected Q, K, V and the
// concatenated heads, and expects the caller to allocate it.  Some callers
// cannot call cudaMalloc: code running inside a host framework that owns all
// device memory through its own pool and forbids other allocations, or code
// on a latency-critical path that must not risk the device-wide
// synchronisation an allocation can cause.  mha_forward_noalloc serves them:
// its workspace is the file-scope array below, which exists once per GPU that
// loads this library and stays allocated until the process exits.
//
// Set-up: the first call on each device looks up the array's device address
// with cudaGetSymbolAddress (with that device current) and caches it; that
// first call should come before any stream capture.  The host-side name of
// the array is only a stand-in for the symbol and is never passed to a kernel.
//
// The cached address belongs to the device's primary context: after
// cudaDeviceReset (or anything else that destroys that context) the process
// must not call the library again, as for the library's other per-device state.
//
// Every call shares the one array and it keeps the last call's contents.
// Nothing in it needs to start at zero: each call writes the projected Q, K, V
// and the heads completely before they are read.  Calls that overlap on the
// GPU (for example on two streams) race on the array and must be ordered by
// the caller.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sdpa.h"

namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(SDPA_MHA_NOALLOC_MAX_WORKSPACE);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_mha_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_mha_scratch on the current device (looked up once).
sdpa_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SDPA_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return SDPA_ERR_UNSUPPORTED_DEVICE;
    }
    if (major != 10 || minor != 3) return SDPA_ERR_UNSUPPORTED_DEVICE;
    void* ptr = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&ptr, g_mha_scratch);
    if (err != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return SDPA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return SDPA_OK;
}

}  // namespace

extern "C" sdpa_status mha_forward_noalloc(const void* xq, const void* xkv, const void* wq,
                                           const void* wk, const void* wv, const void* wo,
                                           void* y, int b, int n_q, int n_k, int d_model, int h,
                                           int d_k, int d_v, int mask_kind,
                                           const int32_t* kv_lengths, float scale,
                                           void* stream) {
  void* scratch = nullptr;
  const sdpa_status st = scratch_for_current_device(&scratch);
  if (st != SDPA_OK) return st;
  // mha_forward checks every argument first, then returns SDPA_ERR_WORKSPACE
  // (with nothing enqueued) when the problem needs more than the array holds,
  // so a bad or unsupported argument gets the same status as from mha_forward.
  return mha_forward(xq, xkv, wq, wk, wv, wo, y, scratch, kNoAllocScratchBytes, b, n_q, n_k,
                     d_model, h, d_k, d_v, mask_kind, kv_lengths, scale, stream);
}
