// fa_decode_noalloc: Flash-Decoding without any device allocation.
//
// fa_decode takes its split-partials workspace from a stream-ordered pool on every
// call. Some callers cannot allocate device memory at call time: a serving
// engine that hands nearly all of HBM to its own KV-cache pool at start-up and
// forbids allocation afterwards, or a latency-critical decode loop where an
// allocation may stall on the pool or fail under fragmentation. This entry
// point runs the very same split and merge kernels, but their workspace is a
// fixed array in device memory that belongs to this library (file-scope
// `__device__`), so a call allocates nothing.
//
// Properties a caller must know:
//   * the array holds kNoallocWorkspaceFloats fp32 values (16 MiB); every GPU
//     that loads libfa.so keeps it until the process exits;
//   * a call needs B * H * num_splits * (d + 1) values of it and is rejected
//     with FA_ERR_INVALID_ARG (see fa_last_error_string) above that;
//   * all calls on a device share the one array and it keeps whatever the last
//     call wrote. Nothing in it has to start at zero: the split kernel writes
//     every partial (also those of empty splits) before the merge kernel reads
//     it. Calls whose kernels may overlap on the GPU (different streams without
//     ordering between them) race on the array and must not be issued;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make that
//     first call before any stream capture. The cached address belongs to the
//     CUDA context of that moment: after cudaDeviceReset the library must not
//     be used again in the process (fa_decode and the other calls cache the
//     device error word's address the same way).
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr size_t kNoallocWorkspaceFloats = size_t(1) << 22;  // 16 MiB of fp32
constexpr int kMaxDevices = 64;

// The shared workspace. In host code this name is only a stand-in for the
// symbol, never a device address: kernels get the address looked up below.
static __device__ __align__(256) float g_noalloc_workspace[kNoallocWorkspaceFloats];

std::mutex g_ws_mutex;
float* g_ws_ptr[kMaxDevices] = {};

// Device address of the workspace on the current device (looked up once per device).
fa_status workspace_ptr(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error_text("cudaGetDevice", e);
    return FA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_error_text("device index", "out of range");
    return FA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  if (g_ws_ptr[dev] == nullptr) {
    float* p = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_workspace);
    if (e != cudaSuccess) {
      set_error_text("cudaGetSymbolAddress(g_noalloc_workspace)", e);
      return FA_ERR_CUDA;
    }
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* seqlens, void* o, float* lse, int B, int H, int L, int d,
                                       int num_splits, fa_stream_t stream) {
  using namespace fa;
  fa_status st = check_decode_args(q, k_cache, v_cache, seqlens, o, lse, B, H, L, d, num_splits);
  if (st != FA_OK) return st;
  const size_t parts = static_cast<size_t>(B) * H * num_splits;
  const size_t need = parts * (d + 1);
  if (need > kNoallocWorkspaceFloats) {
    char buf[160];
    std::snprintf(buf, sizeof(buf), "needs B*H*num_splits*(d+1) = %zu fp32 values; the static workspace holds %zu",
                  need, kNoallocWorkspaceFloats);
    set_error_text("fa_decode_noalloc", buf);
    return FA_ERR_INVALID_ARG;
  }
  int dev = -1;
  st = checked_device(&dev);
  if (st != FA_OK) return st;
  float* ws = nullptr;
  st = workspace_ptr(&ws);
  if (st != FA_OK) return st;
  return launch_decode(q, k_cache, v_cache, seqlens, o, lse, B, H, L, d, num_splits, ws, ws + parts * d,
                       reinterpret_cast<cudaStream_t>(stream));
}
