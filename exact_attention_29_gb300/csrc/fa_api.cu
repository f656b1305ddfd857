// C ABI of libfa.so (declared in include/fa.h): argument checks, per-device
// lookups, tensor-map encoding, the device error word, and dispatch to the
// kernels. No attention arithmetic lives here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {

// The device error word (flags, first site); see fa_common.cuh.
__device__ unsigned int g_error_word[2];

namespace {

constexpr int kMaxDevices = 64;
thread_local char t_error_text[512] = "";
thread_local int t_error_site = 0;  // site of the last failed wait or check seen by fa_check_device_error

std::mutex g_mutex;
unsigned int* g_err_ptr[kMaxDevices] = {};
int g_dev_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
int g_num_sms[kMaxDevices] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Current device, checked once to be compute capability 10.3.
fa_status current_device(int* dev_out) {
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
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) {
      set_error_text("cudaDeviceGetAttribute", e);
      return FA_ERR_CUDA;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      set_error_text("cudaDeviceGetAttribute(multiProcessorCount)", e);
      return FA_ERR_CUDA;
    }
    g_num_sms[dev] = sms;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_dev_ok[dev] != 1) {
    set_error_text("device", "kernels are built for sm_103a only");
    return FA_ERR_UNSUPPORTED;
  }
  *dev_out = dev;
  return FA_OK;
}

// Workspaces come from a memory pool the library owns on each device, which
// keeps up to kPoolKeepBytes mapped between calls (the default pool returns
// its memory at every synchronisation, and mapping it again costs about
// 0.1 ms per call). Allocation and release are stream-ordered.
constexpr uint64_t kPoolKeepBytes = 4ull << 30;
cudaMemPool_t g_pool[kMaxDevices] = {};

fa_status ws_alloc(int dev, void** ptr, size_t bytes, cudaStream_t stream, const char* what) {
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_pool[dev] == nullptr) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.handleTypes = cudaMemHandleTypeNone;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t pool = nullptr;
      cudaError_t e = cudaMemPoolCreate(&pool, &props);
      if (e == cudaSuccess) {
        uint64_t keep = kPoolKeepBytes;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
      }
      if (e == cudaSuccess) {
        // Blocks are reused by the stream that released them (and across an
        // event dependency the caller made), never by making one stream wait for
        // another nor by taking another stream's block as soon as it is free.
        // A caller that pipelines steps over several streams then keeps one
        // workspace per stream, instead of streams stealing blocks from each
        // other, the pool growing in the middle of the pipeline, or hidden waits
        // serialising the streams.
        int no = 0;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolReuseAllowInternalDependencies, &no);
        if (e == cudaSuccess) e = cudaMemPoolSetAttribute(pool, cudaMemPoolReuseAllowOpportunistic, &no);
      }
      if (e != cudaSuccess) {
        set_error_text("cudaMemPoolCreate(workspace pool)", e);
        return FA_ERR_CUDA;
      }
      g_pool[dev] = pool;
    }
  }
  const cudaError_t e = cudaMallocFromPoolAsync(ptr, bytes, g_pool[dev], stream);
  if (e != cudaSuccess) {
    set_error_text(what, e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

void set_error_text(const char* what, cudaError_t err) {
  std::snprintf(t_error_text, sizeof(t_error_text), "%s: %s (%s)", what, cudaGetErrorName(err),
                cudaGetErrorString(err));
}

void set_error_text(const char* what, const char* detail) {
  std::snprintf(t_error_text, sizeof(t_error_text), "%s: %s", what, detail);
}

unsigned int* device_error_word() {
  int dev = -1;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) {
    set_error_text("cudaGetDevice", ge);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_error_text("device index", "out of range");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) {
      set_error_text("cudaGetSymbolAddress(g_error_word)", e);
      return nullptr;
    }
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_err_ptr[dev];
}

namespace {

// A 3-D map over [outer][rows][inner] with 128-byte swizzle, rows row_pitch
// bytes apart, and a box of box_inner x box_rows x 1 elements
// (box_inner x elem_bytes = 128 bytes).
bool encode_3d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t box_inner, const void* base, uint64_t inner,
               uint64_t rows, uint64_t outer, uint32_t box_rows, uint64_t row_pitch) {
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                             cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
        set_error_text("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", e);
        return false;
      }
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  const cuuint64_t dims[3] = {inner, rows, outer};
  const cuuint64_t strides[2] = {row_pitch, rows * row_pitch};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[64];
    std::snprintf(buf, sizeof(buf), "CUresult %d", static_cast<int>(r));
    set_error_text("cuTensorMapEncodeTiled", buf);
    return false;
  }
  return true;
}

}  // namespace

bool encode_bf16_map(CUtensorMap* map, const void* base, uint64_t d, uint64_t rows, uint64_t outer,
                     uint32_t box_rows) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, base, d, rows, outer, box_rows, d * 2);
}

bool encode_u8_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t outer,
                   uint32_t box_rows, uint64_t row_pitch) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 128, base, inner, rows, outer, box_rows, row_pitch);
}

bool encode_f32_map(CUtensorMap* map, const void* base, uint64_t d, uint64_t rows, uint64_t outer,
                    uint32_t box_rows) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 32, base, d, rows, outer, box_rows, d * 4);
}

fa_status reject(fa_status status, const char* failed_check) {
  set_error_text("argument rejected", failed_check);
  return status;
}

fa_status checked_device(int* dev) { return current_device(dev); }

// The checks fa_decode and fa_decode_noalloc share.
fa_status check_decode_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens,
                            const void* o, const float* lse, int B, int H, int L, int d, int num_splits) {
  FA_REJECT_IF(!q || !k_cache || !v_cache || !seqlens || !o || !lse, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned4(seqlens) || !aligned4(o) ||
                   !aligned4(lse),
               FA_ERR_INVALID_ARG);
  FA_REJECT_IF(B < 1 || H < 1 || L < 1 || d < 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(num_splits < 1 || num_splits > 64, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(d != 64 && d != 128, FA_ERR_UNSUPPORTED);
  FA_REJECT_IF(static_cast<long long>(B) * H > 0x7fffffffLL || H > 65535 || B > 65535, FA_ERR_INVALID_ARG);
  return FA_OK;
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(fa_status status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dimension or device";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
    case FA_ERR_CHECK: return "FA_ERR_CHECK: a kernel's roles disagreed on their protocol counts (FA_DEBUG build)";
  }
  return "unknown fa_status";
}

const char* fa_last_error_string(void) { return t_error_text; }

int fa_last_error_site(void) { return t_error_site; }

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 int causal, float scale, fa_stream_t stream) {
  FA_REJECT_IF(!q || !k || !v || !o || !lse, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(B < 1 || H < 1 || N < 1 || d < 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!(scale > 0.f) || !std::isfinite(scale), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(causal != 0 && causal != 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(d != 64 && d != 128, FA_ERR_UNSUPPORTED);
  const long long bh = static_cast<long long>(B) * H;
  const long long pairs = (static_cast<long long>(N) + 255) / 256;
  FA_REJECT_IF(bh > 0x7fffffffLL || pairs > 65535 || bh * pairs > 0x7fffffffLL, FA_ERR_INVALID_ARG);
  int dev = -1;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  unsigned int* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  return launch_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, reinterpret_cast<cudaStream_t>(stream), err,
                    g_num_sms[dev]);
}

namespace {

// True when the runtime knows `p` as memory of a device (not host, managed or
// unregistered host memory). Such a pointer is refused where the call copies
// from or to the host.
bool device_memory(const void* p) {
  cudaPointerAttributes a = {};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice;
}

}  // namespace

fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                      int causal, float scale, fa_stream_t stream) {
  FA_REJECT_IF(!q || !k || !v || !o || !lse, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(B < 1 || H < 1 || N < 1 || d < 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!(scale > 0.f) || !std::isfinite(scale), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(causal != 0 && causal != 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(d != 64 && d != 128, FA_ERR_UNSUPPORTED);
  const long long bh = static_cast<long long>(B) * H;
  const long long pairs = (static_cast<long long>(N) + 255) / 256;
  FA_REJECT_IF(bh > 0x7fffffffLL || pairs > 65535 || bh * pairs > 0x7fffffffLL, FA_ERR_INVALID_ARG);
  int dev = -1;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  unsigned int* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // one pool buffer: q, k, v, o (bf16, 256-byte multiples apart) then lse
  const size_t tensor = static_cast<size_t>(bh) * N * d * 2;
  const size_t slot = (tensor + 255) / 256 * 256;
  const size_t lse_bytes = static_cast<size_t>(bh) * N * sizeof(float);
  void* ws = nullptr;
  for (const void* p : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse)}) {
    if (device_memory(p)) {
      set_error_text("fa_fwd_host: a buffer is device memory (use fa_fwd)", cudaErrorInvalidValue);
      return FA_ERR_INVALID_ARG;
    }
  }
  st = ws_alloc(dev, &ws, 4 * slot + lse_bytes, s, "workspace allocation (host-buffer prefill)");
  if (st != FA_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* dq = base;
  void* dk = base + slot;
  void* dv = base + 2 * slot;
  void* dout = base + 3 * slot;
  float* dlse = reinterpret_cast<float*>(base + 4 * slot);
  cudaError_t e = cudaSuccess;
  const char* what = nullptr;
  if ((e = cudaMemcpyAsync(dq, q, tensor, cudaMemcpyHostToDevice, s)) != cudaSuccess) what = "cudaMemcpyAsync(q)";
  else if ((e = cudaMemcpyAsync(dk, k, tensor, cudaMemcpyHostToDevice, s)) != cudaSuccess) what = "cudaMemcpyAsync(k)";
  else if ((e = cudaMemcpyAsync(dv, v, tensor, cudaMemcpyHostToDevice, s)) != cudaSuccess) what = "cudaMemcpyAsync(v)";
  if (what) {
    set_error_text(what, e);
    cudaFreeAsync(ws, s);
    return FA_ERR_CUDA;
  }
  st = launch_fwd(dq, dk, dv, dout, dlse, B, H, N, d, causal, scale, s, err, g_num_sms[dev]);
  if (st == FA_OK) {
    if ((e = cudaMemcpyAsync(o, dout, tensor, cudaMemcpyDeviceToHost, s)) != cudaSuccess) what = "cudaMemcpyAsync(o)";
    else if ((e = cudaMemcpyAsync(lse, dlse, lse_bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
      what = "cudaMemcpyAsync(lse)";
    if (what) {
      set_error_text(what, e);
      st = FA_ERR_CUDA;
    }
  }
  e = cudaFreeAsync(ws, s);
  if (st == FA_OK && e != cudaSuccess) {
    set_error_text("cudaFreeAsync(host-buffer prefill)", e);
    st = FA_ERR_CUDA;
  }
  return st;
}

fa_status fa_fwd_sparse(const void* q, const void* k, const void* v, const uint8_t* mask, int mask_heads, void* o,
                        float* lse, int B, int H, int N, int d, int causal, float scale, fa_stream_t stream) {
  FA_REJECT_IF(!q || !k || !v || !mask || !o || !lse, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(B < 1 || H < 1 || N < 1 || d < 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(mask_heads != 1 && mask_heads != H, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!(scale > 0.f) || !std::isfinite(scale), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(causal != 0 && causal != 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(d != 64 && d != 128, FA_ERR_UNSUPPORTED);
  const long long bh = static_cast<long long>(B) * H;
  // the step lists hold a K/V tile index + 1 in 16 bits
  const long long tiles_ll = (static_cast<long long>(N) + 127) / 128;
  FA_REJECT_IF(bh > 0x7fffffffLL || tiles_ll > 65535 || bh * ((tiles_ll + 1) / 2) > 0x7fffffffLL,
               FA_ERR_INVALID_ARG);
  int dev = -1;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  unsigned int* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t tiles = (static_cast<size_t>(N) + 127) / 128;
  const size_t rows = static_cast<size_t>(mask_heads) * ((static_cast<size_t>(N) + 255) / 256);
  void* ws = nullptr;
  // step lists, their counts, and the forward's run-time item counter
  st = ws_alloc(dev, &ws, rows * tiles * sizeof(uint32_t) + (3 * rows + 1) * sizeof(int), s,
                "workspace allocation (block-sparse step lists)");
  if (st != FA_OK) return st;
  cudaError_t e = cudaSuccess;
  uint32_t* list = static_cast<uint32_t*>(ws);
  int* cnt = reinterpret_cast<int*>(list + rows * tiles);
  st = launch_fwd_sparse(q, k, v, mask, mask_heads, o, lse, B, H, N, d, causal, scale, list, cnt, s, err,
                         g_num_sms[dev]);
  e = cudaFreeAsync(ws, s);
  if (st == FA_OK && e != cudaSuccess) {
    set_error_text("cudaFreeAsync(block-sparse step lists)", e);
    st = FA_ERR_CUDA;
  }
  return st;
}

fa_status fa_fwd_sparse_plan(const uint8_t* mask, int mask_heads, int B, int H, int N, int causal,
                             long long* pairs_allowed, long long* pairs_computed) {
  FA_REJECT_IF(!mask || !pairs_allowed || !pairs_computed || B < 1 || H < 1 || N < 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(mask_heads != 1 && mask_heads != H, FA_ERR_INVALID_ARG);
  const int T = (N + 127) / 128;
  long long allowed = 0, computed = 0;
  for (int h = 0; h < H; ++h) {
    const uint8_t* mk = mask + static_cast<size_t>(mask_heads == 1 ? 0 : h) * T * T;
    auto ok = [&](int i, int j) { return (!causal || j <= i) && mk[static_cast<size_t>(i) * T + j] != 0; };
    for (int i = 0; i < T; ++i)
      for (int j = 0; j < T; ++j) allowed += ok(i, j) ? 1 : 0;
    // each Q tile computes exactly the (Q tile, K/V tile) pairs its mask keeps
    computed = allowed;
  }
  *pairs_allowed = allowed * B;
  *pairs_computed = computed * B;
  return FA_OK;
}

fa_status fa_quantize_fp8(const void* x, const float* signs, void* codes, float* scales, int B, int H, int N, int d,
                          int per_head, int transpose, int v_pitch, fa_stream_t stream) {
  FA_REJECT_IF(!x || !codes || !scales, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!aligned16(x) || !aligned16(codes) || !aligned4(scales) || (signs && !aligned4(signs)),
               FA_ERR_INVALID_ARG);
  FA_REJECT_IF(B < 1 || H < 1 || N < 1 || d < 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF((per_head != 0 && per_head != 1) || (transpose != 0 && transpose != 1), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(transpose && (v_pitch < N || v_pitch % 16 != 0), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(d != 128, FA_ERR_UNSUPPORTED);
  const long long bh = static_cast<long long>(B) * H;
  const long long tiles = (static_cast<long long>(N) + 127) / 128;
  FA_REJECT_IF(bh > 65535 || tiles > 0x7fffffffLL, FA_ERR_INVALID_ARG);
  int dev = -1;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  st = ws_alloc(dev, &ws, static_cast<size_t>(bh * tiles) * sizeof(float), s,
                "workspace allocation (quantize workspace)");
  if (st != FA_OK) return st;
  cudaError_t e = cudaSuccess;
  st = launch_quantize_fp8(x, signs, codes, scales, B, H, N, per_head, transpose, transpose ? v_pitch : 0,
                           static_cast<float*>(ws), s);
  e = cudaFreeAsync(ws, s);
  if (st == FA_OK && e != cudaSuccess) {
    set_error_text("cudaFreeAsync(quantize workspace)", e);
    st = FA_ERR_CUDA;
  }
  return st;
}

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale, const float* k_scale,
                     const float* v_scale, void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                     int v_pitch, fa_stream_t stream) {
  FA_REJECT_IF(!q8 || !k8 || !vt8 || !q_scale || !k_scale || !v_scale || !o || !lse, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) || !aligned4(lse) ||
                   !aligned4(q_scale) || !aligned4(k_scale) || !aligned4(v_scale),
               FA_ERR_INVALID_ARG);
  FA_REJECT_IF(B < 1 || H < 1 || N < 1 || d < 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!(scale > 0.f) || !std::isfinite(scale), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(causal != 0 && causal != 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(v_pitch < N || v_pitch % 16 != 0, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(d != 128, FA_ERR_UNSUPPORTED);
  const long long bh = static_cast<long long>(B) * H;
  const long long pairs = (static_cast<long long>(N) + 255) / 256;
  FA_REJECT_IF(bh > 0x7fffffffLL || pairs > 65535 || bh * pairs > 0x7fffffffLL, FA_ERR_INVALID_ARG);
  int dev = -1;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  unsigned int* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  return launch_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, B, H, N, d, causal, scale, v_pitch,
                        reinterpret_cast<cudaStream_t>(stream), err, g_num_sms[dev]);
}

fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens, void* o,
                    float* lse, int B, int H, int L, int d, int num_splits, fa_stream_t stream) {
  fa_status st = check_decode_args(q, k_cache, v_cache, seqlens, o, lse, B, H, L, d, num_splits);
  if (st != FA_OK) return st;
  int dev = -1;
  st = current_device(&dev);
  if (st != FA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t parts = static_cast<size_t>(B) * H * num_splits;
  void* ws = nullptr;
  st = ws_alloc(dev, &ws, parts * (d + 1) * sizeof(float), s, "workspace allocation (decode workspace)");
  if (st != FA_OK) return st;
  cudaError_t e = cudaSuccess;
  float* ws_o = static_cast<float*>(ws);
  float* ws_lse = ws_o + parts * d;
  st = launch_decode(q, k_cache, v_cache, seqlens, o, lse, B, H, L, d, num_splits, ws_o, ws_lse, s);
  e = cudaFreeAsync(ws, s);
  if (st == FA_OK && e != cudaSuccess) {
    set_error_text("cudaFreeAsync(decode workspace)", e);
    st = FA_ERR_CUDA;
  }
  return st;
}

fa_status fa_decode_gqa(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens, void* o,
                        float* lse, int B, int Hq, int Hkv, int L, int d, int num_splits, fa_stream_t stream) {
  FA_REJECT_IF(!q || !k_cache || !v_cache || !seqlens || !o || !lse, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned4(seqlens) || !aligned4(o) ||
                   !aligned4(lse),
               FA_ERR_INVALID_ARG);
  FA_REJECT_IF(B < 1 || Hq < 1 || Hkv < 1 || L < 1 || d < 1 || Hq % Hkv != 0, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(num_splits < 1 || num_splits > 64, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(d != 64 && d != 128, FA_ERR_UNSUPPORTED);
  const long long groups = (Hq / Hkv + 15) / 16;
  FA_REJECT_IF(B > 65535 || static_cast<long long>(Hkv) * groups > 65535 ||
                   static_cast<long long>(B) * Hq > 0x7fffffffLL,
               FA_ERR_INVALID_ARG);
  int dev = -1;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  unsigned int* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t parts = static_cast<size_t>(B) * Hq * num_splits;
  void* ws = nullptr;
  st = ws_alloc(dev, &ws, parts * (d + 1) * sizeof(float), s, "workspace allocation (decode workspace)");
  if (st != FA_OK) return st;
  cudaError_t e = cudaSuccess;
  float* ws_o = static_cast<float*>(ws);
  float* ws_lse = ws_o + parts * d;
  st = launch_decode_gqa_split(q, k_cache, v_cache, seqlens, B, Hq, Hkv, L, d, num_splits, ws_o, ws_lse, s, err);
  if (st == FA_OK) st = launch_decode_merge(ws_o, ws_lse, o, lse, static_cast<long long>(B) * Hq, d, num_splits, s);
  e = cudaFreeAsync(ws, s);
  if (st == FA_OK && e != cudaSuccess) {
    set_error_text("cudaFreeAsync(decode workspace)", e);
    st = FA_ERR_CUDA;
  }
  return st;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, fa_stream_t stream) {
  FA_REJECT_IF(!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
                   !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv),
               FA_ERR_INVALID_ARG);
  FA_REJECT_IF(B < 1 || H < 1 || N < 1 || d < 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(!(scale > 0.f) || !std::isfinite(scale), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(causal != 0 && causal != 1, FA_ERR_INVALID_ARG);
  FA_REJECT_IF(d != 64 && d != 128, FA_ERR_UNSUPPORTED);
  const long long bh = static_cast<long long>(B) * H;
  FA_REJECT_IF(bh > 0x7fffffffLL || (static_cast<long long>(N) + 127) / 128 > 65535, FA_ERR_INVALID_ARG);
  int dev = -1;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  unsigned int* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(bh) * N;
  void* ws = nullptr;
  st = ws_alloc(dev, &ws, rows * (d + 1) * sizeof(float), s, "workspace allocation (backward workspace)");
  if (st != FA_OK) return st;
  cudaError_t e = cudaSuccess;
  float* dq_acc = static_cast<float*>(ws);
  float* delta = dq_acc + rows * d;
  st = launch_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale, dq_acc, delta, s, err);
  e = cudaFreeAsync(ws, s);
  if (st == FA_OK && e != cudaSuccess) {
    set_error_text("cudaFreeAsync(backward workspace)", e);
    st = FA_ERR_CUDA;
  }
  return st;
}

fa_status fa_bwd_plan(int N, int d, int block, int causal, long long* dq_atomic_adds) {
  FA_REJECT_IF(N < 1 || d < 1 || block < 1 || !dq_atomic_adds, FA_ERR_INVALID_ARG);
  const long long t = (static_cast<long long>(N) + block - 1) / block;
  long long adds = 0;
  for (long long j = 0; j < t; ++j) {
    // Q tiles that see K/V tile j, each adding its rows (clipped to N) to dQ
    for (long long i = (causal ? j : 0); i < t; ++i) {
      const long long rows = (i * block + block <= N) ? block : (N - i * block);
      adds += rows * d;
    }
  }
  *dq_atomic_adds = adds;
  return FA_OK;
}

fa_status fa_check_device_error(fa_stream_t stream) {
  t_error_site = 0;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_error_text("cudaStreamSynchronize", e);
    return FA_ERR_CUDA;
  }
  unsigned int* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  unsigned int host[2] = {0, 0};
  e = cudaMemcpy(host, err, sizeof(host), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && host[0] != 0) e = cudaMemset(err, 0, sizeof(host));
  if (e != cudaSuccess) {
    set_error_text("reading the device error word", e);
    return FA_ERR_CUDA;
  }
  if ((host[0] & (kErrTimeout | kErrCheck)) == 0) return FA_OK;
  t_error_site = static_cast<int>(host[1]);
  char buf[96];
  std::snprintf(buf, sizeof(buf), "site %d (%s)", t_error_site,
                (host[0] & kErrTimeout) ? "a bounded wait ran out" : "protocol check failed");
  set_error_text("device error word", buf);
  return (host[0] & kErrTimeout) ? FA_ERR_TIMEOUT : FA_ERR_CHECK;
}

fa_status fa_fwd_plan(int N, int block, int causal, long long* pairs_total, long long* pairs_computed) {
  FA_REJECT_IF(N < 1 || block < 1 || !pairs_total || !pairs_computed, FA_ERR_INVALID_ARG);
  const long long t = (static_cast<long long>(N) + block - 1) / block;
  long long done = 0;
  for (long long i = 0; i < t; ++i) done += fwd_kv_tiles(static_cast<int>(i * block), N, block, causal);
  *pairs_total = t * t;
  *pairs_computed = done;
  return FA_OK;
}

fa_status fa_selftest_mma(int mode, const void* a, const void* b, float* d, int n, int k, fa_stream_t stream) {
  FA_REJECT_IF(!a || !b || !d || !aligned16(a) || !aligned16(b) || !aligned4(d), FA_ERR_INVALID_ARG);
  FA_REJECT_IF(mode < 0 || mode > 5, FA_ERR_INVALID_ARG);
  int dev = -1;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  unsigned int* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  return launch_selftest_mma(mode, a, b, d, n, k, reinterpret_cast<cudaStream_t>(stream), err);
}

fa_status fa_selftest_wait_timeout(unsigned int timeout_us, fa_stream_t stream) {
  FA_REJECT_IF(timeout_us == 0 || timeout_us > 5000000u, FA_ERR_INVALID_ARG);
  int dev = -1;
  fa_status st = current_device(&dev);
  if (st != FA_OK) return st;
  unsigned int* err = device_error_word();
  if (!err) return FA_ERR_CUDA;
  return launch_selftest_wait(timeout_us, reinterpret_cast<cudaStream_t>(stream), err);
}

}  // extern "C"
