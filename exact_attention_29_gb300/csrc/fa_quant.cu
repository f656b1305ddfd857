// Block quantization of bf16 Q, K or V to e4m3 for the FP8 forward, with the
// incoherent rotation ("已有的几种大模型上下文支持情况" §4.4, FA-3):
//   - §4.4.2: a row x becomes y = (x o signs) H / sqrt(d), H the Sylvester-
//     Hadamard matrix and signs a random +-1 vector supplied by the caller; the
//     rotation is orthogonal, so (QR)(KR)^T = Q K^T, and it spreads an outlier
//     dimension over all of them;
//   - §4.4.1: every 128-row tile of a (batch, head) gets its own scale
//     amax / 448 (or one scale per head for V), so the largest magnitude maps
//     to the largest e4m3 value.
// d = 128. One thread transforms one row in registers (a fast Walsh-Hadamard
// transform, 7 butterfly stages); kernel 1 reduces the tile maxima, kernel 2
// recomputes the rows, scales and rounds them (cvt.rn.satfinite) and writes
// the codes row-major or transposed (V^T, rows of v_pitch bytes).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;  // rows per tile = threads per block
constexpr float kE4m3Max = 448.f;

// Row `row` of x, rotated if signs != nullptr.
__device__ __forceinline__ void load_row(const __nv_bfloat16* __restrict__ x, const float* __restrict__ signs,
                                         size_t row, float (&y)[kD]) {
  const uint4* src = reinterpret_cast<const uint4*>(x + row * kD);
#pragma unroll
  for (int i = 0; i < kD / 8; ++i) {
    const uint4 u = src[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      y[8 * i + 2 * e] = __uint_as_float(w[e] << 16);
      y[8 * i + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  }
  if (signs == nullptr) return;
#pragma unroll
  for (int i = 0; i < kD; ++i) y[i] *= __ldg(signs + i);
  // y <- H y, H symmetric: butterflies over strides 1, 2, ..., 64
#pragma unroll
  for (int h = 1; h < kD; h <<= 1) {
#pragma unroll
    for (int i = 0; i < kD; ++i) {
      if ((i & h) == 0) {
        const float a = y[i], b = y[i + h];
        y[i] = a + b;
        y[i + h] = a - b;
      }
    }
  }
  const float inv = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
  for (int i = 0; i < kD; ++i) y[i] *= inv;
}

// amax[bh][tile] over the (rotated) tile.
__global__ void __launch_bounds__(kRows) quant_amax_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const float* __restrict__ signs, float* __restrict__ amax,
                                                           int N, int tiles) {
  __shared__ float red[kRows / 32];
  const int tile = blockIdx.x, bh = blockIdx.y;
  const int n = tile * kRows + threadIdx.x;
  float m = 0.f;
  if (n < N) {
    float y[kD];
    load_row(x, signs, static_cast<size_t>(bh) * N + n, y);
#pragma unroll
    for (int i = 0; i < kD; ++i) m = fmaxf(m, fabsf(y[i]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = red[0];
#pragma unroll
    for (int i = 1; i < kRows / 32; ++i) t = fmaxf(t, red[i]);
    amax[static_cast<size_t>(bh) * tiles + tile] = t;
  }
}

__global__ void __launch_bounds__(kRows) quant_write_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ signs,
                                                            const float* __restrict__ amax, uint8_t* __restrict__ codes,
                                                            float* __restrict__ scales, int N, int tiles, int per_head,
                                                            int transpose, int v_pitch) {
  const int tile = blockIdx.x, bh = blockIdx.y;
  float a;
  if (per_head) {
    a = 0.f;
    for (int t = 0; t < tiles; ++t) a = fmaxf(a, amax[static_cast<size_t>(bh) * tiles + t]);
  } else {
    a = amax[static_cast<size_t>(bh) * tiles + tile];
  }
  const float scale = (a > 0.f) ? a / kE4m3Max : 1.f;
  if (threadIdx.x == 0) {
    if (per_head) {
      if (tile == 0) scales[bh] = scale;
    } else {
      scales[static_cast<size_t>(bh) * tiles + tile] = scale;
    }
  }
  const int n = tile * kRows + threadIdx.x;
  if (n >= N) return;
  float y[kD];
  load_row(x, signs, static_cast<size_t>(bh) * N + n, y);
  const float inv = 1.f / scale;
  if (!transpose) {
    uint4* dst = reinterpret_cast<uint4*>(codes + (static_cast<size_t>(bh) * N + n) * kD);
#pragma unroll
    for (int i = 0; i < kD / 16; ++i) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = 16 * i + 4 * e;
        w[e] = pack_e4m3x2(y[c] * inv, y[c + 1] * inv) | (pack_e4m3x2(y[c + 2] * inv, y[c + 3] * inv) << 16);
      }
      dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    // V^T: byte (c, n) of head bh at bh * 128 * v_pitch + c * v_pitch + n;
    // a warp writes 32 consecutive keys of each row c
    uint8_t* dst = codes + static_cast<size_t>(bh) * kD * v_pitch + n;
#pragma unroll
    for (int c = 0; c < kD; c += 2) {
      const uint32_t two = pack_e4m3x2(y[c] * inv, y[c + 1] * inv);
      dst[static_cast<size_t>(c) * v_pitch] = static_cast<uint8_t>(two & 0xffu);
      dst[static_cast<size_t>(c + 1) * v_pitch] = static_cast<uint8_t>(two >> 8);
    }
  }
}

}  // namespace

fa_status launch_quantize_fp8(const void* x, const float* signs, void* codes, float* scales, int B, int H, int N,
                              int per_head, int transpose, int v_pitch, float* amax_ws, cudaStream_t stream) {
  const int tiles = (N + kRows - 1) / kRows;
  const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(B * H));
  quant_amax_kernel<<<grid, kRows, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), signs, amax_ws, N, tiles);
  quant_write_kernel<<<grid, kRows, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), signs, amax_ws,
                                                 static_cast<uint8_t*>(codes), scales, N, tiles, per_head, transpose,
                                                 v_pitch);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("quantize kernels launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace fa
