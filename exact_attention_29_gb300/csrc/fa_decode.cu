// Flash-Decoding for sm_103a: split-KV partial attention + log-sum-exp merge.
//
// CMU 15-779 Lecture 5 notes §8.4: for one query token per (batch, head) the
// K/V cache is cut along the sequence into S segments (views, no copies);
// one thread block per segment computes a partial output and the segment's
// log-sum-exp; a small reduction kernel reweights the partials by their
// log-sum-exp. The reweighting is the combine operator on (m, l, o) of §4.4-4.5.
//
// The split kernel is bound by HBM bandwidth (arithmetic intensity about 1
// FLOP per byte, §8.3). Each key row (d bf16) is read by d/8 lanes with one
// 16-byte load each, so a warp reads 2 (d = 128) or 4 (d = 64) whole rows
// per instruction; every lane keeps 16 loads (8 keys of K and of V) in
// flight. The dot product of a key is reduced across its lanes with warp
// shuffles; each lane group keeps an online (m, l, o) state for the keys it
// saw, and the block combines its groups through shared memory.
// Partials are stored normalised: o_s = acc_s / l_s and lse_s = m_s + log2 l_s
// (log2 units), with an empty segment stored as o_s = 0, lse_s = -inf.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "fa_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kSplitWarps = 4;
constexpr int kSplitThreads = 32 * kSplitWarps;
constexpr int kUnroll = 8;
constexpr uint32_t kFull = 0xffffffffu;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Keys of split s of a sequence of length len: chunks of ceil(len/S) keys
// rounded up to a multiple of 64.
__device__ __forceinline__ void split_range(int len, int S, int s, int& begin, int& end) {
  const int per = (((len + S - 1) / S) + 63) / 64 * 64;
  const long long b = static_cast<long long>(s) * per;
  begin = static_cast<int>(b < len ? b : len);
  end = (begin + per < len) ? begin + per : len;
}

template <int D>
__global__ void __launch_bounds__(kSplitThreads) decode_split_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc, const __nv_bfloat16* __restrict__ vc,
    const int32_t* __restrict__ seqlens, float* __restrict__ ws_o, float* __restrict__ ws_lse, int H, int L, int S,
    float scale_log2) {
  constexpr int kLanesPerKey = D / 8;            // 16-byte slices per key row
  constexpr int kKeysPerWarp = 32 / kLanesPerKey;  // rows one warp-wide load covers
  constexpr int kGroups = kSplitWarps * kKeysPerWarp;
  constexpr int kStep = kSplitWarps * kKeysPerWarp * kUnroll;  // keys per block iteration
  constexpr int kVecPerRow = D / 8;

  __shared__ float sh_m[kGroups];
  __shared__ float sh_l[kGroups];
  __shared__ __align__(16) float sh_acc[kGroups][D];

  const int s = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerKey;   // which row of the warp-wide load
  const int part = lane % kLanesPerKey;  // which 16-byte slice of the row

  int len = seqlens[b];
  len = len < 0 ? 0 : (len > L ? L : len);
  int k_begin, k_end;
  split_range(len, S, s, k_begin, k_end);

  const size_t head = static_cast<size_t>(b) * H + h;
  float qf[8];
  bf16x8_to_f32(reinterpret_cast<const uint4*>(q + head * D)[part], qf);
#pragma unroll
  for (int e = 0; e < 8; ++e) qf[e] *= scale_log2;  // scores in log2 units

  const uint4* kbase = reinterpret_cast<const uint4*>(kc + head * static_cast<size_t>(L) * D) + part;
  const uint4* vbase = reinterpret_cast<const uint4*>(vc + head * static_cast<size_t>(L) * D) + part;

  float m = -INFINITY, l = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;

  for (int base = k_begin + warp * kKeysPerWarp * kUnroll; base < k_end; base += kStep) {
    uint4 kr[kUnroll], vr[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int key = base + u * kKeysPerWarp + sub;
      if (key < k_end) {
        kr[u] = ldg_stream(kbase + static_cast<size_t>(key) * kVecPerRow);
        vr[u] = ldg_stream(vbase + static_cast<size_t>(key) * kVecPerRow);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float kf[8];
      bf16x8_to_f32(kr[u], kf);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) dot = fmaf(qf[e], kf[e], dot);
#pragma unroll
      for (int off = kLanesPerKey / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(kFull, dot, off);
      x[u] = (base + u * kKeysPerWarp + sub < k_end) ? dot : -INFINITY;
    }
    float mb = x[0];
#pragma unroll
    for (int u = 1; u < kUnroll; ++u) mb = fmaxf(mb, x[u]);
    const float m_new = fmaxf(m, mb);
    if (m_new == -INFINITY) continue;  // no visible key for this lane group yet
    const float alpha = ex2_approx(m - m_new);  // 0 when m was -inf
    l *= alpha;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float pu = ex2_approx(x[u] - m_new);
      float vf[8];
      bf16x8_to_f32(vr[u], vf);
      l += pu;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(pu, vf[e], acc[e]);
    }
    m = m_new;
  }

  // Combine the lane groups of the block: (m, l, acc) summaries.
  const int g = warp * kKeysPerWarp + sub;
  float4* dst = reinterpret_cast<float4*>(&sh_acc[g][part * 8]);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  if (part == 0) {
    sh_m[g] = m;
    sh_l[g] = l;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += kSplitThreads) {
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kGroups; ++i) M = fmaxf(M, sh_m[i]);
    float lsum = 0.f, o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int i = 0; i < kGroups; ++i) {
        const float w = (sh_m[i] == -INFINITY) ? 0.f : ex2_approx(sh_m[i] - M);
        lsum = fmaf(w, sh_l[i], lsum);
        o = fmaf(w, sh_acc[i][c], o);
      }
    }
    const size_t idx = head * S + s;
    ws_o[idx * D + c] = (lsum > 0.f) ? o / lsum : 0.f;
    if (c == 0) ws_lse[idx] = (lsum > 0.f) ? M + log2f(lsum) : -INFINITY;
  }
}

// One block per (batch, head), d threads: reweight the S partials by
// 2^(lse_s - max) (max and sum over splits by warp shuffles in warp 0).
template <int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(const float* __restrict__ ws_o,
                                                         const float* __restrict__ ws_lse,
                                                         __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                         int S) {
  __shared__ float sh_w[64];
  __shared__ float sh_max, sh_sum;
  const size_t head = blockIdx.x;
  const int c = threadIdx.x;
  if (c < 32) {
    const float a = (c < S) ? ws_lse[head * S + c] : -INFINITY;
    const float b = (c + 32 < S) ? ws_lse[head * S + c + 32] : -INFINITY;
    float M = fmaxf(a, b);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    const float wa = (a == -INFINITY) ? 0.f : ex2_approx(a - M);
    const float wb = (b == -INFINITY) ? 0.f : ex2_approx(b - M);
    float sum = wa + wb;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (c < S) sh_w[c] = wa;
    if (c + 32 < S) sh_w[c + 32] = wb;
    if (c == 0) {
      sh_max = M;
      sh_sum = sum;
    }
  }
  __syncthreads();
  float acc = 0.f;
  for (int s = 0; s < S; ++s) acc = fmaf(sh_w[s], ws_o[(head * S + s) * D + c], acc);
  const float sum = sh_sum;
  o[head * D + c] = __float2bfloat16_rn(sum > 0.f ? acc / sum : 0.f);
  if (c == 0) lse[head] = (sum > 0.f) ? (sh_max + log2f(sum)) * kLn2 : -INFINITY;
}

template <int D>
fa_status launch(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens, void* o,
                 float* lse, int B, int H, int L, int S, float* ws_o, float* ws_lse, cudaStream_t stream) {
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  dim3 grid(static_cast<unsigned>(S), static_cast<unsigned>(H), static_cast<unsigned>(B));
  decode_split_kernel<D><<<grid, kSplitThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k_cache),
      static_cast<const __nv_bfloat16*>(v_cache), seqlens, ws_o, ws_lse, H, L, S, scale_log2);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("decode_split_kernel launch", e);
    return FA_ERR_CUDA;
  }
  decode_merge_kernel<D><<<static_cast<unsigned>(B * H), D, 0, stream>>>(
      ws_o, ws_lse, static_cast<__nv_bfloat16*>(o), lse, S);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("decode_merge_kernel launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

fa_status launch_decode_merge(const float* ws_o, const float* ws_lse, void* o, float* lse, long long heads, int d,
                              int num_splits, cudaStream_t stream) {
  if (d == 128)
    decode_merge_kernel<128><<<static_cast<unsigned>(heads), 128, 0, stream>>>(
        ws_o, ws_lse, static_cast<__nv_bfloat16*>(o), lse, num_splits);
  else if (d == 64)
    decode_merge_kernel<64><<<static_cast<unsigned>(heads), 64, 0, stream>>>(
        ws_o, ws_lse, static_cast<__nv_bfloat16*>(o), lse, num_splits);
  else
    return FA_ERR_UNSUPPORTED;
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("decode_merge_kernel launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

fa_status launch_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens, void* o,
                        float* lse, int B, int H, int L, int d, int num_splits, float* ws_o, float* ws_lse,
                        cudaStream_t stream) {
  if (d == 128) return launch<128>(q, k_cache, v_cache, seqlens, o, lse, B, H, L, num_splits, ws_o, ws_lse, stream);
  if (d == 64) return launch<64>(q, k_cache, v_cache, seqlens, o, lse, B, H, L, num_splits, ws_o, ws_lse, stream);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
