// Self-tests of the building blocks the attention kernels rely on, callable
// through the C ABI so the test suite can check each one on the GPU alone:
//   * one tensor-core product through the same TMA staging, shared-memory
//     descriptors and TMEM placement as the prefill kernel (issue_qk and
//     issue_pv from fa_mma.cuh, bf16; issue_qk_f8 and issue_pv_f8, e4m3);
//   * the bounded-wait path: a wait on a barrier nothing arrives at must give
//     up, record the timeout and return.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_internal.h"
#include "fa_mma.cuh"

namespace fa {
namespace {

constexpr int kTileBytes = 128 * 128 * 2;
constexpr int kSmem = 2 * kTileBytes + 64 + 1024;

template <int K, int N>
__global__ void __launch_bounds__(128, 1)
    mma_test_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __nv_bfloat16* __restrict__ a_gmem, float* __restrict__ d, int mode, unsigned int* err) {
  extern __shared__ uint8_t raw[];
  uint8_t* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  uint8_t* sa = base;
  uint8_t* sb = base + kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 2 * kTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);  // D in columns [0, 128), A (mode 1) in [128, 192)
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  if (mode == 1) {
    // A[128][K] rows go to TMEM lanes as packed bf16 pairs, one row per thread
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(a_gmem + static_cast<size_t>(threadIdx.x) * K);
    uint32_t r[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) r[i] = arow[i];
    tmem_st_x64(tmem + lane_base + 128, r);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();

  if (threadIdx.x == 0) {
    tc_fence_after();
    if (mode == 0) {
      mbar_arrive_expect_tx(&bars[0], 2 * 128 * K * 2);
      for (int c = 0; c < K / 64; ++c) {
        tma_load_3d(sa + c * kChunkBytes, &tm_a, &bars[0], c * 64, 0, 0);
        tma_load_3d(sb + c * kChunkBytes, &tm_b, &bars[0], c * 64, 0, 0);
      }
    } else {
      mbar_arrive_expect_tx(&bars[0], 128 * N * 2);
      for (int c = 0; c < N / 64; ++c) tma_load_3d(sb + c * kChunkBytes, &tm_b, &bars[0], c * 64, 0, 0);
    }
    const bool ok = bounded_wait(&bars[0], 0, nullptr, err, kSiteSelftest);
    if (ok) {
      tc_fence_after();
      if (mode == 0)
        issue_qk<K>(tmem, smem_u32(sa), smem_u32(sb));
      else
        issue_pv<N>(tmem, tmem + 128, smem_u32(sb), false);
    }
    umma_commit(&bars[1]);
  }
  __syncwarp();
  const bool done = bounded_wait(&bars[1], 0, nullptr, err, kSiteSelftest);
  if (__all_sync(0xffffffffu, done)) {
    tc_fence_after();
    const int row = warp * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < N; c += 32) {
      uint32_t r[32];
      tmem_ld_x32(tmem + lane_base + c, r);
#pragma unroll
      for (int i = 0; i < 32; ++i) d[static_cast<size_t>(row) * N + c + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// e4m3 products, 128 x 128 x 128:
//   mode 2: D = A B^T, A [128][128] and B [128][128] e4m3 K-major (issue_qk_f8)
//   mode 3: D = A B^T with A placed in TMEM (four e4m3 per column) and B
//           [128][128] K-major in shared memory (issue_pv_f8, B = V^T)
__global__ void __launch_bounds__(128, 1)
    mma_f8_test_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                       const uint8_t* __restrict__ a_gmem, float* __restrict__ d, int mode, unsigned int* err) {
  extern __shared__ uint8_t raw[];
  uint8_t* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  constexpr int kT = 128 * 128;
  uint8_t* sa = base;
  uint8_t* sb = base + kT;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 2 * kT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);  // D in [0, 128), A (mode 3) in [128, 160)
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  if (mode == 3) {
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(a_gmem + static_cast<size_t>(threadIdx.x) * 128);
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = arow[i];
    tmem_st_x32(tmem + lane_base + 128, r);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    tc_fence_after();
    mbar_arrive_expect_tx(&bars[0], mode == 2 ? 2 * kT : kT);
    if (mode == 2) tma_load_3d(sa, &tm_a, &bars[0], 0, 0, 0);
    tma_load_3d(sb, &tm_b, &bars[0], 0, 0, 0);
    const bool ok = bounded_wait(&bars[0], 0, nullptr, err, kSiteSelftest);
    if (ok) {
      tc_fence_after();
      if (mode == 2)
        issue_qk_f8(tmem, smem_u32(sa), smem_u32(sb));
      else
        issue_pv_f8(tmem, tmem + 128, smem_u32(sb), false);
    }
    umma_commit(&bars[1]);
  }
  __syncwarp();
  const bool done = bounded_wait(&bars[1], 0, nullptr, err, kSiteSelftest);
  if (__all_sync(0xffffffffu, done)) {
    tc_fence_after();
    const int row = warp * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      uint32_t r[32];
      tmem_ld_x32(tmem + lane_base + c, r);
#pragma unroll
      for (int i = 0; i < 32; ++i) d[static_cast<size_t>(row) * 128 + c + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

fa_status launch_mma_f8(int mode, const void* a, const void* b, float* d, cudaStream_t stream, unsigned int* err) {
  CUtensorMap ta, tb;
  if (!encode_u8_map(&ta, a, 128, 128, 1, 128, 128) || !encode_u8_map(&tb, b, 128, 128, 1, 128, 128))
    return FA_ERR_CUDA;
  constexpr int smem = 2 * 128 * 128 + 64 + 1024;
  cudaError_t e = cudaFuncSetAttribute(mma_f8_test_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    set_error_text("cudaFuncSetAttribute(mma_f8_test_kernel)", e);
    return FA_ERR_CUDA;
  }
  mma_f8_test_kernel<<<1, 128, smem, stream>>>(ta, tb, static_cast<const uint8_t*>(a), d, mode, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("mma_f8_test_kernel launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// Products of a CTA pair (M = 256, tcgen05 .cta_group::2), both operands in
// shared memory; CTA r holds rows [128r, 128r + 128) of A and receives the
// same rows of D:
//   mode 4: D[256][128] = A[256][128] * B[128][128]^T, B K-major, CTA r holds
//           B rows [64r, 64r + 64) (the S = Q K^T product of the pair kernel);
//   mode 5: D[256][128] = A[256][128] * B[128][128], B MN-major, CTA r holds B
//           columns [64r, 64r + 64) (the O += P V product with P in shared memory).
// d also receives, after the 256 x 128 values, each CTA's TMEM base address.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    pair_mma_test_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         float* __restrict__ d, int mode, unsigned int* err) {
  extern __shared__ uint8_t raw[];
  uint8_t* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  uint8_t* sa = base;                    // 2 chunks of 128 rows x 128 B
  uint8_t* sb = base + 2 * kChunkBytes;  // mode 4: 2 chunks of 64 rows; mode 5: 1 chunk of 128 rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 3 * kChunkBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);  // this CTA's operands landed
    mbar_init(&bars[1], 1);  // the pair's product is done (commit to both CTAs)
    mbar_init(&bars[2], 2);  // even CTA: both CTAs' operands landed
    fence_barrier_init();
  }
  cluster_sync();
  if (warp == 0) {
    tmem_alloc_pair(tmem_slot, 256);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[0], 3 * kChunkBytes);
    for (int c = 0; c < 2; ++c)
      tma_load_3d(sa + c * kChunkBytes, &tm_a, &bars[0], c * 64, 128 * static_cast<int>(rank), 0);
    if (mode == 4) {
      for (int c = 0; c < 2; ++c)
        tma_load_3d(sb + c * (kChunkBytes / 2), &tm_b, &bars[0], c * 64, 64 * static_cast<int>(rank), 0);
    } else {
      tma_load_3d(sb, &tm_b, &bars[0], 64 * static_cast<int>(rank), 0, 0);
    }
    bounded_wait(&bars[0], 0, nullptr, err, kSiteSelftest);
    mbar_arrive_cluster(mapa_shared(&bars[2], 0));
    if (rank == 0) {
      const bool ok = bounded_wait_cluster(&bars[2], 0, nullptr, err, kSiteSelftest);
      if (ok) {
        tc_fence_after();
        const uint64_t ad = smem_desc_sw128(smem_u32(sa), 16, 1024);
        if (mode == 4) {
          constexpr uint32_t idesc = idesc_bf16_f32(256, 128, false, false);
          const uint64_t bd = smem_desc_sw128(smem_u32(sb), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t k32 = static_cast<uint32_t>((kk % 4) * 32);
            umma_ss_pair(tmem, ad + desc_step((kk / 4) * kChunkBytes + k32),
                         bd + desc_step((kk / 4) * (kChunkBytes / 2) + k32), idesc, kk > 0 ? 1u : 0u);
          }
        } else {
          constexpr uint32_t idesc = idesc_bf16_f32(256, 128, false, true);
          const uint64_t bd = smem_desc_sw128(smem_u32(sb), kChunkBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss_pair(tmem, ad + desc_step((kk / 4) * kChunkBytes + (kk % 4) * 32), bd + desc_step(kk * 2048),
                         idesc, kk > 0 ? 1u : 0u);
        }
      }
      umma_commit_pair(&bars[1]);
    }
  }
  __syncwarp();
  const bool done = bounded_wait(&bars[1], 0, nullptr, err, kSiteSelftest);
  if (__all_sync(0xffffffffu, done)) {
    tc_fence_after();
    const int row = 128 * static_cast<int>(rank) + warp * 32 + lane;
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      uint32_t r[32];
      tmem_ld_x32(tmem + lane_base + c, r);
#pragma unroll
      for (int i = 0; i < 32; ++i) d[static_cast<size_t>(row) * 128 + c + i] = __uint_as_float(r[i]);
    }
  }
  if (threadIdx.x == 0) d[256 * 128 + rank] = __uint_as_float(tmem);
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, 256);
  }
  cluster_sync();
}

fa_status launch_pair_mma(int mode, const void* a, const void* b, float* d, cudaStream_t stream, unsigned int* err) {
  CUtensorMap ta, tb;
  // A [256][128] K-major, 128-row boxes; B [128][128]: K-major 64-row boxes (mode 4)
  // or MN-major (rows = contraction index) 128-row boxes of 64 columns (mode 5)
  if (!encode_bf16_map(&ta, a, 128, 256, 1, 128) || !encode_bf16_map(&tb, b, 128, 128, 1, mode == 4 ? 64 : 128))
    return FA_ERR_CUDA;
  constexpr int smem = 3 * kChunkBytes + 64 + 1024;
  cudaError_t e = cudaFuncSetAttribute(pair_mma_test_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    set_error_text("cudaFuncSetAttribute(pair_mma_test_kernel)", e);
    return FA_ERR_CUDA;
  }
  pair_mma_test_kernel<<<2, 128, smem, stream>>>(ta, tb, d, mode, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("pair_mma_test_kernel launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

__global__ void wait_test_kernel(unsigned int* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: this wait must run out and return
  if (threadIdx.x == 0) bounded_wait(&bar, 0, nullptr, err, kSiteSelftest, timeout_ns);
}

template <int K, int N>
fa_status launch_mma(int mode, const void* a, const void* b, float* d, cudaStream_t stream, unsigned int* err) {
  CUtensorMap ta, tb;
  if (mode == 0) {
    // A [128][K], B [N][K]: K-major tiles of 128 rows
    if (!encode_bf16_map(&ta, a, K, 128, 1, 128) || !encode_bf16_map(&tb, b, K, N, 1, 128)) return FA_ERR_CUDA;
  } else {
    // B [K = 128][N]: rows are the contraction index, N contiguous (MN-major)
    if (!encode_bf16_map(&tb, b, N, 128, 1, 128)) return FA_ERR_CUDA;
    ta = tb;
  }
  cudaError_t e = cudaFuncSetAttribute(mma_test_kernel<K, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) {
    set_error_text("cudaFuncSetAttribute(mma_test_kernel)", e);
    return FA_ERR_CUDA;
  }
  mma_test_kernel<K, N><<<1, 128, kSmem, stream>>>(ta, tb, static_cast<const __nv_bfloat16*>(a), d, mode, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("mma_test_kernel launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

fa_status launch_selftest_mma(int mode, const void* a, const void* b, float* d, int n, int k, cudaStream_t stream,
                              unsigned int* err) {
  if (mode == 0 && n == 128 && k == 128) return launch_mma<128, 128>(0, a, b, d, stream, err);
  if (mode == 0 && n == 128 && k == 64) return launch_mma<64, 128>(0, a, b, d, stream, err);
  if (mode == 1 && n == 128 && k == 128) return launch_mma<128, 128>(1, a, b, d, stream, err);
  if (mode == 1 && n == 64 && k == 128) return launch_mma<128, 64>(1, a, b, d, stream, err);
  if ((mode == 2 || mode == 3) && n == 128 && k == 128) return launch_mma_f8(mode, a, b, d, stream, err);
  if ((mode == 4 || mode == 5) && n == 128 && k == 128) return launch_pair_mma(mode, a, b, d, stream, err);
  return FA_ERR_UNSUPPORTED;
}

fa_status launch_selftest_wait(unsigned int timeout_us, cudaStream_t stream, unsigned int* err) {
  wait_test_kernel<<<1, 32, 0, stream>>>(err, static_cast<unsigned long long>(timeout_us) * 1000ull);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("wait_test_kernel launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace fa
