// Backward pass of exact attention with recomputation, for sm_103a.
//
// CMU 15-779 Lecture 5 notes §7.2-7.4 and "FlashAttention 完全拆解（一）",
// backward section: the forward stores only O and the per-row L = m + ln l;
// the backward recomputes P = exp(S - L) block by block,
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D)  with  D_i = dO_i . O_i,
//   dQ = scale dS K,  dK = scale dS^T Q,
// with K/V blocks in the outer loop (one CTA each): dK and dV accumulate on
// chip and are written once; every K/V block adds its share of dQ into an fp32
// buffer with atomic adds (§7.4).
//
// Mapping onto one CTA (one K/V tile of 128 keys of one head, 128 threads):
//   TMEM columns: [0,128) S^T = K Q^T, then P^T (bf16 pairs, first 64
//   columns), then the dQ share dS K; [128,256) dP^T = V dO^T, then dS^T;
//   [256, 256+D) dV; [384, 384+D) dK.
//   Thread r owns key row r of S^T, dP^T, dV and dK, and query row r of the
//   dQ share. Thread 0 issues every TMA copy and tensor-core product; the
//   phases of a Q tile are separated by mbarrier waits and block barriers.
//   dS^T also goes to shared memory in the 128-byte-swizzled MN-major layout
//   so that dS (queries x keys) can be the A operand of dQ = dS K.
// Every wait is bounded (fa_common.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "fa_common.cuh"
#include "fa_internal.h"
#include "fa_mma.cuh"

namespace fa {
namespace {

constexpr int kBwdThreads = 128;
constexpr uint32_t kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;  // a K, V, Q or dO tile
  static constexpr int kChunks = D / 64;
  static constexpr int kDsBytes = 128 * 128 * 2;  // dS^T, 128 keys x 128 queries
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;
  static constexpr int kDoOff = 3 * kTileBytes;
  static constexpr int kDsOff = 4 * kTileBytes;
  static constexpr int kVecOff = kDsOff + kDsBytes;  // lse2[128], delta[128]
  static constexpr int kBarOff = kVecOff + 2 * 128 * 4;
  static constexpr int kSmemBytes = kBarOff + 8 * 8 + 1024;
  static constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 384;
};

struct BwdParams {
  const float* lse;     // [BH][N] natural log
  const float* delta;   // [BH][N] D_i = dO_i . O_i
  float* dq_acc;        // [BH][N][D] fp32, zeroed before the launch
  __nv_bfloat16* dk;    // [BH][N][D]
  __nv_bfloat16* dv;    // [BH][N][D]
  unsigned int* err;
  int N;
  int num_kv_tiles;
  int causal;
  float scale;
  float scale_log2;
};

// D_i = sum_c dO_ic O_ic in fp32, one thread per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dout,
                                                         float* __restrict__ delta, long long rows) {
  const long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= rows) return;
  const uint4* po = reinterpret_cast<const uint4*>(o + row * D);
  const uint4* pd = reinterpret_cast<const uint4*>(dout + row * D);
  float acc = 0.f;
#pragma unroll 4
  for (int i = 0; i < D / 8; ++i) {
    const uint4 a = po[i], b = pd[i];
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(wa[e] << 16), __uint_as_float(wb[e] << 16), acc);
      acc = fmaf(__uint_as_float(wa[e] & 0xffff0000u), __uint_as_float(wb[e] & 0xffff0000u), acc);
    }
  }
  delta[row] = acc;
}

// dQ (bf16) from the fp32 accumulation buffer.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                              __nv_bfloat16* __restrict__ dq, long long n4) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 v = reinterpret_cast<const float4*>(acc)[i];
  uint2 w;
  w.x = pack_bf16x2(v.x, v.y);
  w.y = pack_bf16x2(v.z, v.w);
  reinterpret_cast<uint2*>(dq)[i] = w;
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sk = base + C::kKOff;
  uint8_t* sv = base + C::kVOff;
  uint8_t* sq = base + C::kQOff;
  uint8_t* sdo = base + C::kDoOff;
  uint8_t* sds = base + C::kDsOff;
  float* lse2 = reinterpret_cast<float*>(base + C::kVecOff);
  float* dlt = lse2 + 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  uint64_t* kv_bar = &bars[0];
  uint64_t* qdo_bar = &bars[1];
  uint64_t* mma_bar = &bars[2];
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[4]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&bars[5]);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // grid (heads, K/V tiles): blocks launch in order of K/V tile, and under the
  // causal mask tile 0 (seen by every Q tile) is the heaviest
  const int bh = blockIdx.x;
  const int j = blockIdx.y;
  const int kv0 = j * 128;
  const int num_q_tiles = (p.N + 127) / 128;
  const int i_first = p.causal ? j : 0;  // Q tiles whose rows see some key of this tile

  if (tid == 0) {
    mbar_init(kv_bar, 1);
    mbar_init(qdo_bar, 1);
    mbar_init(mma_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const int row = warp * 32 + lane;  // key row (S^T, dP^T, dV, dK) and query row (dQ share)

  if (tid == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    mbar_arrive_expect_tx(kv_bar, 2 * C::kTileBytes);
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c) {
      tma_load_3d(sk + c * kChunkBytes, &tm_k, kv_bar, c * 64, kv0, bh);
      tma_load_3d(sv + c * kChunkBytes, &tm_v, kv_bar, c * 64, kv0, bh);
    }
  }
  bool ok = bounded_wait(kv_bar, 0, abort_flag, p.err, kSiteKvFull);
  uint32_t mma_phase = 0;
  int qdo_issued = 0;  // Q/dO tile pairs requested by thread 0
  const size_t head_rows = static_cast<size_t>(bh) * p.N;

  for (int i = i_first; i < num_q_tiles && ok; ++i) {
    const int q0 = i * 128;
    const int it = i - i_first;
    // (a) Q_i and dO_i by TMA; the row statistics by plain loads
    if (tid == 0) {
      mbar_arrive_expect_tx(qdo_bar, 2 * C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(sq + c * kChunkBytes, &tm_q, qdo_bar, c * 64, q0, bh);
        tma_load_3d(sdo + c * kChunkBytes, &tm_do, qdo_bar, c * 64, q0, bh);
      }
      ++qdo_issued;
    }
    {
      const int qr = q0 + tid;
      // rows beyond N: L = +inf makes P = 0 there, and D = 0
      lse2[tid] = (qr < p.N) ? p.lse[head_rows + qr] * kLog2e : INFINITY;
      dlt[tid] = (qr < p.N) ? p.delta[head_rows + qr] : 0.f;
    }
    __syncthreads();
    ok = bounded_wait(qdo_bar, it & 1, abort_flag, p.err, kSiteQFull);
    ok = __all_sync(kFull, ok) && ok;
    if (!__syncthreads_and(ok)) break;

    // (b) S^T = K Q^T and dP^T = V dO^T
    if (tid == 0) {
      tc_fence_after();
      issue_qk<D>(tmem + C::kColS, smem_u32(sk), smem_u32(sq));
      issue_qk<D>(tmem + C::kColDp, smem_u32(sv), smem_u32(sdo));
      umma_commit(mma_bar);
    }
    __syncwarp();
    ok = bounded_wait(mma_bar, mma_phase & 1, abort_flag, p.err, kSiteSFull);
    ++mma_phase;
    ok = __all_sync(kFull, ok);
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();

    // (c) P^T and dS^T for key row `row`, 32 queries at a time
    const int key = kv0 + row;
    const bool key_ok = key < p.N;
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t s[32], dp[32];
      tmem_ld_x32(tmem + lane_base + C::kColS + 32 * ch, s);
      tmem_ld_x32(tmem + lane_base + C::kColDp + 32 * ch, dp);
      uint32_t pw[16], dw[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float pv[2], dv[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = 32 * ch + 2 * e + h;
          const int q = q0 + c;
          float pr = ex2_approx(fmaf(__uint_as_float(s[2 * e + h]), p.scale_log2, -lse2[c]));
          if (!key_ok || (p.causal && key > q)) pr = 0.f;
          pv[h] = pr;
          dv[h] = pr * (__uint_as_float(dp[2 * e + h]) - dlt[c]);
        }
        pw[e] = pack_bf16x2(pv[0], pv[1]);
        dw[e] = pack_bf16x2(dv[0], dv[1]);
      }
      // P^T and dS^T pairs overwrite score columns this thread has already read
      tmem_st_x16(tmem + lane_base + C::kColS + 16 * ch, pw);
      tmem_st_x16(tmem + lane_base + C::kColDp + 16 * ch, dw);
      // dS^T row `row`, queries [32ch, 32ch + 32): four 16-byte units of the
      // 128-byte row of chunk (ch / 2), swizzled by the row index
      uint8_t* rowp = sds + (ch >> 1) * kChunkBytes + row * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int unit = (ch & 1) * 4 + u;
        *reinterpret_cast<uint4*>(rowp + ((unit ^ (row & 7)) << 4)) =
            make_uint4(dw[4 * u], dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
      }
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // (d) dV += P^T dO, dK += dS^T Q, dQ share = dS K
    if (tid == 0) {
      tc_fence_after();
      issue_pv<D>(tmem + C::kColDv, tmem + C::kColS, smem_u32(sdo), it > 0);
      issue_pv<D>(tmem + C::kColDk, tmem + C::kColDp, smem_u32(sq), it > 0);
      issue_mn_mn<D>(tmem + C::kColS, smem_u32(sds), smem_u32(sk));
      umma_commit(mma_bar);
    }
    __syncwarp();
    ok = bounded_wait(mma_bar, mma_phase & 1, abort_flag, p.err, kSitePFull);
    ++mma_phase;
    ok = __all_sync(kFull, ok);
    if (!__syncthreads_and(ok)) break;
    tc_fence_after();

    // (e) add scale * (dS K) for query row `row` into dQ
    {
      const int q = q0 + row;
      float* dst = p.dq_acc + (head_rows + (q < p.N ? q : 0)) * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld_x32(tmem + lane_base + C::kColS + c, r);
        if (q < p.N) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            red_add_v4(dst + c + 4 * e, __uint_as_float(r[4 * e]) * p.scale, __uint_as_float(r[4 * e + 1]) * p.scale,
                       __uint_as_float(r[4 * e + 2]) * p.scale, __uint_as_float(r[4 * e + 3]) * p.scale);
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // the next S^T overwrites these columns
  }

  // dK = scale * acc and dV = acc for key row `row`, written once
  if (ok && i_first < num_q_tiles) {
    tc_fence_after();
    const int key = kv0 + row;
    const size_t out = (head_rows + (key < p.N ? key : 0)) * D;
#pragma unroll 1
    for (int c = 0; c < D; c += 32) {
      uint32_t a[32], b[32];
      tmem_ld_x32(tmem + lane_base + C::kColDk + c, a);
      tmem_ld_x32(tmem + lane_base + C::kColDv + c, b);
      if (key < p.N) {
        uint32_t wk[16], wv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          wk[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
          wv[e] = pack_bf16x2(__uint_as_float(b[2 * e]), __uint_as_float(b[2 * e + 1]));
        }
        uint4* pk = reinterpret_cast<uint4*>(p.dk + out + c);
        uint4* pv = reinterpret_cast<uint4*>(p.dv + out + c);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pk[e] = make_uint4(wk[4 * e], wk[4 * e + 1], wk[4 * e + 2], wk[4 * e + 3]);
          pv[e] = make_uint4(wv[4 * e], wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
        }
      }
    }
  } else if (ok) {
    // no Q tile sees this K/V tile (cannot happen for N >= 1, kept for safety): zero gradients
    const int key = kv0 + row;
    if (key < p.N) {
      uint4* pk = reinterpret_cast<uint4*>(p.dk + (head_rows + key) * D);
      uint4* pv = reinterpret_cast<uint4*>(p.dv + (head_rows + key) * D);
      for (int e = 0; e < D / 8; ++e) pk[e] = pv[e] = make_uint4(0, 0, 0, 0);
    }
  }
  // teardown: every copy must have landed and every product completed before
  // the CTA exits and TMEM is freed
  if (tid == 0) {
    bounded_wait(kv_bar, 0, nullptr, p.err, kSiteDrain);
    if (qdo_issued > 0) bounded_wait(qdo_bar, (qdo_issued - 1) & 1, nullptr, p.err, kSiteDrain);
    umma_commit(mma_bar);
    bounded_wait(mma_bar, mma_phase & 1, nullptr, p.err, kSiteDrain);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
fa_status launch(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int H, int N, int causal, float scale, float* dq_acc,
                 float* delta, cudaStream_t stream, unsigned int* err) {
  using C = BwdCfg<D>;
  const uint64_t bh = static_cast<uint64_t>(B) * H;
  const long long rows = static_cast<long long>(bh) * N;
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, static_cast<size_t>(rows) * D * sizeof(float), stream);
  if (e != cudaSuccess) {
    set_error_text("cudaMemsetAsync(dQ accumulator)", e);
    return FA_ERR_CUDA;
  }
  bwd_delta_kernel<D><<<static_cast<unsigned>((rows + 255) / 256), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), delta, rows);
  CUtensorMap tq, tk, tv, tdo;
  if (!encode_bf16_map(&tq, q, D, N, bh, 128) || !encode_bf16_map(&tk, k, D, N, bh, 128) ||
      !encode_bf16_map(&tv, v, D, N, bh, 128) || !encode_bf16_map(&tdo, dout, D, N, bh, 128))
    return FA_ERR_CUDA;
  BwdParams prm;
  prm.lse = lse;
  prm.delta = delta;
  prm.dq_acc = dq_acc;
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  prm.err = err;
  prm.N = N;
  prm.num_kv_tiles = (N + 127) / 128;
  prm.causal = causal ? 1 : 0;
  prm.scale = scale;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  e = cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) {
    set_error_text("cudaFuncSetAttribute(bwd_kernel)", e);
    return FA_ERR_CUDA;
  }
  dim3 grid(static_cast<unsigned>(bh), static_cast<unsigned>(prm.num_kv_tiles));
  bwd_kernel<D><<<grid, kBwdThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, prm);
  const long long n4 = rows * D / 4;
  bwd_dq_convert_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, stream>>>(
      dq_acc, static_cast<__nv_bfloat16*>(dq), n4);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("backward kernels launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

fa_status launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, float* dq_acc,
                     float* delta, cudaStream_t stream, unsigned int* err) {
  if (d == 128)
    return launch<128>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, causal, scale, dq_acc, delta, stream, err);
  if (d == 64)
    return launch<64>(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, causal, scale, dq_acc, delta, stream, err);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
