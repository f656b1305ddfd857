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
// One CTA owns one K/V tile (128 keys) of one head and walks the Q tiles that
// see it. Everything is computed transposed, keys on the 128 TMEM lanes:
//   TMEM columns [0,128)    S^T = K Q^T, then P^T as bf16 pairs
//            [128,256)  dP^T = V dO^T, then dS^T as bf16 pairs, then the
//                       dQ share dS K (lanes = queries, D columns)
//            [256,256+D) dV,  [384,384+D) dK  (fp32 accumulators)
// Warp roles (14 warps):
//   warp 12     TMA: K and V once; Q (two buffers) and dO (one buffer) per Q
//               tile, plus that tile's row statistics (L log2 e, D) into shared
//               memory.
//   warp 13     one thread issues every tensor-core product, in the order
//                 dV_i, S_{i+1}, dK_i, dQ_i, dP_{i+1}
//               so that S of the next tile runs while P/dS warps finish dS_i,
//               and dP_{i+1} waits only for the read-out of dQ_i.
//   warps 4-11  P and dS: warp w takes key rows 32(w%4).. and query columns
//               64((w-4)/4)..; P = exp2(S log2e scale - L log2e) rounded to bf16
//               pairs, to TMEM (for dV) and kept in registers, then
//               dS = P (dP - D) from those bf16 P values to TMEM (for dK) and,
//               transposed, to shared memory (for dQ = dS K, whose A operand
//               must be query-major).
//   warps 0-3   read the dQ share out of TMEM and add scale * dQ to the fp32
//               accumulator (the atomic additions of §7.4). d = 128: the share
//               is dQ^T (d on the lanes); each warp loads three 32-column
//               slices, adds the first with coalesced red.global.add (one
//               128-byte segment of a dQ row per instruction), loads the fourth
//               and returns the columns to the next dP before adding the rest.
//               d = 64: the share is dQ; it is staged in shared memory and added
//               with bulk tensor reductions on whole 128-byte rows.
// Every wait is bounded (fa_common.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "fa_common.cuh"
#include "fa_internal.h"
#include "fa_mma.cuh"

namespace fa {
namespace {

constexpr int kLoadWarp = 12;
constexpr int kMmaWarp = 13;
// 14 warps: each SM sub-partition holds at most four of them, so a thread can
// have 16,384 / (4 x 32) = 128 registers.
constexpr int kBwdThreads = 14 * 32;
constexpr uint32_t kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;  // a K, V, Q or dO tile
  static constexpr int kChunks = D / 64;
  static constexpr int kDsBytes = 128 * 128 * 2;  // dS^T, 128 keys x 128 queries
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;  // two buffers
  static constexpr int kDoOff = 4 * kTileBytes;
  static constexpr int kDsOff = 5 * kTileBytes;
  static constexpr int kBoxBytes = 128 * 32 * 4;  // d = 64 dQ staging: 128 rows x 32 fp32 (4 warps' boxes)
  static constexpr int kVecOff = kDsOff + kDsBytes;  // [2][128] L log2 e, then [2][128] D
  static constexpr int kBarOff = kVecOff + 4 * 128 * 4;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
  static constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 384;
};

// barrier slots
enum BwdBar : int {
  kBarKv = 0,
  kBarQFull = 1,   // +buffer
  kBarQEmpty = 3,  // +buffer
  kBarDoFull = 5,
  kBarDoEmpty = 6,
  kBarVec = 7,  // +buffer
  kBarS = 9,
  kBarDp = 10,
  kBarP = 11,
  kBarDs = 12,
  kBarDq = 13,
  kBarDqEmpty = 14,
  kBarAcc = 15,
  kBarStageFree = 16,  // the read-out's reductions have read the dS^T buffer
  kNumBars = 17,
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

// Before the main kernel, in one pass over the rows: D_i = sum_c dO_ic O_ic in
// fp32, and the row's fp32 dQ accumulator set to zero. D / 8 lanes share a row
// (16 bytes of O and of dO each), so a warp's loads and stores cover whole
// consecutive rows; the row sum is finished with shuffles.
constexpr int kPrepThreads = 256;

template <int D>
__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                                const __nv_bfloat16* __restrict__ dout,
                                                                float* __restrict__ delta, float* __restrict__ dq_acc,
                                                                long long rows) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = static_cast<int>(threadIdx.x & 31);
  const long long warp = (static_cast<long long>(blockIdx.x) * kPrepThreads + threadIdx.x) >> 5;
  const long long warps = (static_cast<long long>(gridDim.x) * kPrepThreads) >> 5;
  for (long long r0 = warp * kRowsPerWarp; r0 < rows; r0 += warps * kRowsPerWarp) {
    const long long row = r0 + lane / kLanesPerRow;
    const int c = lane % kLanesPerRow;
    float acc = 0.f;
    if (row < rows) {
      const uint4 a = reinterpret_cast<const uint4*>(o + row * D)[c];
      const uint4 b = reinterpret_cast<const uint4*>(dout + row * D)[c];
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(__uint_as_float(wa[e] << 16), __uint_as_float(wb[e] << 16), acc);
        acc = fmaf(__uint_as_float(wa[e] & 0xffff0000u), __uint_as_float(wb[e] & 0xffff0000u), acc);
      }
    }
#pragma unroll
    for (int w = kLanesPerRow / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (row < rows && c == 0) delta[row] = acc;
    // the accumulator rows r0 .. r0 + kRowsPerWarp - 1: D floats each, D / 4 float4
    float4* z = reinterpret_cast<float4*>(dq_acc + r0 * D);
    const long long n4 = (rows - r0 < kRowsPerWarp ? rows - r0 : kRowsPerWarp) * (D / 4);
    for (long long i = lane; i < n4; i += 32) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
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

__device__ __forceinline__ void red_add_f32(float* addr, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sk = base + C::kKOff;
  uint8_t* sv = base + C::kVOff;
  uint8_t* sq = base + C::kQOff;
  uint8_t* sdo = base + C::kDoOff;
  uint8_t* sds = base + C::kDsOff;
  float* vec_l = reinterpret_cast<float*>(base + C::kVecOff);  // [2][128]
  float* vec_d = vec_l + 256;                                  // [2][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[kNumBars]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&bars[kNumBars + 1]);
  // [4] Q tiles completed by the load, MMA, P/dS and read-out roles (FA_DEBUG builds)
  uint32_t* dbg = reinterpret_cast<uint32_t*>(&bars[kNumBars + 2]);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // grid (heads, K/V tiles): blocks start in order of K/V tile, and under the
  // causal mask tile 0 (seen by every Q tile) is the heaviest
  const int bh = blockIdx.x;
  const int j = blockIdx.y;
  const int kv0 = j * 128;
  const int num_q_tiles = (p.N + 127) / 128;
  const int i_first = p.causal ? j : 0;  // first Q tile whose rows see a key of this tile
  const int n_it = num_q_tiles - i_first;  // >= 1 since j < num_q_tiles
  const size_t head_rows = static_cast<size_t>(bh) * p.N;

  if (tid == 0) {
    mbar_init(&bars[kBarKv], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kBarQFull + b], 1);
      mbar_init(&bars[kBarQEmpty + b], 1);
      mbar_init(&bars[kBarVec + b], 32);
    }
    mbar_init(&bars[kBarDoFull], 1);
    mbar_init(&bars[kBarDoEmpty], 1);
    mbar_init(&bars[kBarS], 1);
    mbar_init(&bars[kBarDp], 1);
    mbar_init(&bars[kBarP], 8);
    mbar_init(&bars[kBarDs], 8);
    mbar_init(&bars[kBarDq], 1);
    mbar_init(&bars[kBarDqEmpty], 4);
    mbar_init(&bars[kBarAcc], 1);
    mbar_init(&bars[kBarStageFree], 4);
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) dbg[i] = 0;
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

  if (warp == kLoadWarp) {
    // ---------------------------------------------------------------- loads
    int q_cnt0 = 0, q_cnt1 = 0, do_cnt = 0;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(&bars[kBarKv], 2 * C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(sk + c * kChunkBytes, &tm_k, &bars[kBarKv], c * 64, kv0, bh);
        tma_load_3d(sv + c * kChunkBytes, &tm_v, &bars[kBarKv], c * 64, kv0, bh);
      }
    }
    bool ok = true;
    int it = 0;
    for (; it < n_it && ok; ++it) {
      const int b = it & 1;
      const int q0 = (i_first + it) * 128;
      if (it >= 2) ok = bounded_wait(&bars[kBarQEmpty + b], ((it - 2) >> 1) & 1, abort_flag, p.err, kSiteQEmpty);
      if (!__all_sync(kFull, ok)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[kBarQFull + b], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sq + b * C::kTileBytes + c * kChunkBytes, &tm_q, &bars[kBarQFull + b], c * 64, q0, bh);
        if (b == 0)
          ++q_cnt0;
        else
          ++q_cnt1;
      }
      // row statistics of this Q tile; rows beyond N get L = +inf (P = 0) and D = 0
#pragma unroll
      for (int r = lane; r < 128; r += 32) {
        const int qr = q0 + r;
        vec_l[b * 128 + r] = (qr < p.N) ? p.lse[head_rows + qr] * kLog2e : INFINITY;
        vec_d[b * 128 + r] = (qr < p.N) ? p.delta[head_rows + qr] : 0.f;
      }
      mbar_arrive(&bars[kBarVec + b]);
      if (it >= 1) ok = bounded_wait(&bars[kBarDoEmpty], (it - 1) & 1, abort_flag, p.err, kSiteOEmpty);
      if (!__all_sync(kFull, ok)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[kBarDoFull], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sdo + c * kChunkBytes, &tm_do, &bars[kBarDoFull], c * 64, q0, bh);
        ++do_cnt;
      }
    }
#ifdef FA_DEBUG
    if (lane == 0) dbg[0] = static_cast<uint32_t>(it);
#endif
    // every copy issued must land before the CTA exits
    if (lane == 0) {
      bounded_wait(&bars[kBarKv], 0, nullptr, p.err, kSiteDrain);
      if (q_cnt0 > 0) bounded_wait(&bars[kBarQFull], (q_cnt0 - 1) & 1, nullptr, p.err, kSiteDrain);
      if (q_cnt1 > 0) bounded_wait(&bars[kBarQFull + 1], (q_cnt1 - 1) & 1, nullptr, p.err, kSiteDrain);
      if (do_cnt > 0) bounded_wait(&bars[kBarDoFull], (do_cnt - 1) & 1, nullptr, p.err, kSiteDrain);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- products
    if (lane == 0) {
      const uint32_t s_tm = tmem + C::kColS, dp_tm = tmem + C::kColDp;
      bool ok = bounded_wait(&bars[kBarKv], 0, abort_flag, p.err, kSiteKvFull) &&
                bounded_wait(&bars[kBarQFull], 0, abort_flag, p.err, kSiteQFull);
      if (ok) {
        tc_fence_after();
        issue_qk<D>(s_tm, smem_u32(sk), smem_u32(sq));
        umma_commit(&bars[kBarS]);
        ok = bounded_wait(&bars[kBarDoFull], 0, abort_flag, p.err, kSiteQFull);
      }
      if (ok) {
        tc_fence_after();
        issue_qk<D>(dp_tm, smem_u32(sv), smem_u32(sdo));
        umma_commit(&bars[kBarDp]);
      }
      int it = 0;
      for (; it < n_it && ok; ++it) {
        const int b = it & 1;
        const bool more = it + 1 < n_it;
        // dV += P^T dO as soon as P^T is in TMEM
        if (!(ok = bounded_wait(&bars[kBarP], it & 1, abort_flag, p.err, kSitePFull))) break;
        tc_fence_after();
        issue_pv<D>(tmem + C::kColDv, s_tm, smem_u32(sdo), it > 0, 32);
        umma_commit(&bars[kBarDoEmpty]);
        // S of the next Q tile overwrites P^T behind the dV product
        if (more) {
          if (!(ok = bounded_wait(&bars[kBarQFull + (b ^ 1)], ((it + 1) >> 1) & 1, abort_flag, p.err, kSiteQFull)))
            break;
          tc_fence_after();
          issue_qk<D>(s_tm, smem_u32(sk), smem_u32(sq + (b ^ 1) * C::kTileBytes));
          umma_commit(&bars[kBarS]);
        }
        // dK += dS^T Q, then the dQ share dS K into the dP columns
        if (!(ok = bounded_wait(&bars[kBarDs], it & 1, abort_flag, p.err, kSitePFull))) break;
        tc_fence_after();
        issue_pv<D>(tmem + C::kColDk, dp_tm, smem_u32(sq + b * C::kTileBytes), it > 0, 32);
        umma_commit(&bars[kBarQEmpty + b]);
        if constexpr (D == 128) {
          // dQ^T = K^T dS^T: d on the TMEM lanes, so that each read-out warp
          // instruction adds one whole 128-byte segment of a dQ row
          issue_mn_mn<128>(dp_tm, smem_u32(sk), smem_u32(sds));
        } else {
          issue_mn_mn<D>(dp_tm, smem_u32(sds), smem_u32(sk));
        }
        umma_commit(&bars[kBarDq]);
        // dP of the next tile once the dQ share has been read out
        if (more) {
          if (!(ok = bounded_wait(&bars[kBarDqEmpty], it & 1, abort_flag, p.err, kSiteOEmpty))) break;
          if (!(ok = bounded_wait(&bars[kBarDoFull], (it + 1) & 1, abort_flag, p.err, kSiteQFull))) break;
          tc_fence_after();
          issue_qk<D>(dp_tm, smem_u32(sv), smem_u32(sdo));
          umma_commit(&bars[kBarDp]);
        }
      }
#ifdef FA_DEBUG
      dbg[1] = static_cast<uint32_t>(it);
#endif
      // completes once every product above has; the epilogue reads dK and dV after it
      umma_commit(&bars[kBarAcc]);
      bounded_wait(&bars[kBarAcc], 0, nullptr, p.err, kSiteDrain);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- P and dS
    const int quad = warp & 3, half = (warp - 4) >> 2;
    const int row = quad * 32 + lane;  // key row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int key = kv0 + row;
    const bool key_ok = key < p.N;
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint32_t s_tm = tmem + lane_base + C::kColS + 64 * half;
    const uint32_t dp_tm = tmem + lane_base + C::kColDp + 64 * half;
    uint8_t* ds_row = sds + half * kChunkBytes + row * 128;
    bool ok = true;
    int it = 0;
    for (; it < n_it; ++it) {
      const int b = it & 1;
      const int i = i_first + it;
      ok = bounded_wait(&bars[kBarS], it & 1, abort_flag, p.err, kSiteSFull) &&
           bounded_wait(&bars[kBarVec + b], (it >> 1) & 1, abort_flag, p.err, kSiteQFull);
      if (!__all_sync(kFull, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P^T for this row and 64 queries, 32 at a time, as bf16 pairs: to TMEM for
      // dV, and kept for dS (32 registers)
      uint32_t pw[32];
      const float4* l4 = reinterpret_cast<const float4*>(vec_l + b * 128 + 64 * half);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t s[32];
        tmem_ld_x32(s_tm + 32 * h2, s);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l = l4[8 * h2 + e4];
          const uint64_t a = f2_fma(f2_pack(__uint_as_float(s[4 * e4]), __uint_as_float(s[4 * e4 + 1])), sc2,
                                    f2_pack(-l.x, -l.y));
          const uint64_t c = f2_fma(f2_pack(__uint_as_float(s[4 * e4 + 2]), __uint_as_float(s[4 * e4 + 3])), sc2,
                                    f2_pack(-l.z, -l.w));
          float x0, x1, x2, x3;
          f2_unpack(a, x0, x1);
          f2_unpack(c, x2, x3);
          const int e = 32 * h2 + 4 * e4;
          float p4[4] = {ex2_approx(x0), ex2_approx(x1), ex2_approx(x2), ex2_approx(x3)};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            // no key beyond N; on the diagonal tile query 64 half + e + u sees this key only if not earlier
            if (!key_ok || (p.causal && i == j && row > 64 * half + e + u)) p4[u] = 0.f;
          }
          pw[e / 2] = pack_bf16x2(p4[0], p4[1]);
          pw[e / 2 + 1] = pack_bf16x2(p4[2], p4[3]);
        }
      }
      tmem_st_x32(s_tm, pw);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarP]);

      // dS = P (dP - D)
      ok = bounded_wait(&bars[kBarDp], it & 1, abort_flag, p.err, kSiteSFull);
      if (!__all_sync(kFull, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the dS^T buffer held dQ boxes of the previous tile: their reads must be done
      if (D == 64 && it > 0) {
        ok = bounded_wait(&bars[kBarStageFree], (it - 1) & 1, abort_flag, p.err, kSiteOEmpty);
        if (!__all_sync(kFull, ok)) {
          ok = false;
          break;
        }
      }
      const float4* d4 = reinterpret_cast<const float4*>(vec_d + b * 128 + 64 * half);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dp[32];
        tmem_ld_x32(dp_tm + 32 * c, dp);
        uint32_t dw[16];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 dl = d4[8 * c + e4];
          const int e = 32 * c + 4 * e4;
          const uint32_t p01 = pw[e / 2], p23 = pw[e / 2 + 1];
          const uint64_t a = f2_mul(f2_pack(__uint_as_float(p01 << 16), __uint_as_float(p01 & 0xffff0000u)),
                                    f2_add(f2_pack(__uint_as_float(dp[4 * e4]), __uint_as_float(dp[4 * e4 + 1])),
                                           f2_pack(-dl.x, -dl.y)));
          const uint64_t q = f2_mul(f2_pack(__uint_as_float(p23 << 16), __uint_as_float(p23 & 0xffff0000u)),
                                    f2_add(f2_pack(__uint_as_float(dp[4 * e4 + 2]), __uint_as_float(dp[4 * e4 + 3])),
                                           f2_pack(-dl.z, -dl.w)));
          float x0, x1, x2, x3;
          f2_unpack(a, x0, x1);
          f2_unpack(q, x2, x3);
          dw[2 * e4] = pack_bf16x2(x0, x1);
          dw[2 * e4 + 1] = pack_bf16x2(x2, x3);
        }
        // dS^T pairs overwrite dP columns of this chunk that are already read
        tmem_st_x16(dp_tm + 16 * c, dw);
        // dS^T row `row`, queries 64 half + 32 c + [0, 32): 16-byte units
        // 4c..4c+3 of the 128-byte row, swizzled by the row index
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(ds_row + (((4 * c + u) ^ (row & 7)) << 4)) =
              make_uint4(dw[4 * u], dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarDs]);
    }
#ifdef FA_DEBUG
    if (warp == 4 && lane == 0) dbg[2] = static_cast<uint32_t>(it);
#endif
    // dK = scale * acc and dV = acc for this key row, columns of this half of d
    if (ok) ok = bounded_wait(&bars[kBarAcc], 0, abort_flag, p.err, kSiteOFull);
    if (__all_sync(kFull, ok)) {
      tc_fence_after();
      const size_t out = (head_rows + (key_ok ? key : 0)) * D;
#pragma unroll 1
      for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
        uint32_t a[32], v[32];
        tmem_ld_x32(tmem + lane_base + C::kColDk + c, a);
        tmem_ld_x32(tmem + lane_base + C::kColDv + c, v);
        if (key_ok) {
          uint32_t wk[16], wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            wk[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
            wv[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
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
    }
  } else {
    // ---------------------------------------------------------------- dQ read-out
    // d = 128: the share is dQ^T (lane = column d of dQ, TMEM column = query
    // row). Each warp instruction adds 32 consecutive floats (one 128-byte
    // segment) of one dQ row with a plain reduction; the TMEM columns are
    // released as soon as the last slice has been loaded.
    // d = 64: the share is dQ (lane = query row); warp w owns rows 32w.. and
    // stages its two 32-column slices (scaled) into 4 KB shared-memory boxes
    // in the tensor map's swizzled layout; lane 0 adds each box into the fp32
    // accumulator with a bulk tensor reduction (rows beyond N are clipped by
    // the map). The boxes lie in the two halves of the dS^T buffer, free once
    // the dQ product is complete and until the P/dS warps write the next dS^T,
    // which they do after kBarStageFree.
    const uint32_t dq_tm = tmem + (static_cast<uint32_t>(warp * 32) << 16) + C::kColDp;
    if constexpr (D == 128) {
      const int dcol = warp * 32 + lane;
      int it = 0;
      for (; it < n_it; ++it) {
        const bool ok = bounded_wait(&bars[kBarDq], it & 1, abort_flag, p.err, kSitePFull);
        if (!__all_sync(kFull, ok)) break;
        tc_fence_after();
        const int q0 = (i_first + it) * 128;
        const int nq = min(128, p.N - q0);
        float* dst = p.dq_acc + (head_rows + q0) * D + dcol;
        // 32 queries (TMEM columns c0 ..) of this dQ column: scaled reductions.
        // `paced`: a 20 ns pause after every second reduction. The reductions
        // that follow the release of the TMEM columns overlap the P/dS warps'
        // next dS phase, whose shared-memory stores of dS^T queue behind them
        // in the load/store path; spread over about a third of a Q-tile period
        // they leave it free (measured: +5 to +7 % on the Llama and 16k shapes;
        // 20 ns or more per reduction, or a pause after each one, loses ~20 %:
        // the read-out then holds up the next release).
        auto add32 = [&](const uint32_t (&r)[32], int c0, bool paced) {
          if (c0 + 32 <= nq) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              red_add_f32(dst + static_cast<size_t>(c0 + e) * D, __uint_as_float(r[e]) * p.scale);
              if (paced && (e & 1)) __nanosleep(20);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c0 + e < nq) red_add_f32(dst + static_cast<size_t>(c0 + e) * D, __uint_as_float(r[e]) * p.scale);
          }
        };
        // Three slices in registers, the first one added, the fourth loaded into
        // its registers: the TMEM columns go back to the next dP after 32
        // reductions instead of 96.
        uint32_t r0[32], r1[32], r2[32];
        tmem_ld_x32(dq_tm, r0);
        tmem_ld_x32(dq_tm + 32, r1);
        tmem_ld_x32(dq_tm + 64, r2);
        add32(r0, 0, false);
        tmem_ld_x32(dq_tm + 96, r0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarDqEmpty]);
        add32(r1, 32, true);
        add32(r2, 64, true);
        add32(r0, 96, true);
      }
#ifdef FA_DEBUG
      if (warp == 0 && lane == 0) dbg[3] = static_cast<uint32_t>(it);
#endif
    } else {
      static_assert(D == 64, "one 64-column pair");
      if (lane == 0 && warp == 0) tma_prefetch_desc(&tm_dq);
      int it = 0;
      for (; it < n_it; ++it) {
        const bool ok = bounded_wait(&bars[kBarDq], it & 1, abort_flag, p.err, kSitePFull);
        if (!__all_sync(kFull, ok)) break;
        tc_fence_after();
        const int q0 = (i_first + it) * 128;
        uint32_t r[64];
        tmem_ld_x64(dq_tm, r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarDqEmpty]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint8_t* rowp = sds + h * C::kBoxBytes + warp * 4096 + lane * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(rowp + ((u ^ (lane & 7)) << 4)) = make_float4(
                __uint_as_float(r[32 * h + 4 * u]) * p.scale, __uint_as_float(r[32 * h + 4 * u + 1]) * p.scale,
                __uint_as_float(r[32 * h + 4 * u + 2]) * p.scale, __uint_as_float(r[32 * h + 4 * u + 3]) * p.scale);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tm_dq, sds + h * C::kBoxBytes + warp * 4096, 32 * h, q0 + 32 * warp, bh);
            bulk_commit_group();
          }
        }
        if (lane == 0) {
          bulk_wait_group_read<0>();
          mbar_arrive(&bars[kBarStageFree]);
        }
        __syncwarp();
      }
      // the additions must be complete before the CTA exits
      if (lane == 0) bulk_wait_group<0>();
#ifdef FA_DEBUG
      if (warp == 0 && lane == 0) dbg[3] = static_cast<uint32_t>(it);
#endif
    }
  }

  tc_fence_before();
  __syncthreads();
#ifdef FA_DEBUG
  // protocol check: every role completed every Q tile of this K/V tile
  if (tid == 0 && *abort_flag == 0) {
    const uint32_t n = static_cast<uint32_t>(n_it);
    if (dbg[0] != n || dbg[1] != n || dbg[2] != n || dbg[3] != n) record_check(p.err, kSiteCheckBwd);
  }
#endif
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
  {
    // enough warps for every row group, at most a few waves of the GPU
    const long long groups = (rows + (32 / (D / 8)) - 1) / (32 / (D / 8));
    const long long blocks = (groups + kPrepThreads / 32 - 1) / (kPrepThreads / 32);
    const unsigned grid = static_cast<unsigned>(blocks < 152 * 16 ? blocks : 152 * 16);
    bwd_prep_kernel<D><<<grid, kPrepThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                          static_cast<const __nv_bfloat16*>(dout), delta, dq_acc,
                                                          rows);
  }
  cudaError_t e = cudaSuccess;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!encode_bf16_map(&tq, q, D, N, bh, 128) || !encode_bf16_map(&tk, k, D, N, bh, 128) ||
      !encode_bf16_map(&tv, v, D, N, bh, 128) || !encode_bf16_map(&tdo, dout, D, N, bh, 128) ||
      !encode_f32_map(&tdq, dq_acc, D, N, bh, 32))
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
  bwd_kernel<D><<<grid, kBwdThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, prm);
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
