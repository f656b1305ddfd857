// Fused prefill attention for sm_103a: tcgen05 tensor cores with TMEM
// accumulators, TMA-fed shared-memory pipeline, warp-specialised roles.
//
// What is computed (per (batch, head), FlashAttention-2 order):
//   "已有的几种大模型上下文支持情况" (cicada blog) §3.2 and CMU 15-779
//   Lecture 5 notes §5.1: each Q tile stays on chip while K/V tiles stream
//   through; S_ij = Q_i K_j^T; running max m and normaliser l with the
//   rescale factor exp(m_old - m_new); the un-normalised P~ V accumulates;
//   one divide by l at the end; L_i = m_i + ln l_i is written out.
//   Causal mode skips K/V tiles entirely above the diagonal and masks only
//   the diagonal tile (Lecture 5 notes §6.2). Rescaling is conditional
//   (cicada blog §5, FlashAttention-4: only when the maximum grows by more
//   than a slack tau); the result stays exact because l and the output
//   share the same stale base and the final O / l and L use it consistently.
//
// Mapping onto one CTA (one SM; TMEM holds 512 columns x 128 lanes):
//   * two Q tiles of 128 rows each (256 query rows of one head);
//   * warps 0-3: softmax of Q tile 0, warps 4-7: softmax of Q tile 1
//     (thread r of a warpgroup owns row r; a row's max and sum are in-thread);
//   * warp 8: one thread issues every tcgen05.mma and commit;
//   * warp 9: one thread issues every TMA copy (Q once, then K_j, V_j into a
//     ring of shared-memory slots).
//   TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
//   P (bf16 pairs) overwrites the first 64 columns of its S tile and is the
//   TMEM A operand of O += P V. While warpgroup 0 runs the softmax of S0 the
//   tensor core works on tile 1's products, and the other way round.
//
// Every wait is bounded (fa_common.cuh); a wait that runs out records the
// site, raises the CTA abort flag, and every role drains its in-flight copies
// or products before TMEM is freed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "fa_common.cuh"
#include "fa_internal.h"
#include "fa_mma.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;       // 8 softmax warps + MMA warp + load warp
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr float kRescaleSlack = 8.0f;  // log2 units: rescale only when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kFull = 0xffffffffu;

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kBN * D * 2;  // one Q, K or V tile
  static constexpr int kChunks = D / 64;
  static constexpr int kStages = (D == 128) ? 4 : 8;  // K/V ring slots
  // TMEM column of S (and P) and of O for Q tile t
  __host__ __device__ static constexpr uint32_t s_col(int t) { return t ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t o_col(int t) { return t ? 256u + D : 256u; }
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
  static constexpr int kNumBars = 2 + 2 * kStages + 2 + 2 + 2 + 1;
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;  // + slack to align to 1 KB
};

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  unsigned int* err;
  int N;
  int num_pairs;
  int causal;
  float scale_log2;  // scale * log2(e)
};

struct Smem {
  uint8_t* q[2];
  uint8_t* ring;
  uint64_t* q_full;    // [2]   Q tile landed
  uint64_t* kv_full;   // [S]   K or V tile landed in a ring slot
  uint64_t* kv_empty;  // [S]   ring slot free again (committed by the MMA thread)
  uint64_t* s_full;    // [2]   S = Q K^T done (also: every earlier product of that tile done)
  uint64_t* p_full;    // [2]   P written to TMEM and O rescaled (128 arrivals)
  uint64_t* o_full;    // [2]   last O += P V done
  uint64_t* mma_done;  // [1]   every product done (teardown)
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

template <int D>
__device__ __forceinline__ Smem carve(uint8_t* raw) {
  using C = Cfg<D>;
  const uint32_t a = smem_u32(raw);
  uint8_t* base = raw + ((1024u - (a & 1023u)) & 1023u);
  Smem s;
  s.q[0] = base;
  s.q[1] = base + C::kTileBytes;
  s.ring = base + C::kRingOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  s.q_full = bars;
  s.kv_full = bars + 2;
  s.kv_empty = s.kv_full + C::kStages;
  s.s_full = s.kv_empty + C::kStages;
  s.p_full = s.s_full + 2;
  s.o_full = s.p_full + 2;
  s.mma_done = s.o_full + 2;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.mma_done + 1);
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  return s;
}

// ---------------------------------------------------------------- TMA producer (one thread)
template <int D>
__device__ void load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v, const Smem& sm,
                          unsigned int* err, int bh, int q0, const int (&n_kv)[2], int n_max) {
  using C = Cfg<D>;
  tma_prefetch_desc(tm_q);
  tma_prefetch_desc(tm_k);
  tma_prefetch_desc(tm_v);
  for (int t = 0; t < 2; ++t) {
    if (n_kv[t] == 0) continue;
    mbar_arrive_expect_tx(&sm.q_full[t], C::kTileBytes);
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c)
      tma_load_3d(sm.q[t] + c * kChunkBytes, tm_q, &sm.q_full[t], c * 64, q0 + t * kBM, bh);
  }
  int item = 0;  // K_j is item 2j, V_j is item 2j+1
  bool ok = true;
  for (int j = 0; j < n_max && ok; ++j) {
    for (int kind = 0; kind < 2; ++kind) {
      const int slot = item % C::kStages;
      const int use = item / C::kStages;
      if (use > 0) {
        ok = bounded_wait(&sm.kv_empty[slot], (use - 1) & 1, sm.abort_flag, err, kSiteKvEmpty);
        if (!ok) break;
      }
      uint8_t* dst = sm.ring + slot * C::kTileBytes;
      mbar_arrive_expect_tx(&sm.kv_full[slot], C::kTileBytes);
      const CUtensorMap* map = kind ? tm_v : tm_k;
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(dst + c * kChunkBytes, map, &sm.kv_full[slot], c * 64, j * kBN, bh);
      ++item;
    }
  }
  // Drain: every copy issued must land before the CTA can exit.
  for (int it = (item > C::kStages ? item - C::kStages : 0); it < item; ++it)
    bounded_wait(&sm.kv_full[it % C::kStages], (it / C::kStages) & 1, nullptr, err, kSiteDrain);
  for (int t = 0; t < 2; ++t)
    if (n_kv[t] > 0) bounded_wait(&sm.q_full[t], 0, nullptr, err, kSiteDrain);
}

// ---------------------------------------------------------------- MMA issuer (one thread)
template <int D>
__device__ void mma_role(const Smem& sm, uint32_t tmem, unsigned int* err, const int (&n_kv)[2], int n_max) {
  using C = Cfg<D>;
  const uint32_t ring = smem_u32(sm.ring);
  const uint32_t qa[2] = {smem_u32(sm.q[0]), smem_u32(sm.q[1])};
  auto slot_addr = [&](int item) { return ring + static_cast<uint32_t>((item % C::kStages) * C::kTileBytes); };
  auto wait_item = [&](int item) {
    return bounded_wait(&sm.kv_full[item % C::kStages], (item / C::kStages) & 1, sm.abort_flag, err, kSiteKvFull);
  };

  bool ok = true;
  for (int t = 0; t < 2 && ok; ++t)
    if (n_kv[t] > 0) ok = bounded_wait(&sm.q_full[t], 0, sm.abort_flag, err, kSiteQFull);
  if (ok) ok = wait_item(0);
  if (ok) {
    tc_fence_after();
    for (int t = 0; t < 2; ++t) {
      if (n_kv[t] == 0) continue;
      issue_qk<D>(tmem + C::s_col(t), qa[t], slot_addr(0));
      umma_commit(&sm.s_full[t]);
    }
    umma_commit(&sm.kv_empty[0]);
  }
  for (int j = 0; j < n_max && ok; ++j) {
    const int iv = 2 * j + 1;  // V_j
    const int ik = 2 * j + 2;  // K_{j+1}
    ok = wait_item(iv);
    if (!ok) break;
    bool k_next = false;
    for (int t = 0; t < 2; ++t) {
      if (j >= n_kv[t]) continue;
      ok = bounded_wait(&sm.p_full[t], j & 1, sm.abort_flag, err, kSitePFull);
      if (!ok) break;
      tc_fence_after();
      issue_pv<D>(tmem + C::o_col(t), tmem + C::s_col(t), slot_addr(iv), j > 0);
      if (j + 1 < n_kv[t]) {
        if (!k_next) {
          ok = wait_item(ik);
          if (!ok) break;
          tc_fence_after();
          k_next = true;
        }
        // issued after P V of the same tile: the tensor pipe runs them in order,
        // so P is read before the new S overwrites those columns
        issue_qk<D>(tmem + C::s_col(t), qa[t], slot_addr(ik));
        umma_commit(&sm.s_full[t]);
      } else {
        umma_commit(&sm.o_full[t]);
      }
    }
    if (!ok) break;
    umma_commit(&sm.kv_empty[iv % C::kStages]);
    if (k_next) umma_commit(&sm.kv_empty[ik % C::kStages]);
  }
  // Teardown: every product issued so far must finish before TMEM is freed.
  umma_commit(sm.mma_done);
  bounded_wait(sm.mma_done, 0, nullptr, err, kSiteDrain);
}

// ---------------------------------------------------------------- softmax + epilogue (128 threads per tile)
template <int D>
__device__ void softmax_role(const Smem& sm, uint32_t tmem, const FwdParams& p, int warp, int lane, int bh, int q0,
                             const int (&n_kv)[2]) {
  using C = Cfg<D>;
  const int t = warp >> 2;
  const int quarter = warp & 3;  // this warp may touch TMEM lanes [32*quarter, 32*quarter+32)
  const int row = quarter * 32 + lane;
  const int q_row = q0 + t * kBM + row;
  const int nkv = n_kv[t];
  if (nkv == 0) return;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t s_tm = tmem + lane_base + C::s_col(t);
  const uint32_t o_tm = tmem + lane_base + C::o_col(t);
  const float sl2 = p.scale_log2;
  const int vis_end = p.causal ? min(q_row + 1, p.N) : p.N;  // keys [0, vis_end) are visible to this row

  float m_used = -INFINITY;  // base of every exponent so far (log2 domain, scaled)
  float l = 0.f;
  bool ok = true;
  for (int j = 0; j < nkv; ++j) {
    ok = bounded_wait(&sm.s_full[t], j & 1, sm.abort_flag, p.err, kSiteSFull);
    ok = __all_sync(kFull, ok);
    if (!ok) break;
    tc_fence_after();

    uint32_t ra[64], rb[64];
    tmem_ld_x64(s_tm, ra);
    tmem_ld_x64(s_tm + 64, rb);
    float s[128];
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      s[c] = __uint_as_float(ra[c]);
      s[64 + c] = __uint_as_float(rb[c]);
    }
    const int lim = vis_end - j * kBN;  // visible keys of this tile for this row
    if (lim < kBN) {
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c >= lim) s[c] = -INFINITY;
    }
    float mx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
    for (int c = 8; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], s[c]);
    const float m_tile = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;

    const bool need = (m_used != -INFINITY) && (m_tile > m_used + kRescaleSlack);
    if (__any_sync(kFull, need)) {
      const float alpha = need ? ex2_approx(m_used - m_tile) : 1.f;
      if (need) {
        l *= alpha;
        m_used = m_tile;
      }
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld_x32(o_tm + c, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st_x32(o_tm + c, r);
      }
    }
    if (m_used == -INFINITY) m_used = m_tile;  // first visible scores of this row
    const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;

    uint32_t pk[64];
    float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float p0 = ex2_approx(fmaf(s[2 * i], sl2, -m_sub));
      const float p1 = ex2_approx(fmaf(s[2 * i + 1], sl2, -m_sub));
      sum[i & 3] += p0 + p1;
      pk[i] = pack_bf16x2(p0, p1);
    }
    l += (sum[0] + sum[1]) + (sum[2] + sum[3]);
    tmem_st_x64(s_tm, pk);
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&sm.p_full[t]);
  }
  if (ok) {
    ok = bounded_wait(&sm.o_full[t], 0, sm.abort_flag, p.err, kSiteOFull);
    ok = __all_sync(kFull, ok);
  }
  if (!ok) return;
  tc_fence_after();

  const float inv_l = 1.f / l;
  const bool in_range = q_row < p.N;
  __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.N + (in_range ? q_row : 0)) * D;
#pragma unroll 1
  for (int c = 0; c < D; c += 32) {
    uint32_t r[32];
    tmem_ld_x32(o_tm + c, r);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
    if (in_range) {
      uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
  if (in_range) p.lse[static_cast<size_t>(bh) * p.N + q_row] = (m_used + log2f(l)) * kLn2;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve<D>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  // causal: launch the heaviest Q-tile pairs (largest row index) first
  const int pair = p.causal ? (p.num_pairs - 1 - static_cast<int>(blockIdx.y)) : static_cast<int>(blockIdx.y);
  const int q0 = pair * 2 * kBM;
  const int n_kv[2] = {fwd_kv_tiles(q0, p.N, kBN, p.causal), fwd_kv_tiles(q0 + kBM, p.N, kBN, p.causal)};
  const int n_max = max(n_kv[0], n_kv[1]);

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.q_full[t], 1);
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_full[t], 128);
      mbar_init(&sm.o_full[t], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    mbar_init(sm.mma_done, 1);
    *sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sm.tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot;

  if (warp == kLoadWarp) {
    if (lane == 0) load_role<D>(&tm_q, &tm_k, &tm_v, sm, p.err, bh, q0, n_kv, n_max);
  } else if (warp == kMmaWarp) {
    if (lane == 0) mma_role<D>(sm, tmem, p.err, n_kv, n_max);
  } else {
    softmax_role<D>(sm, tmem, p, warp, lane, bh, q0, n_kv);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
fa_status launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int causal,
                 float scale, cudaStream_t stream, unsigned int* err) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv;
  const uint64_t bh = static_cast<uint64_t>(B) * H;
  if (!encode_bf16_map(&tq, q, D, N, bh, kBM) || !encode_bf16_map(&tk, k, D, N, bh, kBN) ||
      !encode_bf16_map(&tv, v, D, N, bh, kBN))
    return FA_ERR_CUDA;
  const int num_pairs = (N + 2 * kBM - 1) / (2 * kBM);
  FwdParams prm;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.err = err;
  prm.N = N;
  prm.num_pairs = num_pairs;
  prm.causal = causal ? 1 : 0;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) {
    set_error_text("cudaFuncSetAttribute(fwd_kernel)", e);
    return FA_ERR_CUDA;
  }
  dim3 grid(static_cast<unsigned>(bh), static_cast<unsigned>(num_pairs));
  fwd_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("fwd_kernel launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

fa_status launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                     int causal, float scale, cudaStream_t stream, unsigned int* err) {
  if (d == 128) return launch<128>(q, k, v, o, lse, B, H, N, causal, scale, stream, err);
  if (d == 64) return launch<64>(q, k, v, o, lse, B, H, N, causal, scale, stream, err);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
