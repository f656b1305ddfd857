// Flash-Decoding with grouped K/V heads (GQA; MQA when there is one K/V head)
// for sm_103a.
//
// CMU 15-779 Lecture 5 notes, Exercise 7: when g query heads share one K/V
// head, every K/V element read in a decode step serves g queries, so the
// arithmetic intensity rises from about 1 to about g FLOP per byte. The split
// along the keys and the log-sum-exp merge are those of §8.4 (fa_decode.cu).
//
// At g = 8 the two products need about 4 fp32 FMAs per cache byte, close to
// what the CUDA cores can issue at HBM speed, so they run on the tensor cores.
// One CTA handles one (batch, K/V head, group of up to 16 query heads, split):
//   S^T = K Q^T      M = 128 keys (TMEM lanes), N = 16 query heads (padded
//                     with zero rows), K = d; both operands K-major in shared
//                     memory
//   softmax over the keys of each query column (through shared memory: a
//                     thread takes 16 keys of one query), online (m, l) per
//                     query with the conditional rescale of the prefill (tau = 8
//                     in log2 units)
//   O^T += V^T P^T   M = d (TMEM lanes; d = 64 is padded to 128 with a zero
//                     block of shared memory), N = 16, K = 128 keys; A = V
//                     MN-major, B = P^T K-major in shared memory
// Two softmax warpgroups (warps 0-3 and 4-7) take alternate key tiles, each
// with its own running (m, l) and its own O^T accumulator, so one group's
// softmax overlaps the other's; at the end the two summaries are merged with
// the combine operator of §4.4-4.5. Warp 8 issues the TMA copies of K and V (a
// ring of stages), warp 9 issues the products. The partials (o/l, m + log2 l)
// go to the same workspace layout the merge kernel of fa_decode.cu reads.
// Every wait is bounded (fa_common.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "fa_common.cuh"
#include "fa_internal.h"
#include "fa_mma.cuh"

namespace fa {
namespace {

constexpr int kGqaThreads = 10 * 32;
constexpr int kTmaWarp = 8;
constexpr int kIssueWarp = 9;
constexpr int kQCols = 16;  // query heads per CTA (the N of both products)
constexpr uint32_t kFull = 0xffffffffu;
constexpr float kTau = 8.0f;  // conditional rescale threshold, log2 units

template <int D>
struct GqaCfg {
  static constexpr int kTileBytes = 128 * D * 2;  // one K or V tile of 128 keys
  static constexpr int kChunks = D / 64;
  static constexpr int kStages = (D == 128) ? 3 : 4;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kZeroOff = kStages * kStageBytes;  // d = 64: the zero half of V^T
  static constexpr int kZeroBytes = (D == 64) ? 128 * 64 * 2 : 0;
  static constexpr int kQOff = kZeroOff + kZeroBytes;  // Q, 16 rows, K-major
  static constexpr int kQBytes = kQCols * D * 2;
  static constexpr int kPOff = kQOff + kQBytes;  // P^T per warpgroup, 16 rows x 128 keys, K-major
  static constexpr int kPBytes = kQCols * 128 * 2;
  static constexpr int kSOff = kPOff + 2 * kPBytes;  // S^T per warpgroup, fp32 [128 keys][17]
  static constexpr int kSStride = 17;
  static constexpr int kSBytes = 128 * kSStride * 4;
  static constexpr int kVecOff = kSOff + 2 * kSBytes;  // per warpgroup: alpha, l, m per query
  static constexpr int kBarOff = kVecOff + 2 * 3 * kQCols * 4;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
};

enum GqaBar : int {
  kGFull = 0,    // + stage
  kGEmpty = 4,   // + stage
  kGS = 8,       // + warpgroup: its S^T is in TMEM
  kGP = 10,      // + warpgroup: its P^T is in shared memory (and O^T rescaled)
  kGO = 12,      // + warpgroup: its O^T product has completed
  kGQ = 14,      // Q (and the zero block) staged
  kGDone = 15,   // every product issued has completed
  kGNumBars = 16,
};

struct GqaParams {
  const __nv_bfloat16* q;  // [B][Hq][D]
  const int32_t* seqlens;
  float* ws_o;  // [B][Hq][S][D]
  float* ws_lse;  // [B][Hq][S]
  unsigned int* err;
  int Hq, Hkv, L, S, g, groups;
  float scale_log2;
};

// Keys of split s of a sequence of length len: chunks of ceil(len/S) keys
// rounded up to whole 128-key tiles.
__device__ __forceinline__ void gqa_split_range(int len, int S, int s, int& begin, int& end) {
  const int per = (((len + S - 1) / S) + 127) / 128 * 128;
  const long long b = static_cast<long long>(s) * per;
  begin = static_cast<int>(b < len ? b : len);
  end = (begin + per < len) ? begin + per : len;
}

template <int D>
__global__ void __launch_bounds__(kGqaThreads, 1)
    decode_gqa_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const GqaParams p) {
  using C = GqaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sq = base + C::kQOff;
  uint8_t* sp = base + C::kPOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[kGNumBars]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&bars[kGNumBars + 1]);
  // [4] tiles copied, O products issued, tiles of each softmax warpgroup (FA_DEBUG builds)
  uint32_t* dbg = reinterpret_cast<uint32_t*>(&bars[kGNumBars + 2]);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x;
  const int kvh = blockIdx.y / p.groups;
  const int grp = blockIdx.y % p.groups;
  const int b = blockIdx.z;
  const int hq0 = kvh * p.g + grp * kQCols;                         // first query head of the CTA
  const int nq = min(kQCols, p.g - grp * kQCols);                   // query heads it serves
  const int bkv = b * p.Hkv + kvh;                                  // row block of the caches
  int len = p.seqlens[b];
  len = len < 0 ? 0 : (len > p.L ? p.L : len);
  int k_begin, k_end;
  gqa_split_range(len, p.S, s, k_begin, k_end);
  const int n_tiles = (k_end - k_begin + 127) / 128;

  if (n_tiles == 0) {
    // an empty split: the identity of the merge (o = 0, lse = -inf)
    for (int i = tid; i < nq * D; i += kGqaThreads) {
      const int q = i / D, c = i % D;
      const size_t idx = (static_cast<size_t>(b) * p.Hq + hq0 + q) * p.S + s;
      p.ws_o[idx * D + c] = 0.f;
      if (c == 0) p.ws_lse[idx] = -INFINITY;
    }
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars[kGFull + i], 1);
      mbar_init(&bars[kGEmpty + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kGS + i], 1);
      mbar_init(&bars[kGP + i], 1);
      mbar_init(&bars[kGO + i], 1);
    }
    mbar_init(&bars[kGQ], 1);
    mbar_init(&bars[kGDone], 1);
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) dbg[i] = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S^T of warpgroup w at [16w, 16w+16), its O^T at [32+16w, 48+16w)
  constexpr uint32_t kColO = 32;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ K/V copies
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int st = t % C::kStages;
        if (t >= C::kStages &&
            !bounded_wait(&bars[kGEmpty + st], ((t / C::kStages) - 1) & 1, abort_flag, p.err, kSiteKvEmpty))
          break;
        uint8_t* stage = base + st * C::kStageBytes;
        mbar_arrive_expect_tx(&bars[kGFull + st], C::kStageBytes);
        const int row = k_begin + t * 128;
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(stage + c * kChunkBytes, &tm_k, &bars[kGFull + st], c * 64, row, bkv);
          tma_load_3d(stage + C::kTileBytes + c * kChunkBytes, &tm_v, &bars[kGFull + st], c * 64, row, bkv);
        }
        ++issued;
      }
      // every copy issued must land before the CTA exits
      for (int t = (issued > C::kStages ? issued - C::kStages : 0); t < issued; ++t)
        bounded_wait(&bars[kGFull + t % C::kStages], (t / C::kStages) & 1, nullptr, p.err, kSiteDrain);
#ifdef FA_DEBUG
      dbg[0] = static_cast<uint32_t>(issued);
#endif
    }
  } else if (warp == kIssueWarp) {
    // ------------------------------------------------------------ products
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kQCols, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, kQCols, true, false);
      bool ok = bounded_wait(&bars[kGQ], 0, abort_flag, p.err, kSiteQFull);
      const uint32_t q_addr = smem_u32(sq);
      // Issue S_t as soon as tile t has landed (and its warpgroup's S buffer
      // is free, i.e. O_{t-2} has been issued) and O_u as soon as P_u is
      // written, whichever comes first: waiting for the next tile before the
      // pending O product would hold its stage and starve the copies.
      int next_s = 0, next_o = 0;
      uint64_t idle_since = 0;
      while (ok && next_o < n_tiles) {
        bool progressed = false;
        if (next_s < n_tiles && next_s - next_o <= 1 &&
            mbar_try_wait(&bars[kGFull + next_s % C::kStages], (next_s / C::kStages) & 1)) {
          // S^T_t = K_t Q^T into the S buffer of warpgroup t % 2
          const int t = next_s;
          tc_fence_after();
          const uint32_t k_addr = smem_u32(base + (t % C::kStages) * C::kStageBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = k_addr + static_cast<uint32_t>((kk / 4) * kChunkBytes + (kk % 4) * 32);
            const uint32_t qa = q_addr + static_cast<uint32_t>((kk / 4) * (kQCols * 128) + (kk % 4) * 32);
            umma_ss(tmem + static_cast<uint32_t>((t & 1) * kQCols), smem_desc_sw128(ka, 16, 1024),
                    smem_desc_sw128(qa, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars[kGS + (t & 1)]);
          ++next_s;
          progressed = true;
        }
        if (next_o < next_s && mbar_try_wait(&bars[kGP + (next_o & 1)], (next_o >> 1) & 1)) {
          // O^T of warpgroup u % 2 += V_u^T P_u^T
          const int u = next_o, w = u & 1;
          const int st = u % C::kStages;
          tc_fence_after();
          const uint32_t v_addr = smem_u32(base + st * C::kStageBytes + C::kTileBytes);
          // MN-major A: M = d in 64-element chunks; for d = 64 the second chunk
          // is the zero block (its distance from this stage's V tile)
          const uint32_t lbo =
              (D == 128) ? static_cast<uint32_t>(kChunkBytes) : smem_u32(base + C::kZeroOff) - v_addr;
          const uint32_t p_addr = smem_u32(sp + w * C::kPBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t va = v_addr + static_cast<uint32_t>(kk * 2048);
            const uint32_t pa = p_addr + static_cast<uint32_t>((kk / 4) * (kQCols * 128) + (kk % 4) * 32);
            umma_ss(tmem + kColO + static_cast<uint32_t>(w * kQCols), smem_desc_sw128(va, lbo, 1024),
                    smem_desc_sw128(pa, 16, 1024), idesc_o, ((u >> 1) > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bars[kGEmpty + st]);
          umma_commit(&bars[kGO + w]);
          ++next_o;
          progressed = true;
        }
        // bounded: give up when nothing has been ready for the wait limit
        if (progressed) {
          idle_since = 0;
        } else if (*abort_flag) {
          ok = false;
        } else if (idle_since == 0) {
          idle_since = globaltimer_ns();
        } else if (globaltimer_ns() - idle_since > kWaitTimeoutNs) {
          *abort_flag = 1;
          record_timeout(p.err, next_s < n_tiles ? kSiteKvFull : kSitePFull);
          ok = false;
        }
      }
#ifdef FA_DEBUG
      dbg[1] = static_cast<uint32_t>(next_o);
#endif
      // every product must complete before TMEM is freed
      umma_commit(&bars[kGDone]);
      bounded_wait(&bars[kGDone], 0, nullptr, p.err, kSiteDrain);
    }
  } else {
    // ------------------------------------------------------------ softmax, rescale, epilogue
    const int wg = warp >> 2;        // warpgroup: tiles wg, wg + 2, ...
    const int wt = tid & 127;        // thread within the warpgroup
    const int bar_id = 1 + wg;       // its named barrier
    float* sS = reinterpret_cast<float*>(base + C::kSOff + wg * C::kSBytes);
    float* s_alpha = reinterpret_cast<float*>(base + C::kVecOff) + wg * 3 * kQCols;
    float* s_l = s_alpha + kQCols;
    float* s_m = s_l + kQCols;
    // stage Q (rows >= nq are zero) and, for d = 64, the zero block
    for (int i = tid; i < kQCols * (D / 8); i += 256) {
      const int r = i / (D / 8), u = i % (D / 8);  // row, 16-byte unit along d
      uint4 val = make_uint4(0, 0, 0, 0);
      if (r < nq)
        val = reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b) * p.Hq + hq0 + r) * D)[u];
      // chunk u / 8 of 16 rows x 128 bytes, unit (u % 8) swizzled by the row
      *reinterpret_cast<uint4*>(sq + (u / 8) * (kQCols * 128) + r * 128 + (((u % 8) ^ (r & 7)) << 4)) = val;
    }
    if constexpr (D == 64) {
      for (int i = tid; i < C::kZeroBytes / 16; i += 256)
        reinterpret_cast<uint4*>(base + C::kZeroOff)[i] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    named_bar_sync(3, 256);
    if (tid == 0) mbar_arrive(&bars[kGQ]);

    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_col = static_cast<uint32_t>(wg * kQCols);
    const uint32_t o_col = kColO + static_cast<uint32_t>(wg * kQCols);
    const int qi = wt >> 3;   // query column of the transposed phase
    const int seg = wt & 7;   // its 16 keys: seg*16 .. seg*16+15
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int tiles_done = 0;
    for (int t = wg; t < n_tiles; t += 2) {
      const int j = t >> 1;  // this warpgroup's tile count so far
      const int st = t % C::kStages;
      const int valid = min(128, k_end - (k_begin + t * 128));  // keys of this tile inside the split
      ok = bounded_wait(&bars[kGS + wg], j & 1, abort_flag, p.err, kSiteSFull);
      if (!named_bar_and(bar_id, 128, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        // S^T row of key wt -> shared memory [key][query]
        uint32_t r[16];
        tmem_ld_x16(tmem + lane_base + s_col, r);
        float* row = sS + wt * C::kSStride;
#pragma unroll
        for (int q = 0; q < kQCols; ++q) row[q] = __uint_as_float(r[q]);
      }
      named_bar_sync(bar_id, 128);
      // 16 keys of query qi
      float x[16];
      float tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int key = seg * 16 + i;
        x[i] = (key < valid) ? sS[key * C::kSStride + qi] * p.scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, x[i]);
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, off));
      // conditional rescale: move the running max only when it grows by more than tau
      float alpha = 1.f;
      bool rescale = false;
      if (m_run == -INFINITY) {
        m_run = tmax;  // first tile of this group: its O^T is overwritten by the product
      } else if (tmax - m_run > kTau) {
        alpha = ex2_approx(m_run - tmax);
        m_run = tmax;
        rescale = true;
      }
      float sum = 0.f;
      uint32_t pw[8];
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float p0 = ex2_approx(x[i] - m_run), p1 = ex2_approx(x[i + 1] - m_run);
        sum += p0 + p1;
        pw[i / 2] = pack_bf16x2(p0, p1);
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) sum += __shfl_xor_sync(kFull, sum, off);
      l_run = l_run * alpha + sum;
      // P^T row qi, keys seg*16..+15: two 16-byte units of chunk seg / 4
      {
        uint8_t* prow = sp + wg * C::kPBytes + (seg / 4) * (kQCols * 128) + qi * 128;
        const int u0 = (seg % 4) * 2;
        *reinterpret_cast<uint4*>(prow + ((u0 ^ (qi & 7)) << 4)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        *reinterpret_cast<uint4*>(prow + (((u0 + 1) ^ (qi & 7)) << 4)) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
      }
      if (seg == 0) s_alpha[qi] = alpha;
      // cache rows past the split are not part of this product (and may hold
      // anything, NaN included): zero them in the V tile
      if (valid < 128) {
        uint8_t* vt = base + st * C::kStageBytes + C::kTileBytes;
        for (int i = wt; i < (128 - valid) * C::kChunks * 8; i += 128) {
          const int r = valid + i / (C::kChunks * 8);
          const int rem = i % (C::kChunks * 8);
          *reinterpret_cast<uint4*>(vt + (rem / 8) * kChunkBytes + r * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      const bool any_rescale = named_bar_or(bar_id, 128, rescale);
      // this group's previous O^T product must be complete before O^T is touched again
      if (j >= 1) {
        ok = bounded_wait(&bars[kGO + wg], (j - 1) & 1, abort_flag, p.err, kSiteOFull);
        if (!named_bar_and(bar_id, 128, ok)) {
          ok = false;
          break;
        }
      }
      if (any_rescale) {
        tc_fence_after();
        uint32_t r[16];
        tmem_ld_x16(tmem + lane_base + o_col, r);
#pragma unroll
        for (int q = 0; q < kQCols; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) * s_alpha[q]);
        tmem_st_x16(tmem + lane_base + o_col, r);
        tmem_st_wait();
      }
      tc_fence_before();
      named_bar_sync(bar_id, 128);
      if (wt == 0) mbar_arrive(&bars[kGP + wg]);
      ++tiles_done;
    }
    // this group's last product, then its summary (m, l) per query
    if (ok && tiles_done > 0) ok = bounded_wait(&bars[kGO + wg], (tiles_done - 1) & 1, abort_flag, p.err, kSiteOFull);
#ifdef FA_DEBUG
    if (wt == 0) dbg[2 + wg] = static_cast<uint32_t>(tiles_done);
#endif
    if (seg == 0) {
      s_l[qi] = l_run;
      s_m[qi] = m_run;
    }
    // epilogue by warpgroup 0: merge the two groups' (m, l, O^T) (combine
    // operator), then the partials o / l and m + log2 l of every query
    if (named_bar_and(3, 256, ok) && wg == 0) {
      tc_fence_after();
      const float* l1 = s_l + 3 * kQCols;  // warpgroup 1's vectors
      const float* m1 = s_m + 3 * kQCols;
      uint32_t r0[16], r1[16];
      tmem_ld_x16(tmem + lane_base + kColO, r0);
      tmem_ld_x16(tmem + lane_base + kColO + kQCols, r1);
      if (wt < D) {
        for (int q = 0; q < nq; ++q) {
          const size_t idx = (static_cast<size_t>(b) * p.Hq + hq0 + q) * p.S + s;
          const float ma = s_m[q], mb = m1[q];
          const float mx = fmaxf(ma, mb);  // finite: group 0 saw at least one key
          const float wa = ex2_approx(ma - mx);
          const float wb = (mb == -INFINITY) ? 0.f : ex2_approx(mb - mx);
          const float l = wa * s_l[q] + wb * l1[q];
          // group 1's accumulator is never written when it saw no tile
          const float acc = wa * __uint_as_float(r0[q]) + ((wb > 0.f) ? wb * __uint_as_float(r1[q]) : 0.f);
          p.ws_o[idx * D + wt] = (l > 0.f) ? acc / l : 0.f;
          if (wt == 0) p.ws_lse[idx] = (l > 0.f) ? mx + log2f(l) : -INFINITY;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
#ifdef FA_DEBUG
  // protocol check: every tile of the split was copied once, multiplied once
  // into O, and taken by one softmax warpgroup
  if (tid == 0 && *abort_flag == 0) {
    const uint32_t n = static_cast<uint32_t>(n_tiles);
    if (dbg[0] != n || dbg[1] != n || dbg[2] + dbg[3] != n) record_check(p.err, kSiteCheckGqa);
  }
#endif
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

template <int D>
fa_status launch(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens, int B, int Hq,
                 int Hkv, int L, int S, float* ws_o, float* ws_lse, cudaStream_t stream, unsigned int* err) {
  using C = GqaCfg<D>;
  CUtensorMap tk, tv;
  const uint64_t rows = static_cast<uint64_t>(B) * Hkv;
  if (!encode_bf16_map(&tk, k_cache, D, L, rows, 128) || !encode_bf16_map(&tv, v_cache, D, L, rows, 128))
    return FA_ERR_CUDA;
  GqaParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.seqlens = seqlens;
  prm.ws_o = ws_o;
  prm.ws_lse = ws_lse;
  prm.err = err;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.L = L;
  prm.S = S;
  prm.g = Hq / Hkv;
  prm.groups = (prm.g + kQCols - 1) / kQCols;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  cudaError_t e = cudaFuncSetAttribute(decode_gqa_split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) {
    set_error_text("cudaFuncSetAttribute(decode_gqa_split_kernel)", e);
    return FA_ERR_CUDA;
  }
  dim3 grid(static_cast<unsigned>(S), static_cast<unsigned>(Hkv * prm.groups), static_cast<unsigned>(B));
  decode_gqa_split_kernel<D><<<grid, kGqaThreads, C::kSmemBytes, stream>>>(tk, tv, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("decode_gqa_split_kernel launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

}  // namespace

fa_status launch_decode_gqa_split(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens,
                                  int B, int Hq, int Hkv, int L, int d, int num_splits, float* ws_o, float* ws_lse,
                                  cudaStream_t stream, unsigned int* err) {
  if (d == 128)
    return launch<128>(q, k_cache, v_cache, seqlens, B, Hq, Hkv, L, num_splits, ws_o, ws_lse, stream, err);
  if (d == 64)
    return launch<64>(q, k_cache, v_cache, seqlens, B, Hq, Hkv, L, num_splits, ws_o, ws_lse, stream, err);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
