// Fused prefill attention for sm_103a: tcgen05 tensor cores with TMEM
// accumulators, TMA-fed shared-memory pipeline, warp-specialised roles,
// persistent CTAs.
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
// Mapping onto one CTA (one per SM; TMEM holds 512 columns x 128 lanes):
//   * a work item is two Q tiles of 128 rows each (256 query rows of one
//     head); the CTA loops over work items (persistent), so the next item's
//     Q/K loads and first products overlap the current item's epilogue;
//   * items are ordered heaviest first (causal: largest row index first) and
//     dealt to the CTAs in a snake order, which balances the causal load;
//   * warps 0-3: softmax of Q tile 0, warps 4-7: softmax of Q tile 1
//     (thread r of a warpgroup owns row r; a row's max and sum are in-thread);
//   * warp 8: one thread issues every tcgen05.mma and commit;
//   * warp 9: one thread issues every TMA copy (Q, then K_j, V_j into a ring
//     of shared-memory slots);
//   * the epilogue of a tile stages O in 64-column boxes in shared memory and
//     one of its threads stores each box with a TMA tensor store, so the O
//     rows leave through the TMA unit rather than the load/store path.
//   TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
//   P (bf16 pairs) overwrites the first 64 columns of its S tile and is the
//   TMEM A operand of O += P V. While warpgroup 0 runs the softmax of S0 the
//   tensor core works on tile 1's products, and the other way round.
//
// With a block mask (block-sparse FlashAttention, "FlashAttention 完全拆解
// （一）", block-sparse extension) an item's two Q tiles share the copies of
// the union of the K/V tiles their masks keep, and each Q tile computes only
// the K/V tiles its own mask keeps; tiles outside the union are never loaded.
//
// The same kernel runs the FP8 path ("已有的几种大模型上下文支持情况" §4.4,
// FA-3): e4m3 Q and K with one scale per 128-row tile (the product of the two
// tile scales joins the softmax scale of each S tile), V given transposed as
// e4m3 with one scale per head (applied with the final 1 / l), both products
// on kind::f8f6f4, and P rounded to e4m3 (four keys per TMEM column) for the
// P V product while l sums the fp32 values.
//
// Every role walks the same item sequence and keeps its own barrier phase
// counters. Every wait is bounded (fa_common.cuh); a wait that runs out
// records the site, raises the CTA abort flag, and every role drains its
// in-flight copies or products before TMEM is freed.
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
// Block-sparse items are handed out at run time: the loading thread takes the
// next item index from a global counter and publishes it to the CTA's other
// roles through this many shared-memory slots.
constexpr int kItemSlots = 4;
// arrivals that free an item slot: the MMA thread and one lane per softmax warp
constexpr int kItemReaders = 1 + 8;

// F8: e4m3 Q, K and V^T (d = 128 only: a 128-byte row is one swizzle chunk).
template <int D, bool F8 = false>
struct Cfg {
  static_assert(!F8 || D == 128, "e4m3 tiles need 128-byte rows");
  static constexpr int kTileBytes = kBN * D * (F8 ? 1 : 2);  // one Q, K or V tile
  static constexpr int kChunks = F8 ? 1 : D / 64;
  static constexpr int kStages = (D == 128 && !F8) ? 4 : 8;  // K/V ring slots
  // TMEM column of S (and P) and of O for Q tile t
  __host__ __device__ static constexpr uint32_t s_col(int t) { return t ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t o_col(int t) { return t ? 256u + D : 256u; }
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kRingOff = 2 * kTileBytes;
  // epilogue staging: per tile one 64-column box of O (128 rows x 128 bytes, 128-byte swizzle)
  static constexpr int kOStageOff = kRingOff + kStages * kTileBytes;
  static constexpr int kOStageBytes = 128 * 128;
  static constexpr int kBarOff = kOStageOff + 2 * kOStageBytes;
  // q_full, q_empty, s_full, p_full, o_full, o_empty (2 each), kv_full, kv_empty, mma_done,
  // item_full, item_empty
  static constexpr int kNumBars = 12 + 2 * kStages + 1 + 2 * kItemSlots;
  // + TMEM slot, abort flag, output-map address, 16 protocol counters (FA_DEBUG), item slots,
  // slack to align to 1 KB
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 64 + 4 * kItemSlots + 1024;
};

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  unsigned int* err;
  // e4m3 inputs only: per-tile scales of Q and K ([BH][tiles]) and per-head scale of V ([BH])
  const float* sq;
  const float* sk;
  const float* sv;
  int tiles;
  // block-sparse mode only: per (mask head, Q-tile pair) the union of the K/V
  // tiles its two Q tiles keep, as words (tile | allowed for Q tile 0 << 16 |
  // allowed for Q tile 1 << 17), list[(mh * pairs + pair) * tiles + step], and
  // cnt[3 * (mh * pairs + pair) + {0, 1, 2}]: the union's step count and the
  // number of those steps Q tile 0 and Q tile 1 keep
  const uint32_t* list;
  const int* cnt;
  int* next_item;  // block-sparse: the run-time item counter (zeroed by sparse_list_kernel)
  int mask_heads;
  int H;
  int N;
  int BH;          // batch * heads
  int num_pairs;   // Q-tile pairs per head
  int num_items;   // BH * num_pairs
  int causal;
  int swap_tiles;    // dense causal items: tile 0 takes the pair's second 128 rows
  float scale_log2;  // scale * log2(e)
};

struct Smem {
  uint8_t* q[2];
  uint8_t* ring;
  uint8_t* ostage;  // [2][kOStageBytes]
  uint64_t* q_full;    // [2]   Q tile landed
  uint64_t* q_empty;   // [2]   last S = Q K^T of an item done: Q buffer free (softmax arrives)
  uint64_t* s_full;    // [2]   S = Q K^T done (also: every earlier product done)
  uint64_t* p_full;    // [2]   P written to TMEM and O rescaled (128 arrivals)
  uint64_t* o_full;    // [2]   last O += P V of an item done
  uint64_t* o_empty;   // [2]   O read out of TMEM by the epilogue (128 arrivals)
  uint64_t* kv_full;   // [S]   K or V tile landed in a ring slot
  uint64_t* kv_empty;  // [S]   ring slot free again (softmax arrives)
  uint64_t* mma_done;  // [1]   every product done (teardown)
  uint64_t* item_full;   // [kItemSlots] block-sparse: an item index was published in the slot
  uint64_t* item_empty;  // [kItemSlots] block-sparse: every role has read the slot (kItemReaders arrivals)
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  uint32_t* dbg;       // [16] per-role protocol counters, compared at the end (FA_DEBUG builds)
  volatile int* item_q;  // [kItemSlots] block-sparse: published item indices
  // the generic address of the output tensor map (a kernel parameter), read by
  // the epilogue's storing threads only: a register the softmax loop does not hold
  const CUtensorMap* const* tmo;
};

template <int D, bool F8>
__device__ __forceinline__ Smem carve(uint8_t* raw) {
  using C = Cfg<D, F8>;
  const uint32_t a = smem_u32(raw);
  uint8_t* base = raw + ((1024u - (a & 1023u)) & 1023u);
  Smem s;
  s.q[0] = base;
  s.q[1] = base + C::kTileBytes;
  s.ring = base + C::kRingOff;
  s.ostage = base + C::kOStageOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  s.q_full = bars;
  s.q_empty = bars + 2;
  s.s_full = bars + 4;
  s.p_full = bars + 6;
  s.o_full = bars + 8;
  s.o_empty = bars + 10;
  s.kv_full = bars + 12;
  s.kv_empty = s.kv_full + C::kStages;
  s.mma_done = s.kv_empty + C::kStages;
  s.item_full = s.mma_done + 1;
  s.item_empty = s.item_full + kItemSlots;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.item_empty + kItemSlots);
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  s.tmo = reinterpret_cast<const CUtensorMap* const*>(s.tmem_slot + 2);
  s.dbg = reinterpret_cast<uint32_t*>(s.tmem_slot + 4);
  s.item_q = reinterpret_cast<volatile int*>(s.dbg + 16);
  return s;
}

// One work item: Q rows [q0, q0 + 256) of head bh; tile t visits n(t) K/V tiles.
// Dense: tile t visits K/V tiles 0 .. n(t)-1. Block-sparse ("FlashAttention
// 完全拆解（一）", block-sparse extension): the item walks the union of the
// K/V tiles the two tiles' masks keep (sparse_list_kernel), and tile t computes
// the kept(t) steps its own mask keeps; a tile that keeps none writes o = 0 and
// lse = -inf for its rows.
struct Item {
  int bh;
  int q0;
  int r0, r1;  // first query row of tile 0 and of tile 1
  int n0;
  int n1;
  int c0, c1;            // steps tile 0 and tile 1 compute (block-sparse: the steps their masks keep)
  const uint32_t* list;  // block-sparse: this item's steps
  __device__ __forceinline__ int n(int t) const { return t ? n1 : n0; }
  __device__ __forceinline__ int kept(int t) const { return t ? c1 : c0; }
  __device__ __forceinline__ int row(int t) const { return t ? r1 : r0; }
  __device__ __forceinline__ int n_max() const { return n0 > n1 ? n0 : n1; }
};

// K/V tile of step j, and whether Q tile t keeps it.
template <bool SP>
__device__ __forceinline__ uint32_t step_word(const Item& it, int j) {
  if constexpr (!SP) return static_cast<uint32_t>(j) | (3u << 16);
  return __ldg(it.list + j);
}

// Item w of the heavy-first item list, or false past its end.
template <bool SP>
__device__ __forceinline__ bool item_decode(const FwdParams& p, long long w, Item& it) {
  if (w >= p.num_items) return false;
  const int rank = static_cast<int>(w / p.BH);
  it.bh = static_cast<int>(w - static_cast<long long>(rank) * p.BH);
  const int pair = p.causal ? (p.num_pairs - 1 - rank) : rank;
  it.q0 = pair * 2 * kBM;
  if constexpr (!SP) {
    // swap_tiles: tile 0 takes the later rows (under the causal mask one K/V
    // step more), so tile 1's epilogue runs while tile 0 takes that step alone
    it.r0 = p.swap_tiles ? it.q0 + kBM : it.q0;
    it.r1 = p.swap_tiles ? it.q0 : it.q0 + kBM;
    it.n0 = fwd_kv_tiles(it.r0, p.N, kBN, p.causal);
    it.n1 = fwd_kv_tiles(it.r1, p.N, kBN, p.causal);
    it.c0 = it.n0;
    it.c1 = it.n1;
    it.list = nullptr;
  } else {
    const int mh = (p.mask_heads == 1) ? 0 : (it.bh % p.H);
    const size_t row = static_cast<size_t>(mh) * p.num_pairs + pair;
    const int nu = __ldg(p.cnt + 3 * row);
    it.r0 = it.q0;
    it.r1 = it.q0 + kBM;
    it.list = p.list + row * p.tiles;
    it.n0 = nu;
    it.n1 = (it.q0 + kBM < p.N) ? nu : 0;
    it.c0 = __ldg(p.cnt + 3 * row + 1);
    it.c1 = (it.q0 + kBM < p.N) ? __ldg(p.cnt + 3 * row + 2) : 0;
  }
  return true;
}

// Dense: the k-th item of this CTA, dealt in a snake order over the
// heavy-first list (the causal load balances by construction).
__device__ __forceinline__ bool item_at(const FwdParams& p, int k, Item& it) {
  const int G = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  return item_decode<false>(p, static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c), it);
}

// Block-sparse items differ in cost by the number of K/V tiles their masks
// keep (a global row keeps them all), so a static deal leaves some CTAs with
// far more work; they are handed out at run time instead, in list order
// (greedy list scheduling). The loading thread publishes item k of this CTA
// in slot k % kItemSlots; the other roles read it from there (fetch_item).
__device__ __forceinline__ bool publish_item(const Smem& sm, const FwdParams& p, int k, int idx, bool& ok) {
  const int e = k % kItemSlots;
  const uint32_t use = static_cast<uint32_t>(k / kItemSlots);
  if (use > 0) {
    ok = bounded_wait(&sm.item_empty[e], (use - 1) & 1, sm.abort_flag, p.err, kSiteItemEmpty);
    if (!ok) return false;
  }
  sm.item_q[e] = idx;
  mbar_arrive(&sm.item_full[e]);  // releases the store above to the slot's readers
  return true;
}

// Item k of this CTA as published by the loading thread. `warp_reader`: the
// caller is a full warp (one arrival from lane 0 after every lane has read
// the slot); otherwise a single thread (the MMA issuer).
template <bool SP>
__device__ __forceinline__ bool fetch_item(const Smem& sm, const FwdParams& p, int k, Item& it, bool& ok,
                                           bool warp_reader) {
  if constexpr (!SP) {
    return item_at(p, k, it);
  } else {
    const int e = k % kItemSlots;
    ok = bounded_wait(&sm.item_full[e], static_cast<uint32_t>(k / kItemSlots) & 1, sm.abort_flag, p.err,
                      kSiteItemFull);
    if (warp_reader) ok = __all_sync(kFull, ok);
    if (!ok) return false;
    const int idx = sm.item_q[e];
    if (warp_reader) {
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&sm.item_empty[e]);
    } else {
      mbar_arrive(&sm.item_empty[e]);
    }
    return item_decode<true>(p, idx, it);
  }
}

// ---------------------------------------------------------------- TMA producer (one thread)
template <int D, bool F8, bool SP>
__device__ void load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v, const Smem& sm,
                          const FwdParams& p) {
  using C = Cfg<D, F8>;
  tma_prefetch_desc(tm_q);
  tma_prefetch_desc(tm_k);
  tma_prefetch_desc(tm_v);
  uint32_t ring = 0;            // K/V tiles issued so far
  uint32_t q_cnt[2] = {0, 0};   // Q tiles issued per buffer
  bool ok = true;
  Item it;
  // block-sparse: the next item index is taken one item ahead, so the atomic's
  // latency overlaps this item's copies
  int idx_next = SP ? atomicAdd(p.next_item, 1) : 0;
  for (int k = 0; ok; ++k) {
    if constexpr (SP) {
      const int idx = idx_next;
      if (!publish_item(sm, p, k, idx, ok)) break;
      if (!item_decode<true>(p, idx, it)) break;
      idx_next = atomicAdd(p.next_item, 1);
    } else {
      if (!item_at(p, k, it)) break;
    }
    for (int t = 0; t < 2 && ok; ++t) {
      if (it.kept(t) == 0) continue;
      if (q_cnt[t] > 0) {
        ok = bounded_wait(&sm.q_empty[t], (q_cnt[t] - 1) & 1, sm.abort_flag, p.err, kSiteQEmpty);
        if (!ok) break;
      }
      mbar_arrive_expect_tx(&sm.q_full[t], C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(sm.q[t] + c * kChunkBytes, tm_q, &sm.q_full[t], c * 64, it.row(t), it.bh);
      ++q_cnt[t];
    }
    const int n_max = it.n_max();
    uint32_t next_word = SP ? step_word<SP>(it, 0) : 0u;
    for (int j = 0; j < n_max && ok; ++j) {
      int jt = j;  // K/V tile of step j
      if constexpr (SP) {
        jt = static_cast<int>(next_word & 0xffffu);
        if (j + 1 < n_max) next_word = step_word<SP>(it, j + 1);  // one step ahead
      }
      for (int kind = 0; kind < 2; ++kind) {
        const uint32_t slot = ring % C::kStages;
        const uint32_t use = ring / C::kStages;
        if (use > 0) {
          ok = bounded_wait(&sm.kv_empty[slot], (use - 1) & 1, sm.abort_flag, p.err, kSiteKvEmpty);
          if (!ok) break;
        }
        uint8_t* dst = sm.ring + slot * C::kTileBytes;
        // K_j (j >= 1) lands on the barrier of V_(j-1), whose expected bytes
        // counted it, so the MMA thread waits once per step for V_(j-1) and
        // K_j; its own barrier completes its phase with a plain arrival.
        uint64_t* bar = &sm.kv_full[slot];
        if (kind == 0 && j > 0) {
          mbar_arrive(bar);
          bar = &sm.kv_full[(ring - 1) % C::kStages];
        } else {
          mbar_arrive_expect_tx(bar, (kind == 1 && j + 1 < n_max) ? 2 * C::kTileBytes : C::kTileBytes);
        }
        const CUtensorMap* map = kind ? tm_v : tm_k;
        if (F8 && kind) {
          // V^T: rows are d, the 128 keys of tile jt are the inner coordinate
          tma_load_3d(dst, map, bar, jt * kBN, 0, it.bh);
        } else {
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(dst + c * kChunkBytes, map, bar, c * 64, jt * kBN, it.bh);
        }
        ++ring;
      }
    }
  }
  // Drain: every copy issued must land before the CTA can exit.
  for (uint32_t r = (ring > C::kStages ? ring - C::kStages : 0); r < ring; ++r)
    bounded_wait(&sm.kv_full[r % C::kStages], (r / C::kStages) & 1, nullptr, p.err, kSiteDrain);
  for (int t = 0; t < 2; ++t)
    if (q_cnt[t] > 0) bounded_wait(&sm.q_full[t], (q_cnt[t] - 1) & 1, nullptr, p.err, kSiteDrain);
#ifdef FA_DEBUG
  sm.dbg[0] = ring;
  sm.dbg[1] = q_cnt[0];
  sm.dbg[2] = q_cnt[1];
#endif
}

// ---------------------------------------------------------------- MMA issuer (one thread)
template <int D, bool F8>
__device__ __forceinline__ void qk_product(uint32_t s_tmem, uint32_t q_smem, uint32_t k_smem) {
  if constexpr (F8)
    issue_qk_f8(s_tmem, q_smem, k_smem);
  else
    issue_qk<D>(s_tmem, q_smem, k_smem);
}

template <int D, bool F8>
__device__ __forceinline__ void pv_product(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem, bool accumulate) {
  if constexpr (F8)
    issue_pv_f8(o_tmem, p_tmem, v_smem, accumulate);
  else
    issue_pv<D>(o_tmem, p_tmem, v_smem, accumulate);
}

// At every step tile 0's products are issued before tile 1's. The buffer
// releases depend on it: a K or V tile both read is released by tile 1 (its
// last reader) once tile 1's product on it completes, which then implies tile
// 0's. Issuing a tile's products as soon as they are ready, or starting tile 0
// on its next item early, also breaks the lock-step the two tiles need to share
// a K/V ring two steps deep.
template <int D, bool F8, bool SP>
__device__ void mma_role(const Smem& sm, uint32_t tmem, const FwdParams& p) {
  using C = Cfg<D, F8>;
  const uint32_t ring_base = smem_u32(sm.ring);
  const uint32_t qa0 = smem_u32(sm.q[0]);
  const uint32_t qa1 = smem_u32(sm.q[1]);
  auto slot_addr = [&](uint32_t r) { return ring_base + (r % C::kStages) * static_cast<uint32_t>(C::kTileBytes); };
  auto wait_kv = [&](uint32_t r) {
    return bounded_wait(&sm.kv_full[r % C::kStages], (r / C::kStages) & 1, sm.abort_flag, p.err, kSiteKvFull);
  };
  uint32_t ring = 0;                 // K/V tiles consumed so far
  uint32_t q_cnt[2] = {0, 0};        // Q tiles consumed per buffer
  uint32_t p_cnt[2] = {0, 0};        // p_full phases consumed per tile
  uint32_t o_cnt[2] = {0, 0};        // items whose O_t was produced
  bool ok = true;
  Item it;
  for (int k = 0; ok && fetch_item<SP>(sm, p, k, it, ok, false); ++k) {
    for (int t = 0; t < 2 && ok; ++t) {
      if (it.n(t) == 0) continue;
      ok = bounded_wait(&sm.q_full[t], q_cnt[t] & 1, sm.abort_flag, p.err, kSiteQFull);
      ++q_cnt[t];
    }
    if (!ok) break;
    const uint32_t base = ring;  // K_j is base + 2j, V_j is base + 2j + 1
    const int n_max = it.n_max();
    ok = wait_kv(base);
    if (!ok) break;
    tc_fence_after();
    for (int t = 0; t < 2; ++t) {
      if (it.n(t) == 0) continue;
      qk_product<D, F8>(tmem + C::s_col(t), t ? qa1 : qa0, slot_addr(base));
      umma_commit(&sm.s_full[t]);
    }
    for (int j = 0; j < n_max && ok; ++j) {
      const uint32_t iv = base + 2 * j + 1;  // V_j
      const uint32_t ik = base + 2 * j + 2;  // K_{j+1}
      ok = wait_kv(iv);  // V_j, and K_{j+1} if the item has it (both land on V_j's barrier)
      if (!ok) break;
      for (int t = 0; t < 2; ++t) {
        const int nt = it.n(t);
        if (j >= nt) continue;
        ok = bounded_wait(&sm.p_full[t], p_cnt[t] & 1, sm.abort_flag, p.err, kSitePFull);
        ++p_cnt[t];
        if (!ok) break;
        if (j == 0 && o_cnt[t] > 0) {
          // the first O += P V of an item overwrites O_t: the previous item's
          // epilogue must have read it out
          ok = bounded_wait(&sm.o_empty[t], (o_cnt[t] - 1) & 1, sm.abort_flag, p.err, kSiteOEmpty);
          if (!ok) break;
        }
        tc_fence_after();
        pv_product<D, F8>(tmem + C::o_col(t), tmem + C::s_col(t), slot_addr(iv), j > 0);
        if (j + 1 < nt) {
          // issued after P V of the same tile: the tensor pipe runs them in order,
          // so P is read before the new S overwrites those columns
          qk_product<D, F8>(tmem + C::s_col(t), t ? qa1 : qa0, slot_addr(ik));
          umma_commit(&sm.s_full[t]);
        } else {
          umma_commit(&sm.o_full[t]);
          ++o_cnt[t];
        }
      }
      if (!ok) break;
    }
    ring = base + 2 * n_max;
  }
  // Teardown: every product issued so far must finish before TMEM is freed.
  umma_commit(sm.mma_done);
  bounded_wait(sm.mma_done, 0, nullptr, p.err, kSiteDrain);
#ifdef FA_DEBUG
  sm.dbg[3] = ring;
  for (int t = 0; t < 2; ++t) {
    sm.dbg[4 + t] = q_cnt[t];
    sm.dbg[6 + t] = p_cnt[t];
    sm.dbg[8 + t] = o_cnt[t];
  }
#endif
}

// Block-sparse issuer. The two Q tiles walk the union of their masks' K/V tiles
// (one copy of each), but tile t's products run only on the steps its mask
// keeps. Per union step j: O_t += P_t V_j where tile t keeps j, then S_t(j+1)
// where it keeps j+1 (after the tile's last P V, which read the TMEM columns
// S_t overwrites). A tile's next S may lie many steps ahead, so V_j is released
// by a commit after the P V of its last reader rather than by that reader's
// next S, and a tile's O is complete after its last kept step.
template <int D>
__device__ void mma_role_sparse(const Smem& sm, uint32_t tmem, const FwdParams& p) {
  using C = Cfg<D, false>;
  const uint32_t ring_base = smem_u32(sm.ring);
  const uint32_t qa0 = smem_u32(sm.q[0]);
  const uint32_t qa1 = smem_u32(sm.q[1]);
  auto slot_addr = [&](uint32_t r) { return ring_base + (r % C::kStages) * static_cast<uint32_t>(C::kTileBytes); };
  auto wait_kv = [&](uint32_t r) {
    return bounded_wait(&sm.kv_full[r % C::kStages], (r / C::kStages) & 1, sm.abort_flag, p.err, kSiteKvFull);
  };
  auto keeps = [](uint32_t word, int t) { return ((word >> (16 + t)) & 1u) != 0; };
  uint32_t ring = 0;
  uint32_t q_cnt[2] = {0, 0};
  uint32_t p_cnt[2] = {0, 0};
  uint32_t o_cnt[2] = {0, 0};
  bool ok = true;
  Item it;
  for (int k = 0; ok && fetch_item<true>(sm, p, k, it, ok, false); ++k) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (!ok || it.kept(t) == 0) continue;
      ok = bounded_wait(&sm.q_full[t], q_cnt[t] & 1, sm.abort_flag, p.err, kSiteQFull);
      ++q_cnt[t];
    }
    if (!ok) break;
    const uint32_t base = ring;
    const int nu = it.n_max();
    ring = base + 2 * nu;
    if (nu == 0) continue;
    ok = wait_kv(base);
    if (!ok) break;
    uint32_t w = step_word<true>(it, 0);
    tc_fence_after();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (!keeps(w, t)) continue;
      qk_product<D, false>(tmem + C::s_col(t), t ? qa1 : qa0, slot_addr(base));
      umma_commit(&sm.s_full[t]);
    }
    int done[2] = {0, 0};  // kept steps whose P V was issued, per tile
    for (int j = 0; j < nu && ok; ++j) {
      const uint32_t iv = base + 2 * j + 1;  // V_j
      const uint32_t ik = base + 2 * j + 2;  // K_(j+1)
      const uint32_t wn = (j + 1 < nu) ? step_word<true>(it, j + 1) : 0u;
      ok = wait_kv(iv);  // V_j, and K_(j+1) if the union has it (both land on V_j's barrier)
      if (!ok) break;
      const int last_v = keeps(w, 1) ? 1 : 0;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!ok) continue;
        if (keeps(w, t)) {
          ok = bounded_wait(&sm.p_full[t], p_cnt[t] & 1, sm.abort_flag, p.err, kSitePFull);
          ++p_cnt[t];
          if (ok && done[t] == 0 && o_cnt[t] > 0)
            ok = bounded_wait(&sm.o_empty[t], (o_cnt[t] - 1) & 1, sm.abort_flag, p.err, kSiteOEmpty);
          if (!ok) continue;
          tc_fence_after();
          pv_product<D, false>(tmem + C::o_col(t), tmem + C::s_col(t), slot_addr(iv), done[t] > 0);
          ++done[t];
          if (t == last_v) umma_commit(&sm.kv_empty[iv % C::kStages]);
          if (done[t] == it.kept(t)) {
            umma_commit(&sm.o_full[t]);
            ++o_cnt[t];
          }
        }
        if (keeps(wn, t)) {
          qk_product<D, false>(tmem + C::s_col(t), t ? qa1 : qa0, slot_addr(ik));
          umma_commit(&sm.s_full[t]);
        }
      }
      w = wn;
    }
  }
  // Teardown: every product issued so far must finish before TMEM is freed.
  umma_commit(sm.mma_done);
  bounded_wait(sm.mma_done, 0, nullptr, p.err, kSiteDrain);
#ifdef FA_DEBUG
  sm.dbg[3] = ring;
  for (int t = 0; t < 2; ++t) {
    sm.dbg[4 + t] = q_cnt[t];
    sm.dbg[6 + t] = p_cnt[t];
    sm.dbg[8 + t] = o_cnt[t];
  }
#endif
}

// The tile whose products read K_j and V_j last (tile 1 unless it stops earlier).
__device__ __forceinline__ int last_reader(const Item& it, int j) { return (it.n1 > j) ? 1 : 0; }

// Buffer releases, made by one softmax thread per tile with plain mbarrier
// arrivals right after it has seen S_t(j) complete (a tcgen05.commit for each
// release would cost tensor-pipe time). S_t(j) done means every product issued
// before it is done too:
//   K_j      is free when the S of its last reader is done,
//   V_(j-1)  is free when the next S of its last reader is done (the last V of
//            a tile is released after that tile's final O += P V instead),
//   Q_t      is free when the item's last S_t is done.
template <int D, bool F8>
__device__ __forceinline__ void release_after_s(const Smem& sm, const Item& it, int t, int j, uint32_t ring_base) {
  using C = Cfg<D, F8>;
  if (last_reader(it, j) == t) mbar_arrive(&sm.kv_empty[(ring_base + 2 * j) % C::kStages]);
  if (j > 0 && last_reader(it, j - 1) == t) mbar_arrive(&sm.kv_empty[(ring_base + 2 * (j - 1) + 1) % C::kStages]);
  if (j == it.n(t) - 1) mbar_arrive(&sm.q_empty[t]);
}

// ---------------------------------------------------------------- softmax + epilogue (128 threads per tile)
template <int D, bool F8, bool SP>
__device__ void softmax_role(const Smem& sm, uint32_t tmem, const FwdParams& p, int warp, int lane) {
  using C = Cfg<D, F8>;
  const int t = warp >> 2;
  const int quarter = warp & 3;  // this warp may touch TMEM lanes [32*quarter, 32*quarter+32)
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t s_tm = tmem + lane_base + C::s_col(t);
  const uint32_t o_tm = tmem + lane_base + C::o_col(t);
  float sl2 = p.scale_log2;
  uint64_t sl2x2 = f2_pack(sl2, sl2);
  uint32_t s_cnt = 0;  // s_full phases consumed
  uint32_t o_cnt = 0;  // o_full phases consumed
  bool ok = true;
  Item it;
  const bool releaser = (quarter == 0 && lane == 0);  // one thread per tile releases buffers
  uint32_t ring_next = 0;                             // K/V ring position of the next item
  for (int k = 0; ok && fetch_item<SP>(sm, p, k, it, ok, true); ++k) {
    const uint32_t ring_base = ring_next;  // K_j is ring_base + 2j, V_j is ring_base + 2j + 1
    ring_next += 2 * it.n_max();
    const int nkv = it.n(t);
    const int q_row = it.row(t) + row;
    if (SP && it.kept(t) == 0) {
      // the mask keeps no K/V tile for these rows: o = 0, lse = -inf
      if (q_row < p.N) {
        uint4* dst4 = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(it.bh) * p.N + q_row) * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst4[i] = make_uint4(0u, 0u, 0u, 0u);
        p.lse[static_cast<size_t>(it.bh) * p.N + q_row] = -INFINITY;
      }
      continue;
    }
    if (nkv == 0) continue;
    const int vis_end = p.causal ? min(q_row + 1, p.N) : p.N;  // keys [0, vis_end) are visible to this row
    float m_used = -INFINITY;  // base of every exponent so far (log2 domain, scaled)
    float l = 0.f;
    // dense: steps j = 0 .. nkv-1; block-sparse: the kept(t) steps of the union
    // this tile's mask keeps, u walking the union (K_u, V_u at ring_base + 2u)
    const int steps = SP ? it.kept(t) : nkv;
    int u = 0;
    for (int j = 0; j < steps; ++j) {
      int jt = j;  // K/V tile of this step
      bool last_k = false;  // block-sparse: this tile reads K_u last
      if constexpr (SP) {
        uint32_t word = step_word<SP>(it, u);
        while (((word >> (16 + t)) & 1u) == 0) word = step_word<SP>(it, ++u);
        jt = static_cast<int>(word & 0xffffu);
        last_k = t == 1 || ((word >> 17) & 1u) == 0;
      }
      ok = bounded_wait(&sm.s_full[t], s_cnt & 1, sm.abort_flag, p.err, kSiteSFull);
      ++s_cnt;
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      if (releaser) {
        if constexpr (SP) {
          // K_u once its last reader's S is done; V_u is released by the issuing
          // thread's commit after its last P V; Q_t after the tile's last S
          if (last_k) mbar_arrive(&sm.kv_empty[(ring_base + 2 * u) % C::kStages]);
          if (j + 1 == steps) mbar_arrive(&sm.q_empty[t]);
        } else {
          release_after_s<D, F8>(sm, it, t, j, ring_base);
        }
      }
      if constexpr (SP) ++u;
      tc_fence_after();
      if constexpr (F8) {
        // block-wise scales of the e4m3 inputs: Q tile and K tile j of this head
        const size_t sb = static_cast<size_t>(it.bh) * p.tiles;
        sl2 = p.scale_log2 * __ldg(p.sq + sb + it.row(t) / kBM) * __ldg(p.sk + sb + jt);
        sl2x2 = f2_pack(sl2, sl2);
      }

      // visible keys of this tile for this row
      const int lim = vis_end - jt * kBN;
      if constexpr (F8) {
        // e4m3 inputs: one pass over the row. The 128 raw scores are loaded once, their
        // maximum taken (scale > 0, so it commutes with the scaling), then
        // p = 2^(s * scale * log2 e - m) in place, the row sum in packed pairs,
        // and the P values packed in place and stored over the first columns of
        // the S tile. O is rescaled afterwards, when the registers are free.
        uint32_t r[128];
        tmem_ld_x64x2(s_tm, s_tm + 64, r);
        if (lim < kBN) {
  #pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) r[c] = 0xff800000u;  // -inf
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  #pragma unroll
        for (int c = 0; c < 128; c += 8) {
  #pragma unroll
          for (int i = 0; i < 4; ++i)
            mx[i] = fmax3(mx[i], __uint_as_float(r[c + 2 * i]), __uint_as_float(r[c + 2 * i + 1]));
        }
        const float m_tile = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * sl2;

        const bool need = (m_used != -INFINITY) && (m_tile > m_used + kRescaleSlack);
        const float alpha = need ? ex2_approx(m_used - m_tile) : 1.f;
        if (need) m_used = m_tile;
        if (m_used == -INFINITY) m_used = m_tile;  // first visible scores of this row
        const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;

        const uint64_t negm2 = f2_pack(-m_sub, -m_sub);
        uint64_t acc[4] = {0, 0, 0, 0};
  #pragma unroll
        for (int i = 0; i < 64; ++i) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sl2x2, negm2), x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
          r[2 * i] = __float_as_uint(p0);
          r[2 * i + 1] = __float_as_uint(p1);
        }
        // e4m3 P: four keys per column, keys [0, 128) to columns [0, 32)
  #pragma unroll
        for (int i = 0; i < 32; ++i)
          r[i] = pack_e4m3x2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])) |
                 (pack_e4m3x2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])) << 16);
        tmem_st_x32(s_tm, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        float s0, s1, s2, s3;
        f2_unpack(f2_add(acc[0], acc[1]), s0, s1);
        f2_unpack(f2_add(acc[2], acc[3]), s2, s3);
        l = l * alpha + ((s0 + s1) + (s2 + s3));

        if (__any_sync(kFull, need)) {
          const uint64_t alpha2 = f2_pack(alpha, alpha);
  #pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld_x32(o_tm + c, o);
  #pragma unroll
            for (int i = 0; i < 16; ++i) {
              float lo, hi;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), alpha2), lo, hi);
              o[2 * i] = __float_as_uint(lo);
              o[2 * i + 1] = __float_as_uint(hi);
            }
            tmem_st_x32(o_tm + c, o);
          }
        }
      } else {
        // bf16 inputs, pass 1: row maximum of the raw scores (scale > 0, so the
        // maximum commutes with the scaling), both halves of the row loaded
        // together. The exponentials reload the scores 64 at a time: holding all
        // 128 through that pass, as the e4m3 path does, makes this instance spill.
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        {
          uint32_t r[128];
          tmem_ld_x64x2(s_tm, s_tm + 64, r);
          if (lim < kBN) {
  #pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= lim) r[c] = 0xff800000u;  // -inf
          }
  #pragma unroll
          for (int c = 0; c < 128; c += 8) {
  #pragma unroll
            for (int i = 0; i < 4; ++i)
              mx[i] = fmax3(mx[i], __uint_as_float(r[c + 2 * i]), __uint_as_float(r[c + 2 * i + 1]));
          }
        }
        const float m_tile = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * sl2;

        const bool need = (m_used != -INFINITY) && (m_tile > m_used + kRescaleSlack);
        if (__any_sync(kFull, need)) {
          const float alpha = need ? ex2_approx(m_used - m_tile) : 1.f;
          if (need) {
            l *= alpha;
            m_used = m_tile;
          }
          const uint64_t alpha2 = f2_pack(alpha, alpha);
  #pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t r[32];
            tmem_ld_x32(o_tm + c, r);
  #pragma unroll
            for (int i = 0; i < 16; ++i) {
              float lo, hi;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), alpha2), lo, hi);
              r[2 * i] = __float_as_uint(lo);
              r[2 * i + 1] = __float_as_uint(hi);
            }
            tmem_st_x32(o_tm + c, r);
          }
        }
        if (m_used == -INFINITY) m_used = m_tile;  // first visible scores of this row
        const float m_sub = (m_used == -INFINITY) ? 0.f : m_used;

        // Pass 2: p = 2^(s * scale * log2 e - m), two at a time, row sum in
        // packed pairs; the bf16 pairs of keys [64h, 64h + 64) go to P columns
        // [32h, 32h + 32), which only hold scores this pass has already read.
        const uint64_t negm2 = f2_pack(-m_sub, -m_sub);
        uint64_t acc[4] = {0, 0, 0, 0};
  #pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[64];
          tmem_ld_x64(s_tm + 64 * h, r);
          if (lim < kBN) {
  #pragma unroll
            for (int c = 0; c < 64; ++c)
              if (64 * h + c >= lim) r[c] = 0xff800000u;
          }
          // x = s * scale_log2 - m in place, then 2^x in place (MUFU), then pack + sum
  #pragma unroll
          for (int i = 0; i < 32; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sl2x2, negm2), x0, x1);
            r[2 * i] = __float_as_uint(ex2_approx(x0));
            r[2 * i + 1] = __float_as_uint(ex2_approx(x1));
          }
          uint32_t pk[32];
  #pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = __uint_as_float(r[2 * i]);
            const float p1 = __uint_as_float(r[2 * i + 1]);
            acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st_x32(s_tm + 32 * h, pk);
        }
        float s0, s1, s2, s3;
        f2_unpack(f2_add(acc[0], acc[1]), s0, s1);
        f2_unpack(f2_add(acc[2], acc[3]), s2, s3);
        l += (s0 + s1) + (s2 + s3);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sm.p_full[t]);
    }
    if (!ok) break;
    ok = bounded_wait(&sm.o_full[t], o_cnt & 1, sm.abort_flag, p.err, kSiteOFull);
    ++o_cnt;
    // the staging box is free once this tile's previous TMA store has read it;
    // the barrier below publishes that to the warpgroup
    if (releaser) bulk_wait_group_read<0>();
    // one decision for the whole warpgroup: the epilogue below synchronises its
    // 128 threads on named barriers, which every one of them must reach
    ok = named_bar_and(1 + t, 128, ok);
    if (!ok) break;
    // the last P V of this tile is done: its V tile is free if this tile was its last reader
    // (block-sparse: every V is released by the issuing thread)
    if (!SP && releaser && last_reader(it, nkv - 1) == t)
      mbar_arrive(&sm.kv_empty[(ring_base + 2 * (nkv - 1) + 1) % C::kStages]);
    tc_fence_after();

    // Epilogue: O / l to bf16, O's TMEM columns released once read, then stored.
    // (e4m3 V: O carries V's per-head scale)
    // (a row that saw no key, possible under a block mask: o = 0, lse = -inf)
    const float inv_l = (l > 0.f) ? (F8 ? __ldg(p.sv + it.bh) : 1.f) / l : 0.f;
    const uint64_t inv_l2 = f2_pack(inv_l, inv_l);
    // O leaves through the TMA unit in 64-column boxes, staged in shared memory
    // in the 128-byte swizzle of the map (16-byte chunk u of a row at u ^ (row & 7));
    // one thread stores each box, and rows beyond N are outside the map.
    // Columns [0, 64) go straight to the box; the rest wait in registers until
    // the first box has been read.
    uint4* rowp = reinterpret_cast<uint4*>(sm.ostage + t * C::kOStageBytes + row * 128);
    uint32_t w[D > 64 ? (D - 64) / 2 : 1];
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t r[32];
      tmem_ld_x32(o_tm + c, r);
      uint32_t h[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float lo, hi;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), inv_l2), lo, hi);
        h[i] = pack_bf16x2(lo, hi);
      }
      if (c < 64) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          rowp[(c / 8 + u) ^ (row & 7)] = make_uint4(h[4 * u], h[4 * u + 1], h[4 * u + 2], h[4 * u + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[(c - 64) / 2 + i] = h[i];
      }
    }
    tc_fence_before();
    mbar_arrive(&sm.o_empty[t]);
    uint8_t* ost = sm.ostage + t * C::kOStageBytes;
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      if (c > 0) {
        if (releaser) bulk_wait_group_read<0>();  // the previous box has been read
        named_bar_sync(1 + t, 128);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          rowp[u ^ (row & 7)] = make_uint4(w[32 * (c - 1) + 4 * u], w[32 * (c - 1) + 4 * u + 1],
                                           w[32 * (c - 1) + 4 * u + 2], w[32 * (c - 1) + 4 * u + 3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + t, 128);
      if (releaser) {
        tma_store_3d(*sm.tmo, ost, 64 * c, it.row(t), it.bh);
        bulk_commit_group();
      }
    }
    if (q_row < p.N)
      p.lse[static_cast<size_t>(it.bh) * p.N + q_row] = (l > 0.f) ? (m_used + log2f(l)) * kLn2 : -INFINITY;
  }
  if (releaser) bulk_wait_group<0>();  // every O store complete before the CTA can exit
#ifdef FA_DEBUG
  if (releaser) {
    sm.dbg[10 + t] = ring_next;
    sm.dbg[12 + t] = s_cnt;
    sm.dbg[14 + t] = o_cnt;
  }
#endif
}

// Block-sparse step lists: one warp per (mask head, Q-tile pair) compacts, in
// increasing order, the K/V tiles kept by either Q tile of the pair (the block
// mask and, under the causal mask, j <= the Q tile's index), and counts the
// union's steps and the steps each Q tile keeps.
__global__ void __launch_bounds__(32) sparse_list_kernel(const uint8_t* __restrict__ mask, int tiles, int pairs,
                                                         int causal, uint32_t* __restrict__ list,
                                                         int* __restrict__ cnt, int* __restrict__ next_item) {
  const int pair = blockIdx.x, mh = blockIdx.y, lane = threadIdx.x;
  if (pair == 0 && mh == 0 && lane == 0) *next_item = 0;  // the forward's run-time item counter
  const uint8_t* mk = mask + static_cast<size_t>(mh) * tiles * tiles;
  const int i0 = 2 * pair, i1 = 2 * pair + 1;
  uint32_t* out = list + (static_cast<size_t>(mh) * pairs + pair) * tiles;
  int n = 0, n0 = 0, n1 = 0;
  for (int base = 0; base < tiles; base += 32) {
    const int j = base + lane;
    bool a0 = false, a1 = false;
    if (j < tiles) {
      a0 = mk[static_cast<size_t>(i0) * tiles + j] != 0 && (!causal || j <= i0);
      a1 = i1 < tiles && mk[static_cast<size_t>(i1) * tiles + j] != 0 && (!causal || j <= i1);
    }
    const uint32_t keep = __ballot_sync(0xffffffffu, a0 || a1);
    if (a0 || a1)
      out[n + __popc(keep & ((1u << lane) - 1u))] =
          static_cast<uint32_t>(j) | (a0 ? 1u << 16 : 0u) | (a1 ? 1u << 17 : 0u);
    n += __popc(keep);
    n0 += __popc(__ballot_sync(0xffffffffu, a0));
    n1 += __popc(__ballot_sync(0xffffffffu, a1));
  }
  if (lane == 0) {
    int* c = cnt + 3 * (static_cast<size_t>(mh) * pairs + pair);
    c[0] = n;
    c[1] = n0;
    c[2] = n1;
  }
}

template <int D, bool F8, bool SP>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using C = Cfg<D, F8>;
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve<D, F8>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.q_full[t], 1);
      mbar_init(&sm.q_empty[t], 1);
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_full[t], 128);
      mbar_init(&sm.o_full[t], 1);
      mbar_init(&sm.o_empty[t], 128);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    mbar_init(sm.mma_done, 1);
    for (int e = 0; e < kItemSlots; ++e) {
      mbar_init(&sm.item_full[e], 1);
      mbar_init(&sm.item_empty[e], kItemReaders);
    }
    *sm.abort_flag = 0;
    *const_cast<const CUtensorMap**>(sm.tmo) = &tm_o;
    for (int i = 0; i < 16; ++i) sm.dbg[i] = 0;
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
    if (lane == 0) load_role<D, F8, SP>(&tm_q, &tm_k, &tm_v, sm, p);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      if constexpr (SP)
        mma_role_sparse<D>(sm, tmem, p);
      else
        mma_role<D, F8, SP>(sm, tmem, p);
    }
  } else {
    softmax_role<D, F8, SP>(sm, tmem, p, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
#ifdef FA_DEBUG
  // Protocol check: the roles walked the same items (ring positions), and per
  // tile the MMA consumed one Q per item and one P per S the softmax saw, and
  // produced one O per item the epilogue read.
  if (threadIdx.x == 0 && *sm.abort_flag == 0) {
    const uint32_t* d = sm.dbg;
    bool good = d[0] == d[3] && d[0] == d[10] && d[0] == d[11];
    for (int t = 0; t < 2; ++t)
      good = good && d[1 + t] == d[4 + t] && d[4 + t] == d[8 + t] && d[6 + t] == d[12 + t] && d[8 + t] == d[14 + t];
    if (!good) record_check(p.err, kSiteCheckFwd);
  }
#endif
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool F8, bool SP>
fa_status launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                 FwdParams prm, int B, int H,
                 int N, int causal, float scale, cudaStream_t stream, int num_sms) {
  using C = Cfg<D, F8>;
  const uint64_t bh = static_cast<uint64_t>(B) * H;
  const int num_pairs = (N + 2 * kBM - 1) / (2 * kBM);
  const long long items = static_cast<long long>(bh) * num_pairs;
  prm.N = N;
  prm.BH = static_cast<int>(bh);
  prm.num_pairs = num_pairs;
  prm.num_items = static_cast<int>(items);
  prm.causal = causal ? 1 : 0;
  // Which tile of a causal pair goes first is a matter of how the two tiles'
  // chains overlap at item boundaries. Measured: the swapped order (the later
  // tile first) is faster for e4m3 (+2 %) and d = 64 (+6 %); for bf16 d = 128 it
  // lost 1-3 % while the epilogue stored O from registers, and gains 0.2-1 %
  // since O leaves through TMA stores.
  prm.swap_tiles = (!SP && causal) ? 1 : 0;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.tiles = (N + kBM - 1) / kBM;
  prm.H = H;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D, F8, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) {
    set_error_text("cudaFuncSetAttribute(fwd_kernel)", e);
    return FA_ERR_CUDA;
  }
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  fwd_kernel<D, F8, SP><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("fwd_kernel launch", e);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

template <int D>
fa_status launch_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                      int causal, float scale, cudaStream_t stream, unsigned int* err, int num_sms,
                      const uint32_t* list = nullptr, const int* cnt = nullptr, int mask_heads = 0,
                      int* next_item = nullptr) {
  CUtensorMap tq, tk, tv, to;
  const uint64_t bh = static_cast<uint64_t>(B) * H;
  if (!encode_bf16_map(&tq, q, D, N, bh, kBM) || !encode_bf16_map(&tk, k, D, N, bh, kBN) ||
      !encode_bf16_map(&tv, v, D, N, bh, kBN) || !encode_bf16_map(&to, o, D, N, bh, kBM))
    return FA_ERR_CUDA;
  FwdParams prm{};
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.err = err;
  prm.list = list;
  prm.cnt = cnt;
  prm.next_item = next_item;
  prm.mask_heads = mask_heads;
  if (list != nullptr) return launch<D, false, true>(tq, tk, tv, to, prm, B, H, N, causal, scale, stream, num_sms);
  return launch<D, false, false>(tq, tk, tv, to, prm, B, H, N, causal, scale, stream, num_sms);
}

}  // namespace

fa_status launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                     int causal, float scale, cudaStream_t stream, unsigned int* err, int num_sms) {
  if (d == 128) return launch_bf16<128>(q, k, v, o, lse, B, H, N, causal, scale, stream, err, num_sms);
  if (d == 64) return launch_bf16<64>(q, k, v, o, lse, B, H, N, causal, scale, stream, err, num_sms);
  return FA_ERR_UNSUPPORTED;
}

fa_status launch_fwd_sparse(const void* q, const void* k, const void* v, const uint8_t* mask, int mask_heads, void* o,
                            float* lse, int B, int H, int N, int d, int causal, float scale, uint32_t* list_ws,
                            int* cnt_ws, cudaStream_t stream, unsigned int* err, int num_sms) {
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const int tiles = (N + kBM - 1) / kBM;
  const int pairs = (N + 2 * kBM - 1) / (2 * kBM);
  int* next_item = cnt_ws + 3 * static_cast<size_t>(pairs) * mask_heads;
  sparse_list_kernel<<<dim3(static_cast<unsigned>(pairs), static_cast<unsigned>(mask_heads)), 32, 0, stream>>>(
      mask, tiles, pairs, causal ? 1 : 0, list_ws, cnt_ws, next_item);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error_text("sparse_list_kernel launch", e);
    return FA_ERR_CUDA;
  }
  if (d == 128)
    return launch_bf16<128>(q, k, v, o, lse, B, H, N, causal, scale, stream, err, num_sms, list_ws, cnt_ws, mask_heads,
                            next_item);
  return launch_bf16<64>(q, k, v, o, lse, B, H, N, causal, scale, stream, err, num_sms, list_ws, cnt_ws, mask_heads,
                         next_item);
}

fa_status launch_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale, const float* k_scale,
                         const float* v_scale, void* o, float* lse, int B, int H, int N, int d, int causal,
                         float scale, int v_pitch, cudaStream_t stream, unsigned int* err, int num_sms) {
  if (d != 128) return FA_ERR_UNSUPPORTED;
  CUtensorMap tq, tk, tv, to;
  const uint64_t bh = static_cast<uint64_t>(B) * H;
  if (!encode_bf16_map(&to, o, 128, N, bh, kBM)) return FA_ERR_CUDA;
  // Q, K: [BH][N][128] bytes; V^T: [BH][128][v_pitch] bytes, keys inner
  if (!encode_u8_map(&tq, q8, 128, N, bh, kBM, 128) || !encode_u8_map(&tk, k8, 128, N, bh, kBN, 128) ||
      !encode_u8_map(&tv, vt8, N, 128, bh, 128, static_cast<uint64_t>(v_pitch)))
    return FA_ERR_CUDA;
  FwdParams prm{};
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.err = err;
  prm.sq = q_scale;
  prm.sk = k_scale;
  prm.sv = v_scale;
  return launch<128, true, false>(tq, tk, tv, to, prm, B, H, N, causal, scale, stream, num_sms);
}

}  // namespace fa
