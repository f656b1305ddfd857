// Tile geometry and the two tensor-core products of the attention forward,
// shared by the prefill kernel and the tensor-core self-test.
//
// Shared-memory tiles are 128 rows of bf16, written by TMA with 128-byte
// swizzle: each 64-element (128-byte) slice of d forms a 16 KB "chunk" of
// 128 rows x 128 bytes, and chunks are stored one after the other.
#pragma once

#include <cstdint>

#include "sm103.cuh"

namespace fa {

constexpr int kBM = 128;               // query rows per Q tile (= TMEM lanes)
constexpr int kBN = 128;               // keys per K/V tile
constexpr int kChunkBytes = 128 * 128; // one 128-row x 128-byte swizzle chunk

// Each product builds its operands' shared-memory descriptors once; a K step
// adds its byte offset / 16 to the 14-bit address field. Shared-memory
// addresses stay below 256 KB, so the field never carries into the next one.
// (The issuing thread is on the critical path of the kernels: fewer
// instructions per tcgen05.mma measurably shorten it.)
__device__ __forceinline__ constexpr uint64_t desc_step(uint32_t byte_offset) { return byte_offset >> 4; }

// S(tmem, 128 x 128 fp32) = Q(smem, 128 x D, K-major) * K(smem, 128 x D, K-major)^T
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, false);
  const uint64_t qd = smem_desc_sw128(q_smem, 16, 1024);
  const uint64_t kd = smem_desc_sw128(k_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    // 16 bf16 = 32 bytes of the 128-byte swizzled row; 4 steps per chunk
    const uint64_t off = desc_step(static_cast<uint32_t>((kk / 4) * kChunkBytes + (kk % 4) * 32));
    umma_ss(s_tmem, qd + off, kd + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O(tmem, 128 x D fp32) (+)= P(tmem, 128 x 128 bf16, packed pairs) * V(smem, 128 keys x D, MN-major).
// P keys 0-63 sit in TMEM columns [p, p + 32) and keys 64-127 in
// [p + 32 + p_gap, p + 64 + p_gap); each K-step of 16 keys takes 8 columns.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem, bool accumulate,
                                         uint32_t p_gap = 0) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, false, true);
  const uint64_t vd = smem_desc_sw128(v_smem, kChunkBytes, 1024);
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk) {
    // 16 keys = two 8-row groups of 1024 bytes of V
    umma_ts(o_tmem, p_tmem + static_cast<uint32_t>(kk * 8) + (kk >= 4 ? p_gap : 0u),
            vd + desc_step(static_cast<uint32_t>(kk * 2048)), idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// D(tmem, 128 x N fp32) = A(smem, 128 x 128, MN-major) * B(smem, 128 x N, MN-major).
// A is stored transposed (rows are the contraction index, the 128 M values of a
// row contiguous in two 64-element chunks) and B likewise (rows are the
// contraction index, N contiguous): the dQ = dS K product of the backward pass,
// with dS held as dS^T.
template <int N>
__device__ __forceinline__ void issue_mn_mn(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, N, true, true);
  const uint64_t ad = smem_desc_sw128(a_smem, kChunkBytes, 1024);
  const uint64_t bd = smem_desc_sw128(b_smem, kChunkBytes, 1024);
#pragma unroll
  for (int kk = 0; kk < 128 / 16; ++kk) {
    // 16 contraction rows = two 8-row groups of 1024 bytes in both operands
    const uint64_t off = desc_step(static_cast<uint32_t>(kk * 2048));
    umma_ss(d_tmem, ad + off, bd + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// FP8 (e4m3) forms of the two products for d = 128: every 128-row tile row is
// 128 bytes, one swizzle chunk; one instruction covers K = 32 (32 bytes).
// S(tmem, 128 x 128 fp32) = Q(smem, 128 x 128 e4m3, K-major) * K(smem, 128 x 128 e4m3, K-major)^T
__device__ __forceinline__ void issue_qk_f8(uint32_t s_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kBN);
  const uint64_t qd = smem_desc_sw128(q_smem, 16, 1024);
  const uint64_t kd = smem_desc_sw128(k_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint64_t off = desc_step(static_cast<uint32_t>(kk * 32));
    umma_ss_f8(s_tmem, qd + off, kd + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O(tmem, 128 x 128 fp32) (+)= P(tmem, 128 x 128 e4m3, four keys per column) * V,
// V given as V^T (smem, 128 rows of d x 128 keys e4m3, K-major). Keys 32kk..32kk+31
// of P sit in TMEM columns [p + 8kk, p + 8kk + 8).
__device__ __forceinline__ void issue_pv_f8(uint32_t o_tmem, uint32_t p_tmem, uint32_t vt_smem, bool accumulate) {
  constexpr uint32_t idesc = idesc_e4m3_f32(kBM, 128);
  const uint64_t vd = smem_desc_sw128(vt_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    umma_ts_f8(o_tmem, p_tmem + static_cast<uint32_t>(kk * 8), vd + desc_step(static_cast<uint32_t>(kk * 32)), idesc,
               (accumulate || kk > 0) ? 1u : 0u);
  }
}

}  // namespace fa
