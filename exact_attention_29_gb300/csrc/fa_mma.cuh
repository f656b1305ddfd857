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

// S(tmem, 128 x 128 fp32) = Q(smem, 128 x D, K-major) * K(smem, 128 x D, K-major)^T
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    // 16 bf16 = 32 bytes of the 128-byte swizzled row; 4 steps per chunk
    const uint32_t off = static_cast<uint32_t>((kk / 4) * kChunkBytes + (kk % 4) * 32);
    umma_ss(s_tmem, smem_desc_sw128(q_smem + off, 16, 1024), smem_desc_sw128(k_smem + off, 16, 1024), idesc,
            kk > 0 ? 1u : 0u);
  }
}

// O(tmem, 128 x D fp32) (+)= P(tmem, 128 x 128 bf16, packed pairs) * V(smem, 128 keys x D, MN-major).
// P keys 0-63 sit in TMEM columns [p, p + 32) and keys 64-127 in
// [p + 32 + p_gap, p + 64 + p_gap); each K-step of 16 keys takes 8 columns.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem, bool accumulate,
                                         uint32_t p_gap = 0) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBM, D, false, true);
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk) {
    // 16 keys = two 8-row groups of 1024 bytes of V
    umma_ts(o_tmem, p_tmem + static_cast<uint32_t>(kk * 8) + (kk >= 4 ? p_gap : 0u),
            smem_desc_sw128(v_smem + static_cast<uint32_t>(kk * 2048), kChunkBytes, 1024), idesc,
            (accumulate || kk > 0) ? 1u : 0u);
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
#pragma unroll
  for (int kk = 0; kk < 128 / 16; ++kk) {
    // 16 contraction rows = two 8-row groups of 1024 bytes in both operands
    umma_ss(d_tmem, smem_desc_sw128(a_smem + static_cast<uint32_t>(kk * 2048), kChunkBytes, 1024),
            smem_desc_sw128(b_smem + static_cast<uint32_t>(kk * 2048), kChunkBytes, 1024), idesc, kk > 0 ? 1u : 0u);
  }
}

// FP8 (e4m3) forms of the two products for d = 128: every 128-row tile row is
// 128 bytes, one swizzle chunk; one instruction covers K = 32 (32 bytes).
// S(tmem, 128 x 128 fp32) = Q(smem, 128 x 128 e4m3, K-major) * K(smem, 128 x 128 e4m3, K-major)^T
__device__ __forceinline__ void issue_qk_f8(uint32_t s_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kBN);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint32_t off = static_cast<uint32_t>(kk * 32);
    umma_ss_f8(s_tmem, smem_desc_sw128(q_smem + off, 16, 1024), smem_desc_sw128(k_smem + off, 16, 1024), idesc,
               kk > 0 ? 1u : 0u);
  }
}

// O(tmem, 128 x 128 fp32) (+)= P(tmem, 128 x 128 e4m3, four keys per column) * V,
// V given as V^T (smem, 128 rows of d x 128 keys e4m3, K-major). Keys 32kk..32kk+31
// of P sit in TMEM columns [p + 8kk, p + 8kk + 8).
__device__ __forceinline__ void issue_pv_f8(uint32_t o_tmem, uint32_t p_tmem, uint32_t vt_smem, bool accumulate) {
  constexpr uint32_t idesc = idesc_e4m3_f32(kBM, 128);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    umma_ts_f8(o_tmem, p_tmem + static_cast<uint32_t>(kk * 8),
               smem_desc_sw128(vt_smem + static_cast<uint32_t>(kk * 32), 16, 1024), idesc,
               (accumulate || kk > 0) ? 1u : 0u);
  }
}

}  // namespace fa
