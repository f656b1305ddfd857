// Host-side interfaces between the translation units of libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/fa.h"

namespace fa {

// Encode a 3-D bf16 tensor map over [outer][rows][d] with a {64, box_rows, 1}
// box and 128-byte swizzle. Returns false (and sets the error text) on failure.
bool encode_bf16_map(CUtensorMap* map, const void* base, uint64_t d, uint64_t rows, uint64_t outer,
                     uint32_t box_rows);
// A 3-D uint8 (e4m3 codes) map over [outer][rows][inner], rows row_pitch bytes
// apart (a multiple of 16), {128, box_rows, 1} box, 128-byte swizzle.
bool encode_u8_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t outer,
                   uint32_t box_rows, uint64_t row_pitch);
// The same over fp32 elements with a {32, box_rows, 1} box (128-byte rows).
bool encode_f32_map(CUtensorMap* map, const void* base, uint64_t d, uint64_t rows, uint64_t outer,
                    uint32_t box_rows);

// Record the text of a CUDA failure for fa_last_error_string.
void set_error_text(const char* what, cudaError_t err);
void set_error_text(const char* what, const char* detail);

// Record why a call was rejected (the failed check, as source text) and return `status`.
fa_status reject(fa_status status, const char* failed_check);
#define FA_REJECT_IF(cond, status)                  \
  do {                                              \
    if (cond) return ::fa::reject((status), #cond); \
  } while (0)

// The current device, checked to be compute capability 10.3 (FA_ERR_UNSUPPORTED otherwise).
fa_status checked_device(int* dev);

// Argument checks shared by fa_decode and fa_decode_noalloc (pointers, alignment, sizes, d, splits).
fa_status check_decode_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens,
                            const void* o, const float* lse, int B, int H, int L, int d, int num_splits);

// Device error word of the current device (see fa_common.cuh).
unsigned int* device_error_word();

// num_sms: multiprocessor count of the current device (the persistent grid size).
fa_status launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                     int causal, float scale, cudaStream_t stream, unsigned int* err, int num_sms);

// e4m3 block quantization (d = 128); amax_ws: fp32 [B*H][ceil(N/128)] scratch.
fa_status launch_quantize_fp8(const void* x, const float* signs, void* codes, float* scales, int B, int H, int N,
                              int per_head, int transpose, int v_pitch, float* amax_ws, cudaStream_t stream);

// Block-sparse forward: mask [mask_heads][T][T] bytes on the device, T = ceil(N / 128);
// list_ws: uint32 [mask_heads][ceil(N/256)][T] and cnt_ws: int [mask_heads][ceil(N/256)][3] + 1 scratch
// (the last int is the forward's run-time item counter).
fa_status launch_fwd_sparse(const void* q, const void* k, const void* v, const uint8_t* mask, int mask_heads, void* o,
                            float* lse, int B, int H, int N, int d, int causal, float scale, uint32_t* list_ws,
                            int* cnt_ws, cudaStream_t stream, unsigned int* err, int num_sms);

// The e4m3 forward (d = 128): q8, k8 [B*H][N][128] bytes, vt8 [B*H][128][v_pitch]
// bytes, scales [B*H][ceil(N/128)] for Q and K and [B*H] for V.
fa_status launch_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale, const float* k_scale,
                         const float* v_scale, void* o, float* lse, int B, int H, int N, int d, int causal,
                         float scale, int v_pitch, cudaStream_t stream, unsigned int* err, int num_sms);

fa_status launch_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens, void* o,
                        float* lse, int B, int H, int L, int d, int num_splits, float* ws_o, float* ws_lse,
                        cudaStream_t stream);

// The log-sum-exp merge of fa_decode over `heads` (batch, head) rows of partials.
fa_status launch_decode_merge(const float* ws_o, const float* ws_lse, void* o, float* lse, long long heads, int d,
                              int num_splits, cudaStream_t stream);

// The GQA split kernel: partials of [B][Hq][num_splits] into ws_o / ws_lse.
fa_status launch_decode_gqa_split(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens,
                                  int B, int Hq, int Hkv, int L, int d, int num_splits, float* ws_o, float* ws_lse,
                                  cudaStream_t stream, unsigned int* err);

// dq_acc: fp32 [B*H*N*d] scratch (zeroed by the call), delta: fp32 [B*H*N] scratch.
fa_status launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, float* dq_acc,
                     float* delta, cudaStream_t stream, unsigned int* err);

fa_status launch_selftest_mma(int mode, const void* a, const void* b, float* d, int n, int k, cudaStream_t stream,
                              unsigned int* err);
fa_status launch_selftest_wait(unsigned int timeout_us, cudaStream_t stream, unsigned int* err);

}  // namespace fa
