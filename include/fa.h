/*
 * fa.h — C ABI of the GB300 exact-attention library (libfa.so).
 *
 * Two operations, both exact (no approximation beyond floating-point rounding):
 *
 *   fa_fwd     fused prefill attention O = softmax(scale * Q K^T [+ causal mask]) V
 *              with the per-row log-sum-exp written out; the N x N score and
 *              probability matrices never reach device memory.
 *   fa_decode  Flash-Decoding: one query token per (batch, head) against a long
 *              KV cache, split along the keys, the per-split summaries merged
 *              by the log-sum-exp combine (fa_decode_gqa: query heads grouped
 *              over shared K/V heads).
 *   fa_bwd     gradients of fa_fwd, recomputing P from the saved log-sum-exp.
 *
 * Workspaces: calls that need scratch memory take it, ordered on `stream`,
 * from a memory pool the library creates on each device (cudaMemPoolCreate)
 * and give it back on the same stream before returning; the pool keeps up to
 * 4 GiB mapped between calls, so repeated calls do not map memory again. A
 * block is reused by the stream that released it (or across an event
 * dependency the caller made), never by making one stream wait for another:
 * a caller that pipelines calls over several streams keeps one workspace per
 * stream.
 *
 * Conventions for every call:
 *   - Tensor arguments are DEVICE pointers (memory of the current CUDA device),
 *     owned by the caller, contiguous, row-major in the layout stated. The
 *     library keeps no reference to them after the call returns.
 *   - bf16 means IEEE bfloat16 (torch.bfloat16); outputs are rounded to nearest
 *     even. Arithmetic is fp32 (tensor-core accumulation, softmax statistics).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls only
 *     enqueue work on it and return; results are ready when the stream is.
 *   - Argument errors are reported before anything is enqueued. Launch errors
 *     are returned at once. Errors found while the kernels run (a bounded wait
 *     inside a kernel that ran out) are reported by fa_check_device_error.
 *   - The library is thread-safe; it holds no state besides per-device lookups.
 */
#ifndef FA_H_
#define FA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (declared here so the header needs no CUDA headers). */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, misaligned pointer, bad scale */
  FA_ERR_UNSUPPORTED = 2,  /* valid but not implemented here (head dim other than 64 or 128, no sm_103 device) */
  FA_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed; see fa_last_error_string() */
  FA_ERR_TIMEOUT = 4,      /* a kernel's bounded wait ran out; the kernel stopped and its outputs are undefined */
  FA_ERR_CHECK = 5         /* a libfa_debug.so build only: a kernel's roles disagreed on their protocol counts */
} fa_status;

/*
 * Prefill (forward) attention.
 *
 * Defines: "已有的几种大模型上下文支持情况" (cicada blog) §1.2
 *   Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V, §1.3 (causal mask sets
 *   future positions to -inf) and §3.2 (FlashAttention-2: tiles of Q stay on
 *   chip, K/V tiles stream through, running max m and normaliser l, one divide
 *   by l at the end, L_i = m_i + ln l_i written out); CMU 15-779 Lecture 5
 *   notes §5.1 (the tiled forward) and §6.2 (causal block skipping).
 *
 *   q, k, v  bf16 [B][H][N][d], d contiguous. 16-byte aligned.
 *   o        bf16 [B][H][N][d] output.
 *   lse      fp32 [B][H][N] output: natural log of sum_j exp(scale * q_i . k_j)
 *            over the keys row i sees.
 *   B, H, N  >= 1 (N need not be a multiple of any tile size).
 *   d        64 or 128 (FA_ERR_UNSUPPORTED otherwise).
 *   causal   0: every row sees all N keys; 1: row i sees keys 0..i.
 *   scale    > 0 and finite, usually 1/sqrt(d).
 * Errors: FA_ERR_INVALID_ARG for null/misaligned pointers, sizes < 1, a bad
 *   scale, or sizes whose counts overflow (B*H and B*H*ceil(N/256) work items
 *   above 2^31 - 1, ceil(N/256) above 65535); FA_ERR_UNSUPPORTED for d;
 *   FA_ERR_CUDA if the launch fails.
 */
fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N, int d,
                 int causal, float scale, fa_stream_t stream);

/*
 * Prefill from and to host memory: fa_fwd with the host<->device copies inside
 * the call. q, k, v and o, lse are HOST pointers with the layouts of fa_fwd.
 * On `stream` the call enqueues: device buffers for q, k, v, o and lse from
 * the library's stream-ordered pool; one cudaMemcpyAsync per input
 * (host to device); the forward; one cudaMemcpyAsync per output (device to
 * host); the release of the buffers. It returns without waiting.
 *
 * Ownership: the host buffers must stay valid, and the inputs unchanged, until
 * the stream has passed the call (cudaStreamSynchronize or an event). With
 * page-locked (pinned) host memory the copies are asynchronous and the calls
 * of successive steps on different streams overlap their copies with each
 * other's kernels; with pageable memory the copies still complete correctly but
 * synchronise with the host.
 * Errors: as fa_fwd (16-byte alignment applies to the host pointers too);
 *   FA_ERR_INVALID_ARG also when the runtime knows one of the five pointers as
 *   device memory; FA_ERR_CUDA if a copy or the pool allocation fails.
 */
fa_status fa_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N, int d,
                      int causal, float scale, fa_stream_t stream);

/*
 * Block-sparse prefill forward.
 *
 * Defines: "FlashAttention 完全拆解（一）", block-sparse extension: given a
 *   block-level mask, the S_ij blocks it removes are skipped (never loaded,
 *   never multiplied), so IO and work shrink with the mask's density.
 *
 *   q, k, v, o, lse, B, H, N, d, causal, scale: as fa_fwd.
 *   mask     DEVICE bytes [mask_heads][T][T], T = ceil(N / 128) (the kernel's
 *            tile): key j is visible to query i when
 *            mask[i / 128][j / 128] != 0 and, if causal, j <= i.
 *   mask_heads  1 (one mask for every head) or H (head h uses mask h).
 * A row with no visible key gets o = 0 and lse = -inf.
 * Workspace: mask_heads*ceil(N/256)*(T+3)*4 + 4 bytes of stream-ordered
 *   device memory (the per Q-tile-pair step lists and counts a first small
 *   kernel builds, and the counter that hands out work items at run time).
 * Errors: as fa_fwd; FA_ERR_INVALID_ARG also for a NULL mask, another
 *   mask_heads, or T > 65535 (N > 8,388,480).
 */
fa_status fa_fwd_sparse(const void *q, const void *k, const void *v, const uint8_t *mask, int mask_heads, void *o,
                        float *lse, int B, int H, int N, int d, int causal, float scale, fa_stream_t stream);

/*
 * Work plan of fa_fwd_sparse (host only; mask is a HOST pointer, same layout):
 * pairs_allowed = (Q tile, K/V tile) block pairs the mask (and the causal
 * rule) keeps, over all B*H heads; pairs_computed = pairs whose products the
 * kernel runs: each Q tile computes exactly the pairs its mask keeps (the two
 * Q tiles of a work item share the copies of the union of their K/V tiles).
 */
fa_status fa_fwd_sparse_plan(const uint8_t *mask, int mask_heads, int B, int H, int N, int causal,
                             long long *pairs_allowed, long long *pairs_computed);

/*
 * FP8 (e4m3) block quantization for fa_fwd_fp8, with incoherent processing.
 *
 * Defines: "已有的几种大模型上下文支持情况" (cicada blog) §4.4 (FA-3's FP8
 *   support): §4.4.1 every tile entering a tensor-core product has its own
 *   scale factor; §4.4.2 Q and K are multiplied by a random orthogonal matrix
 *   R (a Hadamard matrix with random signs) so that outlier dimensions are
 *   spread out, leaving the scores unchanged: (QR)(KR)^T = Q K^T.
 *
 *   x       bf16 [B][H][N][d], d = 128 (FA_ERR_UNSUPPORTED otherwise).
 *   signs   fp32 [d] of +1 / -1, or NULL for no rotation. With signs, row x
 *           becomes x R with R = diag(signs) H_d / sqrt(d) (H_d Sylvester-
 *           Hadamard). Use the same signs for Q and K, none for V.
 *   codes   e4m3 bytes: [B][H][N][d] (transpose = 0) or [B][H][d][v_pitch]
 *           (transpose = 1, V^T for fa_fwd_fp8; v_pitch >= N, a multiple of 16;
 *           bytes beyond N in a row are not written).
 *   scales  fp32: [B][H][ceil(N/128)] (per_head = 0, one per 128-row tile) or
 *           [B][H] (per_head = 1). scale = max |value| / 448 over the tile
 *           (1 for an all-zero tile); code = e4m3(value / scale), rounded to
 *           nearest even, saturating.
 * Workspace: B*H*ceil(N/128)*4 bytes of stream-ordered device memory.
 * Errors: as fa_fwd.
 */
fa_status fa_quantize_fp8(const void *x, const float *signs, void *codes, float *scales, int B, int H, int N, int d,
                          int per_head, int transpose, int v_pitch, fa_stream_t stream);

/*
 * FP8 prefill forward (FA-3 style, "已有的几种大模型上下文支持情况" §4.4).
 *
 *   q8, k8   e4m3 [B][H][N][128] (rotated by the same R), tile scales
 *            q_scale, k_scale fp32 [B][H][ceil(N/128)] (fa_quantize_fp8,
 *            per_head = 0).
 *   vt8      e4m3 V^T [B][H][128][v_pitch], v_scale fp32 [B][H]
 *            (fa_quantize_fp8, per_head = 1, transpose = 1).
 *   o, lse, B, H, N, causal, scale: as fa_fwd; d must be 128.
 * Computes softmax(scale * Q^ K^T [+ causal mask]) V^ over the dequantized
 * inputs, with both products on e4m3 tensor cores: S tiles carry the product
 * of their Q and K tile scales, P is rounded to e4m3 for the P V product (the
 * normaliser l sums the fp32 values), O carries V's scale. An approximation of
 * fa_fwd: the e4m3 rounding of P is its only error beyond the inputs'.
 * Errors: as fa_fwd; FA_ERR_INVALID_ARG also for v_pitch < N or not a
 * multiple of 16.
 */
fa_status fa_fwd_fp8(const void *q8, const void *k8, const void *vt8, const float *q_scale, const float *k_scale,
                     const float *v_scale, void *o, float *lse, int B, int H, int N, int d, int causal, float scale,
                     int v_pitch, fa_stream_t stream);

/*
 * Backward pass (gradients of fa_fwd) with recomputation.
 *
 * Defines: CMU 15-779 Lecture 5 notes §7.1-7.4 and "FlashAttention 完全拆解
 *   （一）", backward section: with S' = scale Q K^T (+ causal mask),
 *   P = softmax(S'), O = P V and the upstream gradient dO,
 *     dV = P^T dO, dP = dO V^T, dS = P * (dP - D) with D_i = dO_i . O_i,
 *     dQ = scale dS K, dK = scale dS^T Q.
 *   P is recomputed from the forward's per-row log-sum-exp, block by block;
 *   K/V blocks form the outer loop (dK, dV accumulate on chip) and every block
 *   adds its share of dQ with atomic additions in fp32.
 *
 *   q, k, v, o, dout  bf16 [B][H][N][d] (o and lse are fa_fwd's outputs for
 *                     the same q, k, v, causal, scale). 16-byte aligned.
 *   lse      fp32 [B][H][N], natural log.
 *   dq, dk, dv  bf16 [B][H][N][d] outputs.
 *   B, H, N, d, causal, scale: as fa_fwd.
 * Workspace: B*H*N*(d+1)*4 bytes of stream-ordered device memory (the fp32
 *   dQ accumulator and D), see "Workspaces" below.
 * Errors: as fa_fwd.
 */
fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
                 void *dq, void *dk, void *dv, int B, int H, int N, int d, int causal, float scale,
                 fa_stream_t stream);

/*
 * Atomic work plan of fa_bwd (host only): with square tiles of `block` rows,
 * the number of fp32 additions into dQ, i.e. for every K/V tile, the rows of
 * every Q tile that sees it times d. Without the mask this is
 * ceil(N/block) * N * d (CMU 15-779 Lecture 5 notes §7.4). fa_bwd uses 128.
 */
fa_status fa_bwd_plan(int N, int d, int block, int causal, long long *dq_atomic_adds);

/*
 * Decode attention (Flash-Decoding).
 *
 * Defines: CMU 15-779 Lecture 5 notes §8.4 (split K/V along the sequence into
 *   S views; one thread block per split computes a partial result and its
 *   log-sum-exp; a small reduction kernel reweights the partials by their
 *   log-sum-exp), §4.4-4.5 (the combine operator on (m, l, o)) and §8.2 (the
 *   cached step equals the last row of the causal recomputation).
 *
 *   q        bf16 [B][H][d], the single new query of each (batch, head).
 *   k_cache, v_cache  bf16 [B][H][L][d]; L is the cache capacity.
 *   seqlens  DEVICE int32 [B]; sequence b uses cache entries 0..seqlens[b]-1.
 *            Values must lie in 1..L (entries outside are clamped in-kernel to
 *            0..L; a length of 0 gives lse = -inf and o = 0).
 *   o        bf16 [B][H][d] output; lse fp32 [B][H] output (natural log).
 *   d        64 or 128. scale is fixed at 1/sqrt(d).
 *   num_splits  1..64: keys of each sequence are cut into num_splits chunks of
 *            ceil(len/num_splits) rounded up to a multiple of 64 keys.
 * Workspace: B*H*num_splits*(d+1)*4 bytes of stream-ordered device memory,
 *   see "Workspaces" below.
 * Errors: as fa_fwd; FA_ERR_INVALID_ARG also for num_splits outside 1..64.
 */
fa_status fa_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *seqlens, void *o,
                    float *lse, int B, int H, int L, int d, int num_splits, fa_stream_t stream);

/*
 * Decode attention with grouped K/V heads (GQA; MQA when H_kv = 1).
 *
 * Defines: CMU 15-779 Lecture 5 notes, Exercise 7 (g = H_q / H_kv query heads
 *   share one K/V head, so each K/V element read serves g queries and the
 *   arithmetic intensity of decode rises to about g) and §8.4 (the split
 *   along the keys and the log-sum-exp merge, as fa_decode).
 *
 *   q        bf16 [B][H_q][d].
 *   k_cache, v_cache  bf16 [B][H_kv][L][d].
 *   Query head h attends to K/V head h / (H_q / H_kv): the g consecutive query
 *   heads h_kv*g .. h_kv*g + g - 1 share K/V head h_kv.
 *   seqlens, o [B][H_q][d], lse [B][H_q], d, num_splits: as fa_decode
 *   (keys of a sequence are cut into num_splits chunks of ceil(len/num_splits)
 *   rounded up to a multiple of 128 keys). H_q must be a multiple of H_kv.
 *   Cache entries at or beyond seqlens[b] may hold any bits (NaN included).
 * Workspace: B*H_q*num_splits*(d+1)*4 bytes of stream-ordered device memory.
 * Errors: as fa_decode; FA_ERR_INVALID_ARG also when H_q % H_kv != 0.
 */
fa_status fa_decode_gqa(const void *q, const void *k_cache, const void *v_cache, const int32_t *seqlens, void *o,
                        float *lse, int B, int Hq, int Hkv, int L, int d, int num_splits, fa_stream_t stream);

/*
 * Decode attention that allocates nothing.
 *
 * The pages have no counterpart of this call; it exists for callers that
 * cannot allocate device memory when they decode: a serving engine that gives
 * nearly all of HBM to its own KV-cache pool at start-up and forbids later
 * allocations, or a latency-critical decode loop where an allocation could
 * stall on the pool or fail under fragmentation.
 *
 * Arguments, layouts, results and errors are those of fa_decode. The split
 * partials live in one fixed 16 MiB array of device memory owned by libfa.so
 * (every GPU that loads the library holds it until the process exits)
 * instead of a per-call pool allocation; the call never allocates.
 *   - Limit: B * H * num_splits * (d + 1) <= 4,194,304 (fp32 values). Larger
 *     requests return FA_ERR_INVALID_ARG and fa_last_error_string() says why.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents; nothing in it needs to start at zero (every partial is written
 *     before it is read). Calls that may run at the same time on the GPU
 *     (unordered streams) race on it: order them on one stream.
 *   - The first call on each device looks up the array's address with that
 *     device current and caches it; make that first call before any stream
 *     capture.
 */
fa_status fa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, const int32_t *seqlens,
                            void *o, float *lse, int B, int H, int L, int d, int num_splits, fa_stream_t stream);

/* Static text for a status code. Never NULL. */
const char *fa_status_string(fa_status status);

/*
 * Text of the reason for the most recent non-OK status returned on the calling
 * thread ("" if there was none yet): the CUDA call that failed (FA_ERR_CUDA),
 * the argument check that rejected a call (FA_ERR_INVALID_ARG,
 * FA_ERR_UNSUPPORTED; for fa_decode_noalloc also the size of a request beyond
 * its static workspace), or the device error word's site (FA_ERR_TIMEOUT,
 * FA_ERR_CHECK). A later successful call leaves the text as it was.
 */
const char *fa_last_error_string(void);

/*
 * Synchronise `stream`, then read and clear the device error word of the
 * current device. Returns FA_ERR_TIMEOUT if a kernel recorded that one of its
 * bounded waits ran out since the last check, FA_ERR_CHECK if (in a library
 * built with FA_DEBUG) a kernel's end-of-kernel protocol check failed: its
 * roles did not walk the same items, ring positions and barrier phases.
 * FA_ERR_CUDA if the stream reports an error, FA_OK otherwise.
 * The pages define no failure detection: the bounded waits this call reports
 * are the library's own. fa_last_error_site() gives the code of the wait or
 * check that failed.
 */
fa_status fa_check_device_error(fa_stream_t stream);

/*
 * Site code of the first wait or check that failed, as read by the most recent
 * fa_check_device_error on the calling thread (0 if that call found none).
 * Codes: 1 Q landed, 2 K/V landed, 3 K/V slot free, 4 S done, 5 P written,
 * 6 O done, 7 teardown drain, 8 Q buffer free, 9 O read out, 10 block-sparse
 * work item published, 11 block-sparse work item slot free, 20-22 FA_DEBUG
 * protocol checks (forward, backward, GQA decode), 100 the timeout self-test.
 */
int fa_last_error_site(void);

/*
 * Work plan of fa_fwd (host only, no device needed): with square tiles of
 * `block` rows, count the (Q tile, K/V tile) pairs of an N x N problem and how
 * many of them the kernel computes. Causal mode skips every pair that lies
 * entirely above the diagonal (CMU 15-779 Lecture 5 notes §6.2: T(T+1)/2 of
 * T^2 pairs). fa_fwd uses block = 128.
 */
fa_status fa_fwd_plan(int N, int block, int causal, long long *pairs_total, long long *pairs_computed);

/*
 * Self-tests of the kernels' building blocks (used by the test suite).
 *
 * fa_selftest_mma: one 128 x n x k product on the tensor cores through the same
 *   staging the attention kernel uses (TMA with 128-byte swizzle into shared
 *   memory, tcgen05.mma with an fp32 accumulator in tensor memory).
 *   mode 0: D[128][n] = A[128][k] * B[n][k]^T, A and B K-major in shared memory
 *           (the S = Q K^T product), n = 128, k in {64, 128}.
 *   mode 1: D[128][n] = A[128][k] * B[k][n], A placed in tensor memory as packed
 *           bf16 pairs, B MN-major in shared memory (the O += P V product),
 *           k = 128, n in {64, 128}.
 *   mode 2: as mode 0 with e4m3 A and B (kind::f8f6f4), n = k = 128.
 *   mode 3: D = A * B^T with A placed in tensor memory as four e4m3 per 32-bit
 *           column and B [n][k] K-major in shared memory (the O += P V product
 *           with V given transposed), n = k = 128.
 *   mode 4: a pair of CTAs (a cluster of two on two SMs) computes one
 *           M = 256 product with tcgen05 .cta_group::2: D[256][128] =
 *           A[256][128] * B[128][128]^T, B K-major; each CTA holds 128 rows of
 *           A and 64 rows of B and receives its 128 rows of D.
 *   mode 5: as mode 4 with B[128][128] MN-major (rows are the contraction
 *           index), each CTA holding 64 of its columns.
 *   a, b: bf16 (modes 0, 1, 4, 5) or e4m3 byte (modes 2, 3) device pointers;
 *   d: fp32 device pointer [128][n] (modes 4, 5: [256][128] followed by the
 *   two CTAs' TMEM base addresses, 2 more 32-bit values).
 *
 * fa_selftest_wait_timeout: launch one block that waits on a barrier nothing
 *   ever arrives at, bounded by `timeout_us`; the kernel gives up, records
 *   the timeout in the device error word and returns. fa_check_device_error
 *   then reports FA_ERR_TIMEOUT.
 */
fa_status fa_selftest_mma(int mode, const void *a, const void *b, float *d, int n, int k, fa_stream_t stream);
fa_status fa_selftest_wait_timeout(unsigned int timeout_us, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
