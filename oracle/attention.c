/*
 * Exact-attention oracle: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library. The product path
 * (the CUDA library and its Python binding) never calls it, links it or
 * shares code with it.
 *
 * What it computes is the textbook "standard attention", written out step by
 * step exactly as the pages define it, with the N x N score matrix S and the
 * probability matrix P materialised in memory:
 *
 *   step 1  S = Q K^T                       (MatMul 1)
 *   step 2  S = scale * S, and under a causal mask S[i][j] = -inf for j > i
 *   step 3  P = rowwise softmax(S) with the row maximum subtracted first
 *   step 4  O = P V,  and the per-row log-sum-exp  LSE_i = m_i + ln(l_i)
 *
 * Sources:
 *   - "已有的几种大模型上下文支持情况" (cicada blog), §1.2 core formula
 *     Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V and §1.3 "the four
 *     computation steps" (MatMul 1, scale + optional causal mask, softmax
 *     with max subtraction, MatMul 2).
 *   - "FlashAttention 完全拆解（一）", background section, Algorithm 0 (the
 *     three-kernel standard implementation: S = QK^T, P = softmax(S), O = PV).
 *   - CMU 15-779 Lecture 5 notes, §2.3 (scaled dot-product attention and the
 *     causal mask: positions j > i set to -inf, so their weights are 0) and
 *     §4.2 (safe softmax: subtract the row maximum m before exponentiating).
 *   - LSE_i = m_i + ln(l_i): cicada blog §3.2.3 (FA-2 final write of the
 *     log-sum-exp vector L) and Lecture 5 notes §5.1 (L_i = m + log l).
 *
 * Readings where the pages leave a step open:
 *   - the scale multiplies the raw dot products before masking and softmax,
 *     so softmax and LSE are over the scaled scores;
 *   - the LSE uses the natural logarithm;
 *   - the causal mask keeps the diagonal (key j visible to query i iff j <= i),
 *     and a query row's position is given explicitly so that a subset of rows
 *     can be evaluated (each still a full row over all visible keys).
 *
 * No blocking, no fusion, no online softmax: each step runs over whole rows.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

/*
 * Standard attention for one (batch, head) and a list of query rows.
 *
 *   q      [n_rows][d]   the query rows to evaluate
 *   q_pos  [n_rows]      position of each query row in the sequence (used by
 *                        the causal mask only; may be NULL when causal == 0)
 *   k, v   [n_keys][d]   all keys and values of this head
 *   o      [n_rows][d]   output
 *   lse    [n_rows]      output, natural log-sum-exp of the scaled scores
 *   s_out  [n_rows][n_keys] optional copy of the scaled, masked scores (NULL)
 *   p_out  [n_rows][n_keys] optional copy of the probabilities P (NULL)
 *
 * Returns ORACLE_OK, or an error code for bad arguments / allocation failure.
 */
int oracle_attention_rows(const double *q, const int *q_pos, const double *k,
                          const double *v, int n_rows, int n_keys, int d,
                          int causal, double scale, double *o, double *lse,
                          double *s_out, double *p_out) {
  if (n_rows < 0 || n_keys < 1 || d < 1) return ORACLE_ERR_ARG;
  if (causal && q_pos == NULL) return ORACLE_ERR_ARG;
  if (n_rows == 0) return ORACLE_OK;

  size_t nn = (size_t)n_rows * (size_t)n_keys;
  double *S = (double *)malloc(nn * sizeof(double));
  double *P = (double *)malloc(nn * sizeof(double));
  double *m = (double *)malloc((size_t)n_rows * sizeof(double));
  double *l = (double *)malloc((size_t)n_rows * sizeof(double));
  if (!S || !P || !m || !l) {
    free(S); free(P); free(m); free(l);
    return ORACLE_ERR_NOMEM;
  }

  /* Step 1: S = Q K^T (every query row against every key). */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n_rows; ++i) {
    for (int j = 0; j < n_keys; ++j) {
      double acc = 0.0;
      for (int t = 0; t < d; ++t) acc += q[(size_t)i * d + t] * k[(size_t)j * d + t];
      S[(size_t)i * n_keys + j] = acc;
    }
  }

  /* Step 2: scale, then the causal mask (future keys -> -inf). */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n_rows; ++i) {
    for (int j = 0; j < n_keys; ++j) {
      double x = scale * S[(size_t)i * n_keys + j];
      if (causal && j > q_pos[i]) x = -INFINITY;
      S[(size_t)i * n_keys + j] = x;
    }
  }

  /* Step 3: row-wise safe softmax: m = max, e = exp(x - m), l = sum e, P = e / l. */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n_rows; ++i) {
    const double *Si = S + (size_t)i * n_keys;
    double *Pi = P + (size_t)i * n_keys;
    double mi = -INFINITY;
    for (int j = 0; j < n_keys; ++j)
      if (Si[j] > mi) mi = Si[j];
    double li = 0.0;
    for (int j = 0; j < n_keys; ++j) {
      /* a masked score is -inf; exp(-inf - m) is exactly 0 for finite m */
      double e = (Si[j] == -INFINITY) ? 0.0 : exp(Si[j] - mi);
      Pi[j] = e;
      li += e;
    }
    for (int j = 0; j < n_keys; ++j) Pi[j] = Pi[j] / li;
    m[i] = mi;
    l[i] = li;
  }

  /* Step 4: O = P V and LSE = m + ln(l). Each O[i][c] is the sum over keys
   * j = 0, 1, ... of P[i][j] * V[j][c], accumulated in ascending j; the j loop
   * is outside the c loop only so that V is read row by row. */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n_rows; ++i) {
    const double *Pi = P + (size_t)i * n_keys;
    double *Oi = o + (size_t)i * d;
    for (int c = 0; c < d; ++c) Oi[c] = 0.0;
    for (int j = 0; j < n_keys; ++j) {
      const double pij = Pi[j];
      const double *Vj = v + (size_t)j * d;
      for (int c = 0; c < d; ++c) Oi[c] += pij * Vj[c];
    }
    lse[i] = m[i] + log(l[i]);
  }

  if (s_out) memcpy(s_out, S, nn * sizeof(double));
  if (p_out) memcpy(p_out, P, nn * sizeof(double));
  free(S); free(P); free(m); free(l);
  return ORACLE_OK;
}

/*
 * Thread count of the OpenMP loops of later calls made from the calling
 * thread (n >= 1); returns the count now in effect. Used to time the oracle
 * on one core. Every row is computed by one thread in a fixed order, so the
 * results do not depend on it.
 */
int oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/*
 * Batched prefill attention over [B][H][N][d] tensors (all rows of every
 * head), one call of oracle_attention_rows per (batch, head).
 */
int oracle_attention(const double *q, const double *k, const double *v,
                     double *o, double *lse, int B, int H, int N, int d,
                     int causal, double scale) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return ORACLE_ERR_ARG;
  int *pos = (int *)malloc((size_t)N * sizeof(int));
  if (!pos) return ORACLE_ERR_NOMEM;
  for (int i = 0; i < N; ++i) pos[i] = i;
  int rc = ORACLE_OK;
  for (int bh = 0; bh < B * H && rc == ORACLE_OK; ++bh) {
    size_t off = (size_t)bh * N * d;
    rc = oracle_attention_rows(q + off, pos, k + off, v + off, N, N, d, causal,
                               scale, o + off, lse + (size_t)bh * N, NULL, NULL);
  }
  free(pos);
  return rc;
}

/*
 * Decode-time attention: one query token per (batch, head) against the first
 * seqlens[b] entries of a KV cache of capacity L.
 *
 *   q [B][H][d], k_cache / v_cache [B][H][L][d], seqlens [B] (1..L)
 *   o [B][H][d], lse [B][H]; scale = 1/sqrt(d) (the decode call has no
 *   scale argument).
 *
 * The single new query sees every cached key, so there is no mask: CMU 15-779
 * Lecture 5 notes §8.2 (the cached decode step must equal recomputing the
 * full causal sequence, whose last row sees all earlier positions).
 * Flash-Decoding splits this sum along the keys; the split count does not
 * change the result, so the oracle does not split.
 */
int oracle_decode(const double *q, const double *k_cache, const double *v_cache,
                  const int *seqlens, double *o, double *lse, int B, int H,
                  int L, int d) {
  if (B < 1 || H < 1 || L < 1 || d < 1) return ORACLE_ERR_ARG;
  double scale = 1.0 / sqrt((double)d);
  for (int b = 0; b < B; ++b) {
    int len = seqlens[b];
    if (len < 1 || len > L) return ORACLE_ERR_ARG;
    for (int h = 0; h < H; ++h) {
      size_t bh = (size_t)b * H + h;
      int rc = oracle_attention_rows(q + bh * d, NULL, k_cache + bh * (size_t)L * d,
                                     v_cache + bh * (size_t)L * d, 1, len, d, 0,
                                     scale, o + bh * d, lse + bh, NULL, NULL);
      if (rc != ORACLE_OK) return rc;
    }
  }
  return ORACLE_OK;
}

/*
 * Standard attention under a block mask (block-sparse attention).
 *
 *   q, k, v [B][H][N][d]; o [B][H][N][d]; lse [B][H][N];
 *   mask [mask_heads][T][T] bytes, T = ceil(N / block), mask_heads 1 (one
 *   mask for every head) or H (head h uses mask h).
 *
 * "FlashAttention 完全拆解（一）", block-sparse extension: a block-level mask
 * over the N x N score matrix; the scores of masked-out blocks take no part.
 * Key j is visible to query i when mask[i / block][j / block] != 0 and, if
 * causal, j <= i. Each row is the standard softmax over its visible keys
 * (max subtracted, exp, sum, divide, O = P V, LSE = m + ln l). A row with no
 * visible key has o = 0 and lse = -inf (the empty sum; the identity of the
 * combine operator).
 */
int oracle_attention_block_mask(const double *q, const double *k, const double *v,
                                const unsigned char *mask, int mask_heads, int block,
                                double *o, double *lse, int B, int H, int N, int d,
                                int causal, double scale) {
  if (B < 1 || H < 1 || N < 1 || d < 1 || block < 1) return ORACLE_ERR_ARG;
  if (mask_heads != 1 && mask_heads != H) return ORACLE_ERR_ARG;
  int T = (N + block - 1) / block;
  double *s = (double *)malloc((size_t)N * sizeof(double));
  if (!s) return ORACLE_ERR_NOMEM;
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < H; ++h) {
      size_t bh = (size_t)b * H + h;
      const unsigned char *mk = mask + (size_t)(mask_heads == 1 ? 0 : h) * T * T;
      const double *qh = q + bh * (size_t)N * d, *kh = k + bh * (size_t)N * d, *vh = v + bh * (size_t)N * d;
      for (int i = 0; i < N; ++i) {
        double m = -INFINITY;
        for (int j = 0; j < N; ++j) {
          int vis = mk[(size_t)(i / block) * T + (j / block)] != 0 && (!causal || j <= i);
          if (!vis) {
            s[j] = -INFINITY;
            continue;
          }
          double acc = 0.0;
          for (int t = 0; t < d; ++t) acc += qh[(size_t)i * d + t] * kh[(size_t)j * d + t];
          s[j] = acc * scale;
          if (s[j] > m) m = s[j];
        }
        double *orow = o + (bh * N + i) * (size_t)d;
        for (int t = 0; t < d; ++t) orow[t] = 0.0;
        if (m == -INFINITY) {
          lse[bh * N + i] = -INFINITY;
          continue;
        }
        double l = 0.0;
        for (int j = 0; j < N; ++j) {
          if (s[j] == -INFINITY) continue;
          double e = exp(s[j] - m);
          l += e;
          for (int t = 0; t < d; ++t) orow[t] += e * vh[(size_t)j * d + t];
        }
        for (int t = 0; t < d; ++t) orow[t] /= l;
        lse[bh * N + i] = m + log(l);
      }
    }
  }
  free(s);
  return ORACLE_OK;
}

/*
 * Decode with grouped K/V heads (GQA; MQA when H_kv = 1).
 *
 *   q [B][H_q][d]; k_cache, v_cache [B][H_kv][L][d]; seqlens [B];
 *   o [B][H_q][d]; lse [B][H_q]. H_q must be a multiple of H_kv.
 *
 * CMU 15-779 Lecture 5 notes, Exercise 7 (and §8.3): g = H_q / H_kv query
 * heads share one K/V head. Query head h attends to K/V head h / g (the g
 * consecutive query heads h_kv*g .. h_kv*g + g - 1 form one group), over
 * keys 0..seqlens[b]-1, unmasked, scale 1/sqrt(d), exactly as a decode step
 * with its own K/V head would.
 */
int oracle_decode_gqa(const double *q, const double *k_cache, const double *v_cache,
                      const int *seqlens, double *o, double *lse, int B, int Hq,
                      int Hkv, int L, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || d < 1 || Hq % Hkv != 0) return ORACLE_ERR_ARG;
  int g = Hq / Hkv;
  double scale = 1.0 / sqrt((double)d);
  for (int b = 0; b < B; ++b) {
    int len = seqlens[b];
    if (len < 1 || len > L) return ORACLE_ERR_ARG;
    for (int h = 0; h < Hq; ++h) {
      size_t bq = (size_t)b * Hq + h;
      size_t bkv = (size_t)b * Hkv + h / g;
      int rc = oracle_attention_rows(q + bq * d, NULL, k_cache + bkv * (size_t)L * d,
                                     v_cache + bkv * (size_t)L * d, 1, len, d, 0,
                                     scale, o + bq * d, lse + bq, NULL, NULL);
      if (rc != ORACLE_OK) return rc;
    }
  }
  return ORACLE_OK;
}

/*
 * Backward of standard attention for one (batch, head), every intermediate
 * materialised, fp64.
 *
 *   q, k, v, dout  [n][d]; outputs dq, dk, dv [n][d].
 *
 * With S' = scale * Q K^T (+ causal -inf), P = softmax(S') row-wise,
 * O = P V and the upstream gradient dO:
 *   dV = P^T dO
 *   dP = dO V^T
 *   D_i = sum_j P_ij dP_ij            (equal to rowsum(dO_i * O_i))
 *   dS = P * (dP - D)                 (softmax Jacobian diag(p) - p p^T)
 *   dQ = scale * dS K,  dK = scale * dS^T Q
 * Sources: CMU 15-779 Lecture 5 notes §7.1 (the chain rule and the softmax
 * Jacobian), §7.3 (D_i = dO_i . O_i lets dS be formed block by block);
 * "FlashAttention 完全拆解（一）", backward section (dS from P, dP and D).
 * The oracle forms D from its definition sum_j P_ij dP_ij.
 */
int oracle_attention_bwd_head(const double *q, const double *k, const double *v,
                              const double *dout, int n, int d, int causal,
                              double scale, double *dq, double *dk, double *dv) {
  if (n < 1 || d < 1) return ORACLE_ERR_ARG;
  size_t nn = (size_t)n * n;
  double *P = (double *)malloc(nn * sizeof(double));
  double *dP = (double *)malloc(nn * sizeof(double));
  double *Dv = (double *)malloc((size_t)n * sizeof(double));
  if (!P || !dP || !Dv) {
    free(P); free(dP); free(Dv);
    return ORACLE_ERR_NOMEM;
  }
  /* P = softmax(scale * Q K^T + mask), row by row (safe softmax). */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n; ++i) {
    double *Pi = P + (size_t)i * n;
    double mi = -INFINITY;
    for (int j = 0; j < n; ++j) {
      double acc = 0.0;
      for (int t = 0; t < d; ++t) acc += q[(size_t)i * d + t] * k[(size_t)j * d + t];
      double x = scale * acc;
      if (causal && j > i) x = -INFINITY;
      Pi[j] = x;
      if (x > mi) mi = x;
    }
    double li = 0.0;
    for (int j = 0; j < n; ++j) {
      double e = (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - mi);
      Pi[j] = e;
      li += e;
    }
    for (int j = 0; j < n; ++j) Pi[j] /= li;
  }
  /* dP = dO V^T and D_i = sum_j P_ij dP_ij. */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n; ++i) {
    double Di = 0.0;
    for (int j = 0; j < n; ++j) {
      double acc = 0.0;
      for (int t = 0; t < d; ++t) acc += dout[(size_t)i * d + t] * v[(size_t)j * d + t];
      dP[(size_t)i * n + j] = acc;
      Di += P[(size_t)i * n + j] * acc;
    }
    Dv[i] = Di;
  }
  /* dS = P * (dP - D), kept in dP. */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      size_t ij = (size_t)i * n + j;
      dP[ij] = P[ij] * (dP[ij] - Dv[i]);
    }
  /* dQ = scale * dS K. */
#pragma omp parallel for schedule(static)
  for (int i = 0; i < n; ++i) {
    for (int t = 0; t < d; ++t) dq[(size_t)i * d + t] = 0.0;
    for (int j = 0; j < n; ++j) {
      double s = dP[(size_t)i * n + j];
      for (int t = 0; t < d; ++t) dq[(size_t)i * d + t] += s * k[(size_t)j * d + t];
    }
    for (int t = 0; t < d; ++t) dq[(size_t)i * d + t] *= scale;
  }
  /* dK = scale * dS^T Q and dV = P^T dO. */
#pragma omp parallel for schedule(static)
  for (int j = 0; j < n; ++j) {
    for (int t = 0; t < d; ++t) {
      dk[(size_t)j * d + t] = 0.0;
      dv[(size_t)j * d + t] = 0.0;
    }
    for (int i = 0; i < n; ++i) {
      double s = dP[(size_t)i * n + j];
      double p = P[(size_t)i * n + j];
      for (int t = 0; t < d; ++t) {
        dk[(size_t)j * d + t] += s * q[(size_t)i * d + t];
        dv[(size_t)j * d + t] += p * dout[(size_t)i * d + t];
      }
    }
    for (int t = 0; t < d; ++t) dk[(size_t)j * d + t] *= scale;
  }
  free(P); free(dP); free(Dv);
  return ORACLE_OK;
}

/* Backward over [B][H][N][d] tensors, one head at a time. */
int oracle_attention_bwd(const double *q, const double *k, const double *v,
                         const double *dout, double *dq, double *dk, double *dv,
                         int B, int H, int N, int d, int causal, double scale) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return ORACLE_ERR_ARG;
  for (int bh = 0; bh < B * H; ++bh) {
    size_t off = (size_t)bh * N * d;
    int rc = oracle_attention_bwd_head(q + off, k + off, v + off, dout + off, N, d,
                                       causal, scale, dq + off, dk + off, dv + off);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}
