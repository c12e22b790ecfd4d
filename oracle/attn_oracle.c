/*
 * attn_oracle.c -- plain, slow, float64 CPU oracle for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes is the plain definition of scaled-dot-product attention,
 * written out row by row with a two-pass stable softmax:
 *
 *   s_j   = scale * sum_d q[i,d] * k[j,d]           for every visible key j
 *   M     = max_j s_j
 *   Z     = sum_j exp(s_j - M)
 *   O[i]  = sum_j (exp(s_j - M) / Z) * v[j]
 *   LSE[i]= M + ln Z
 *
 * Sources (pages, by title and section):
 *  - "Implementing attention from scratch" (chorfi.xyz), Core ideas:
 *      "Shapes first" (the [B,H,T,D] layout, scores [B,H,T,S]),
 *      "Why scale by sqrt(D)", "Masks" (causal j <= i, key padding, the
 *      fully-masked-row hazard), "Stable softmax" (subtract the row max),
 *      "KV caching" (bottom-right alignment when T != S, GQA head sharing).
 *  - "Hands-on build guide: FlashAttention-style tiled attention kernel in
 *      pure NumPy", Verification: the naive dense attention it compares to.
 *  - "Building a causal self-attention block from scratch in PyTorch",
 *      Step 2 (mask convention: the code marks j > i as masked) and
 *      Step 3 (vanilla attention: scale, -inf fill, softmax, weights @ v).
 *  - "FlashAttention" (Transformers in Action, section 9.4.1): the tiled
 *      method is exact, so the plain definition is the oracle.
 *
 * Readings where the pages are silent:
 *  - Causal alignment is bottom-right: query i sits at key position
 *    i + (S - T); visible(i,j) = (j < L) and (not causal or j <= i + S - T).
 *  - key_lens[b] = L gives the valid length of sequence b for keys AND
 *    queries: query row i is a padded row iff i + (S - T) >= L.  A padded row,
 *    or a row with no visible key, has O = 0 and LSE = -inf.
 *  - GQA grouping is contiguous: query head h reads KV head h / (Hq / Hkv).
 *  - LSE is the natural log of sum_j exp(s_j), s_j already scaled.
 *
 * Chunked prefill against a KV cache ("Implementing attention from
 * scratch", KV caching: new queries sit after the cached positions, so
 * their offset is the cache length plus the position within the chunk):
 * with q_pos[b] given, query row i of sequence b sits at key position
 * q_pos[b] + i instead of i + S - T; visibility and padded rows follow from
 * that position as above.
 *
 * Inputs may be float64, float32 or bfloat16 (raw 16-bit patterns); every
 * element is widened exactly to double before use.  Layouts (contiguous):
 *   prefill  q [B,Hq,T,D], k/v [B,Hkv,S,D], o [.., D] float64, lse float64
 *   decode   q [B,Hq,D],   kcache/vcache [B,Hkv,S_max,D], kv_lens [B]
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F64 = 0, ORACLE_F32 = 1, ORACLE_BF16 = 2 };

/* Widen element `idx` of an array of the given storage type to double. */
static double load_elem(const void* base, int dtype, int64_t idx) {
  if (dtype == ORACLE_F64) return ((const double*)base)[idx];
  if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
  /* bfloat16: the 16 bits are the high half of an IEEE float32. */
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* One output row of the definition.  q_off / k_off / v_off are element
 * offsets of q[i,0], k[0,0], v[0,0] for this (batch, head).  `row_pos` is the
 * query's key position (i + S - T for prefill, kv_len - 1 for decode);
 * `L` the number of valid keys; `n_keys` the number of stored keys.
 * `scores` is caller scratch of n_keys doubles. */
static void attention_row(const void* q, int64_t q_off, const void* k,
                          int64_t k_off, const void* v, int64_t v_off,
                          int dtype, int n_keys, int D, int L, int causal,
                          int64_t row_pos, double scale, double* scores,
                          double* o_row, double* lse_out) {
  int j, d;
  int any = 0;
  double M = -INFINITY, Z = 0.0;
  for (d = 0; d < D; ++d) o_row[d] = 0.0;
  /* A padded query row (its position is past the valid length) is defined
   * as zero output, -inf LSE. */
  if (row_pos >= L) {
    *lse_out = -INFINITY;
    return;
  }
  /* Pass 1: scores of visible keys and their maximum. */
  for (j = 0; j < n_keys; ++j) {
    int visible = (j < L) && (!causal || (int64_t)j <= row_pos);
    if (!visible) {
      scores[j] = -INFINITY;
      continue;
    }
    double dot = 0.0;
    for (d = 0; d < D; ++d)
      dot += load_elem(q, dtype, q_off + d) *
             load_elem(k, dtype, k_off + (int64_t)j * D + d);
    scores[j] = scale * dot;
    if (!any || scores[j] > M) M = scores[j];
    any = 1;
  }
  if (!any) { /* every key masked: defined as O = 0, LSE = -inf */
    *lse_out = -INFINITY;
    return;
  }
  /* Pass 2: normaliser. */
  for (j = 0; j < n_keys; ++j)
    if (scores[j] != -INFINITY) Z += exp(scores[j] - M);
  /* Pass 3: convex combination of the visible value rows. */
  for (j = 0; j < n_keys; ++j) {
    if (scores[j] == -INFINITY) continue;
    double w = exp(scores[j] - M) / Z;
    for (d = 0; d < D; ++d)
      o_row[d] += w * load_elem(v, dtype, v_off + (int64_t)j * D + d);
  }
  *lse_out = M + log(Z);
}

/* ---------------------------------------------------------------- threads */

typedef struct {
  /* problem */
  const void *q, *k, *v;
  int dtype, B, Hq, Hkv, T, S, D, causal, decode;
  const int32_t* lens; /* key_lens (prefill) or kv_lens (decode); may be NULL */
  const int32_t* q_pos; /* prefill: key position of query row 0 per sequence; may be NULL */
  double scale;
  /* which rows: NULL = all, else flat row ids (b*Hq + h)*T + i */
  const int64_t* rows;
  int64_t n_rows;
  double *o, *lse;
  /* work split */
  int64_t begin, end;
  int status;
} job_t;

static void* run_rows(void* arg) {
  job_t* jb = (job_t*)arg;
  int n_keys = jb->S;
  double* scores = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
  if (!scores) {
    jb->status = 1;
    return NULL;
  }
  int G = jb->Hq / jb->Hkv;
  for (int64_t r = jb->begin; r < jb->end; ++r) {
    int64_t flat = jb->rows ? jb->rows[r] : r;
    int64_t i = flat % jb->T;
    int64_t bh = flat / jb->T;
    int h = (int)(bh % jb->Hq);
    int b = (int)(bh / jb->Hq);
    int g = h / G;
    int L = jb->lens ? jb->lens[b] : jb->S;
    int64_t row_pos = jb->decode  ? (int64_t)L - 1
                      : jb->q_pos ? (int64_t)jb->q_pos[b] + i
                                  : i + (jb->S - jb->T);
    int64_t q_off = flat * jb->D;
    int64_t kv_off = ((int64_t)b * jb->Hkv + g) * (int64_t)jb->S * jb->D;
    attention_row(jb->q, q_off, jb->k, kv_off, jb->v, kv_off, jb->dtype,
                  n_keys, jb->D, L, jb->causal || jb->decode, row_pos,
                  jb->scale, scores, jb->o + r * jb->D, jb->lse + r);
  }
  free(scores);
  return NULL;
}

static int run_parallel(job_t* proto, int64_t n_rows, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > n_rows) nthreads = n_rows > 0 ? (int)n_rows : 1;
  pthread_t tid[256];
  job_t jobs[256];
  int started[256] = {0};
  int status = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *proto;
    jobs[t].begin = n_rows * t / nthreads;
    jobs[t].end = n_rows * (t + 1) / nthreads;
    jobs[t].status = 0;
    if (nthreads == 1) {
      run_rows(&jobs[t]);
    } else if (pthread_create(&tid[t], NULL, run_rows, &jobs[t]) == 0) {
      started[t] = 1;
    } else {
      run_rows(&jobs[t]); /* could not spawn: do it on this thread */
    }
  }
  for (int t = 0; t < nthreads; ++t) {
    if (started[t]) pthread_join(tid[t], NULL);
    status |= jobs[t].status;
  }
  return status;
}

static int check_shape(int B, int Hq, int Hkv, int T, int S, int D) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || S <= 0 || D <= 0) return 1;
  if (Hq % Hkv != 0) return 1;
  return 0;
}

/* Prefill forward.  rows == NULL computes every row (o is [B,Hq,T,D],
 * lse [B,Hq,T]); otherwise only the n_rows listed flat row ids, packed
 * (o is [n_rows,D], lse [n_rows]).  q_pos (may be NULL) places query row 0
 * of sequence b at key position q_pos[b] (chunked prefill against a
 * cache); NULL means bottom-right, S - T.  Returns 0 on success. */
int oracle_attn_fwd(const void* q, const void* k, const void* v, int dtype,
                    int B, int Hq, int Hkv, int T, int S, int D, int causal,
                    const int32_t* key_lens, const int32_t* q_pos, double scale,
                    const int64_t* rows, int64_t n_rows, double* o,
                    double* lse, int nthreads) {
  if (check_shape(B, Hq, Hkv, T, S, D)) return 1;
  if (dtype < ORACLE_F64 || dtype > ORACLE_BF16) return 1;
  if (key_lens)
    for (int b = 0; b < B; ++b)
      if (key_lens[b] < 0 || key_lens[b] > S) return 1;
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.q = q; jb.k = k; jb.v = v; jb.dtype = dtype;
  jb.B = B; jb.Hq = Hq; jb.Hkv = Hkv; jb.T = T; jb.S = S; jb.D = D;
  jb.causal = causal; jb.decode = 0; jb.lens = key_lens; jb.q_pos = q_pos;
  jb.scale = scale; jb.rows = rows; jb.o = o; jb.lse = lse;
  int64_t total = rows ? n_rows : (int64_t)B * Hq * T;
  if (rows)
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= (int64_t)B * Hq * T) return 1;
  return run_parallel(&jb, total, nthreads);
}

/* Single-query decode against a KV cache: query (b,h) sits at position
 * kv_lens[b]-1 and sees cache rows 0..kv_lens[b]-1 (bottom-right causal
 * alignment, "Implementing attention from scratch", KV caching).
 * q/o are [B,Hq,D], caches [B,Hkv,S_max,D], lse [B,Hq]. */
int oracle_attn_decode(const void* q, const void* kcache, const void* vcache,
                       int dtype, const int32_t* kv_lens, int B, int Hq,
                       int Hkv, int S_max, int D, double scale, double* o,
                       double* lse, int nthreads) {
  if (check_shape(B, Hq, Hkv, 1, S_max, D) || !kv_lens) return 1;
  if (dtype < ORACLE_F64 || dtype > ORACLE_BF16) return 1;
  for (int b = 0; b < B; ++b)
    if (kv_lens[b] < 0 || kv_lens[b] > S_max) return 1;
  job_t jb;
  memset(&jb, 0, sizeof jb);
  jb.q = q; jb.k = kcache; jb.v = vcache; jb.dtype = dtype;
  jb.B = B; jb.Hq = Hq; jb.Hkv = Hkv; jb.T = 1; jb.S = S_max; jb.D = D;
  jb.causal = 1; jb.decode = 1; jb.lens = kv_lens; jb.scale = scale;
  jb.rows = NULL; jb.o = o; jb.lse = lse;
  return run_parallel(&jb, (int64_t)B * Hq, nthreads);
}

/* Append one token's K/V rows per (batch, kv head) at offset pos[b]
 * ("Building a causal self-attention block", Step 5, KVCache.update, and
 * "Implementing attention from scratch", KV caching: the new token goes at
 * cache length).  Works on raw element storage of `elem_bytes` bytes.
 * Returns the number of (b, g) pairs skipped because pos[b] was out of
 * range [0, S_max). */
int oracle_kv_append(void* kcache, void* vcache, const void* k_new,
                     const void* v_new, const int32_t* pos, int B, int Hkv,
                     int S_max, int D, int elem_bytes) {
  int skipped = 0;
  size_t row = (size_t)D * (size_t)elem_bytes;
  for (int b = 0; b < B; ++b) {
    for (int g = 0; g < Hkv; ++g) {
      if (pos[b] < 0 || pos[b] >= S_max) {
        ++skipped;
        continue;
      }
      size_t dst = (((size_t)b * Hkv + g) * (size_t)S_max + (size_t)pos[b]) * row;
      size_t src = ((size_t)b * Hkv + g) * row;
      memcpy((char*)kcache + dst, (const char*)k_new + src, row);
      memcpy((char*)vcache + dst, (const char*)v_new + src, row);
    }
  }
  return skipped;
}
