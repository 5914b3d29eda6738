/*
 * neox_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of exact causal multi-head self-attention
 * with GPT-NeoX rotary position embedding ("Neox style", rotate-half) applied to
 * the first rotary_dim dims of both Query and Key.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark may load this file's
 * library.  The CUDA path in causal_rope_self_neox_b300/ shares no code with it.
 *
 * Where each step comes from (page title, section):
 *  - exact (not approximated) causal softmax attention, O(n^2) compute:
 *      "gpt-neox - 模型与框架" (pomoai hub page), section "问题二：注意力计算太慢".
 *  - rotary embedding on BOTH Query and Key, Neox style, rotary_embedding=24 of
 *    size_per_head=96 (partial rotary), QK accumulation in fp32 by default,
 *    fused query_key_value projection whose HuggingFace layout
 *    [hidden, num_heads, 3, head_hidden] gives a per-token packed [H,3,D]:
 *      "GPT-NeoX on FasterTransformer" guide, sections "背景", "模型配置（config.ini）"
 *      and "从 HuggingFace 检查点部署".
 *  - rotate-half pairing (dim i with dim i+r/2), inv_freq = base^(-2i/r),
 *    scale 1/sqrt(D), outputs out[B,S,H,D] and the natural-log row
 *    logsumexp lse[B,H,S]: the problem statement of this op (the pages name
 *    the stored attention.rotary_emb.inv_freq tensor but print no formula).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - positions are 0..S-1 for every sequence, the same for Q and K;
 *  - the causal mask keeps keys j <= i (diagonal included);
 *  - the rotation is exact: no rounding of the rotated Q/K anywhere here;
 *  - no dropout, no bias, no ALiBi.
 *
 * Steps are written in the order of the definition, with no tiling, no online
 * softmax and no fusion:  widen bf16 -> fp64;  inv_freq;  rotate q_s and k_s by
 * angle s*inv_freq;  scores q'_i.k'_j / sqrt(D) for j <= i;  max;  exp;  sum;
 * weighted sum of v_j;  lse = max + ln(sum).
 * The backward (neox_oracle_bwd, at the end) applies the chain rule to those same
 * steps, in reverse, for the gradient of sum(dout * out) with respect to qkv.
 * The query_key_value projection that produces the packed qkv (neox_oracle_qkv_proj,
 * last in the file) is one plain product of the token rows with the weight plus the
 * layer's bias, read from the same guide's layer list and HuggingFace weight layout.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_NOMEM (-2)

/* bf16 -> fp64: a bf16 value is the top 16 bits of an IEEE fp32; widening is exact. */
static double bf16_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* inv_freq[i] = base^(-2i / r), i = 0 .. r/2-1. */
void neox_oracle_inv_freq(int r, double base, double* inv_freq) {
  for (int i = 0; i < r / 2; ++i) inv_freq[i] = pow(base, -2.0 * (double)i / (double)r);
}

/* Rotate-half rotary embedding of one head vector x[0..D) at position p:
 *   for i < r/2 with theta = p * inv_freq[i]:
 *     y[i]       = x[i] cos(theta) - x[i+r/2] sin(theta)
 *     y[i+r/2]   = x[i+r/2] cos(theta) + x[i] sin(theta)
 *   y[d] = x[d] for d >= r.                                                    */
void neox_oracle_rotate(const double* x, int D, int r, double base, int64_t p, double* y) {
  int h = r / 2;
  for (int d = 0; d < D; ++d) y[d] = x[d];
  for (int i = 0; i < h; ++i) {
    double theta = (double)p * pow(base, -2.0 * (double)i / (double)r);
    double c = cos(theta), s = sin(theta);
    y[i] = x[i] * c - x[i + h] * s;
    y[i + h] = x[i + h] * c + x[i] * s;
  }
}

/* Element offset of qkv[b, s, h, slot, 0] in the packed [B,S,H,3,D] tensor. */
static int64_t qkv_off(int64_t b, int64_t s, int64_t h, int slot, int S, int H, int D) {
  return (((b * S + s) * H + h) * 3 + slot) * (int64_t)D;
}

typedef struct {
  const uint16_t* qkv;
  int B, S, H, D, r;
  double base;
  /* either all rows (rows == NULL) or the listed (b, h, i) triples */
  const int64_t* rows;
  int64_t n_rows;
  const int64_t* order; /* rows sorted by (b, h): indices into rows */
  double* out;
  double* lse;
  /* work distribution */
  pthread_mutex_t mu;
  int64_t next;
  int64_t n_items;
  int failed;
} job_t;

/* Rotated keys k'_s for s < n of head (b, h), plus raw values v_s. */
static void load_head(const job_t* J, int64_t b, int64_t h, int64_t n, double* Kr, double* V, double* tmp) {
  int D = J->D;
  for (int64_t s = 0; s < n; ++s) {
    const uint16_t* k = J->qkv + qkv_off(b, s, h, 1, J->S, J->H, D);
    const uint16_t* v = J->qkv + qkv_off(b, s, h, 2, J->S, J->H, D);
    for (int d = 0; d < D; ++d) tmp[d] = bf16_to_f64(k[d]);
    neox_oracle_rotate(tmp, D, J->r, J->base, s, Kr + s * D);
    for (int d = 0; d < D; ++d) V[s * D + d] = bf16_to_f64(v[d]);
  }
}

/* One query row i of head (b, h): softmax over keys j <= i of q'_i.k'_j/sqrt(D).
 * Writes out_row[0..D) and *lse_out.  scores has room for i+1 doubles.        */
static void one_row(const job_t* J, int64_t b, int64_t h, int64_t i, const double* Kr, const double* V,
                    double* qraw, double* qr, double* scores, double* out_row, double* lse_out) {
  int D = J->D;
  const uint16_t* q = J->qkv + qkv_off(b, i, h, 0, J->S, J->H, D);
  for (int d = 0; d < D; ++d) qraw[d] = bf16_to_f64(q[d]);
  neox_oracle_rotate(qraw, D, J->r, J->base, i, qr);
  double scale = 1.0 / sqrt((double)D);
  double m = -INFINITY;
  for (int64_t j = 0; j <= i; ++j) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qr[d] * Kr[j * D + d];
    scores[j] = dot * scale;
    if (scores[j] > m) m = scores[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j <= i; ++j) {
    scores[j] = exp(scores[j] - m);
    l += scores[j];
  }
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  for (int64_t j = 0; j <= i; ++j) {
    double w = scores[j] / l;
    for (int d = 0; d < D; ++d) out_row[d] += w * V[j * D + d];
  }
  *lse_out = m + log(l);
}

static int64_t take(job_t* J) {
  pthread_mutex_lock(&J->mu);
  int64_t k = J->next < J->n_items ? J->next++ : -1;
  pthread_mutex_unlock(&J->mu);
  return k;
}

/* Full mode: one work item = one head (b, h); every row of it. */
static void* worker_full(void* arg) {
  job_t* J = (job_t*)arg;
  int S = J->S, H = J->H, D = J->D;
  double* Kr = malloc(sizeof(double) * (size_t)S * D);
  double* V = malloc(sizeof(double) * (size_t)S * D);
  double* tmp = malloc(sizeof(double) * (size_t)D * 2);
  double* scores = malloc(sizeof(double) * (size_t)S);
  double* orow = malloc(sizeof(double) * (size_t)D);
  if (!Kr || !V || !tmp || !scores || !orow) {
    pthread_mutex_lock(&J->mu);
    J->failed = 1;
    pthread_mutex_unlock(&J->mu);
  } else {
    for (int64_t item; (item = take(J)) >= 0;) {
      int64_t b = item / H, h = item % H;
      load_head(J, b, h, S, Kr, V, tmp);
      for (int64_t i = 0; i < S; ++i) {
        double l;
        one_row(J, b, h, i, Kr, V, tmp, tmp + D, scores, orow, &l);
        for (int d = 0; d < D; ++d) J->out[((b * S + i) * H + h) * D + d] = orow[d];
        J->lse[(b * H + h) * S + i] = l;
      }
    }
  }
  free(Kr); free(V); free(tmp); free(scores); free(orow);
  return NULL;
}

/* Rows mode: one work item = one head group of the (b,h)-sorted row list. */
static void* worker_rows(void* arg) {
  job_t* J = (job_t*)arg;
  int S = J->S, D = J->D;
  double* Kr = malloc(sizeof(double) * (size_t)S * D);
  double* V = malloc(sizeof(double) * (size_t)S * D);
  double* tmp = malloc(sizeof(double) * (size_t)D * 2);
  double* scores = malloc(sizeof(double) * (size_t)S);
  if (!Kr || !V || !tmp || !scores) {
    pthread_mutex_lock(&J->mu);
    J->failed = 1;
    pthread_mutex_unlock(&J->mu);
  } else {
    for (int64_t item; (item = take(J)) >= 0;) {
      /* item indexes the sorted order; a group starts where (b,h) changes */
      int64_t k0 = J->order[item];
      int64_t b = J->rows[3 * k0], h = J->rows[3 * k0 + 1];
      if (item > 0) {
        int64_t kp = J->order[item - 1];
        if (J->rows[3 * kp] == b && J->rows[3 * kp + 1] == h) continue; /* not a group start */
      }
      int64_t end = item, maxi = 0;
      while (end < J->n_rows) {
        int64_t k = J->order[end];
        if (J->rows[3 * k] != b || J->rows[3 * k + 1] != h) break;
        if (J->rows[3 * k + 2] > maxi) maxi = J->rows[3 * k + 2];
        ++end;
      }
      load_head(J, b, h, maxi + 1, Kr, V, tmp);
      for (int64_t e = item; e < end; ++e) {
        int64_t k = J->order[e];
        one_row(J, b, h, J->rows[3 * k + 2], Kr, V, tmp, tmp + D, scores, J->out + k * D, J->lse + k);
      }
    }
  }
  free(Kr); free(V); free(tmp); free(scores);
  return NULL;
}

static int check_args(const uint16_t* qkv, int B, int S, int H, int D, int r, double base) {
  if (!qkv || B < 1 || S < 1 || H < 1 || D < 1 || r < 0 || r > D || (r & 1) || !(base > 0.0)) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

static int run(job_t* J, void* (*fn)(void*), int threads) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  pthread_mutex_init(&J->mu, NULL);
  J->next = 0;
  J->failed = 0;
  int started = 0;
  for (int t = 1; t < threads; ++t)
    if (pthread_create(&tid[started], NULL, fn, J) == 0) ++started;
  fn(J);
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&J->mu);
  return J->failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Every row of every head.
 * qkv: bf16 bits [B,S,H,3,D] (slot 0 = Q, 1 = K, 2 = V).
 * out: fp64 [B,S,H,D];  lse: fp64 [B,H,S], natural log of the sum of exp of the
 * scaled scores.  threads: worker threads (>= 1).  Returns 0 or a negative error. */
int neox_oracle_fwd(const uint16_t* qkv, int B, int S, int H, int D, int r, double base,
                    double* out, double* lse, int threads) {
  int e = check_args(qkv, B, S, H, D, r, base);
  if (e || !out || !lse) return ORACLE_ERR_ARG;
  job_t J;
  memset(&J, 0, sizeof J);
  J.qkv = qkv; J.B = B; J.S = S; J.H = H; J.D = D; J.r = r; J.base = base;
  J.out = out; J.lse = lse;
  J.n_items = (int64_t)B * H;
  return run(&J, worker_full, threads);
}

static const int64_t* g_sort_rows; /* only read inside the qsort call below */
static int cmp_bh(const void* a, const void* b) {
  int64_t i = *(const int64_t*)a, j = *(const int64_t*)b;
  const int64_t* R = g_sort_rows;
  if (R[3 * i] != R[3 * j]) return R[3 * i] < R[3 * j] ? -1 : 1;
  if (R[3 * i + 1] != R[3 * j + 1]) return R[3 * i + 1] < R[3 * j + 1] ? -1 : 1;
  return i < j ? -1 : (i > j);
}
static pthread_mutex_t g_sort_mu = PTHREAD_MUTEX_INITIALIZER;

/* Listed rows only.  rows: n triples (b, h, i).  out: fp64 [n, D];  lse: fp64 [n]. */
int neox_oracle_fwd_rows(const uint16_t* qkv, int B, int S, int H, int D, int r, double base,
                         const int64_t* rows, int64_t n, double* out, double* lse, int threads) {
  int e = check_args(qkv, B, S, H, D, r, base);
  if (e || !rows || n < 0 || (n > 0 && (!out || !lse))) return ORACLE_ERR_ARG;
  for (int64_t k = 0; k < n; ++k)
    if (rows[3 * k] < 0 || rows[3 * k] >= B || rows[3 * k + 1] < 0 || rows[3 * k + 1] >= H ||
        rows[3 * k + 2] < 0 || rows[3 * k + 2] >= S)
      return ORACLE_ERR_ARG;
  if (n == 0) return ORACLE_OK;
  int64_t* order = malloc(sizeof(int64_t) * (size_t)n);
  if (!order) return ORACLE_ERR_NOMEM;
  for (int64_t k = 0; k < n; ++k) order[k] = k;
  pthread_mutex_lock(&g_sort_mu);
  g_sort_rows = rows;
  qsort(order, (size_t)n, sizeof(int64_t), cmp_bh);
  pthread_mutex_unlock(&g_sort_mu);
  job_t J;
  memset(&J, 0, sizeof J);
  J.qkv = qkv; J.B = B; J.S = S; J.H = H; J.D = D; J.r = r; J.base = base;
  J.rows = rows; J.n_rows = n; J.order = order; J.out = out; J.lse = lse;
  J.n_items = n;
  int rc = run(&J, worker_rows, threads);
  free(order);
  return rc;
}

/* The explicit probability row of query (b, h, i): p[j] = exp(s_ij - m) / l for
 * j <= i.  p has room for i+1 doubles.  Used by the row-sum and weighting checks. */
int neox_oracle_probs(const uint16_t* qkv, int B, int S, int H, int D, int r, double base,
                      int b, int h, int i, double* p) {
  int e = check_args(qkv, B, S, H, D, r, base);
  if (e || !p || b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= S) return ORACLE_ERR_ARG;
  job_t J;
  memset(&J, 0, sizeof J);
  J.qkv = qkv; J.B = B; J.S = S; J.H = H; J.D = D; J.r = r; J.base = base;
  double* Kr = malloc(sizeof(double) * (size_t)(i + 1) * D);
  double* V = malloc(sizeof(double) * (size_t)(i + 1) * D);
  double* tmp = malloc(sizeof(double) * (size_t)D * 2);
  double* orow = malloc(sizeof(double) * (size_t)D);
  int rc = ORACLE_ERR_NOMEM;
  if (Kr && V && tmp && orow) {
    double l;
    load_head(&J, b, h, i + 1, Kr, V, tmp);
    one_row(&J, b, h, i, Kr, V, tmp, tmp + D, p, orow, &l);
    /* one_row leaves exp(s_ij - m) in p; normalise by their sum */
    double sum = 0.0;
    for (int j = 0; j <= i; ++j) sum += p[j];
    for (int j = 0; j <= i; ++j) p[j] /= sum;
    rc = ORACLE_OK;
  }
  free(Kr); free(V); free(tmp); free(orow);
  return rc;
}

/* ------------------------------------------------------------------------------
 * Incremental decode (one new token per sequence against a cache of earlier ones).
 *
 * The FasterTransformer guide ("GPT-NeoX on FasterTransformer", section "背景")
 * names a per-token decoder that extends a growing context; it prints no
 * interface.  Reading used here (listed in the design notes):
 *  - sequence b already holds pos[b] tokens, at positions 0..pos[b]-1; the new
 *    token sits at position pos[b];
 *  - the cache keeps the projections as they came, keys NOT rotated:
 *    k_cache[b,h,p,:], v_cache[b,h,p,:] for p < pos[b] (bf16, [B,H,Smax,D]);
 *  - the new token's packed projection is qkv_new[b,h,0|1|2,:] (bf16, [B,H,3,D]),
 *    the per-token [H,3,D] packing of the prefill input;
 *  - the new query attends to keys 0..pos[b] (itself included), each rotated at
 *    its own position exactly as in the prefill, scaled by 1/sqrt(D).
 * The result is by definition row pos[b] of the prefill over the whole sequence.
 * Cache rows p >= pos[b] are never read.
 * out: fp64 [B,H,D];  lse: fp64 [B,H] (natural log).  Returns 0 or < 0.          */
typedef struct {
  const uint16_t *qkv_new, *k_cache, *v_cache;
  const int* pos;
  int B, H, Smax, D, r;
  double base;
  double *out, *lse;
  pthread_mutex_t mu;
  int64_t next, n_items;
  int failed;
} djob_t;

static void* worker_decode(void* arg) {
  djob_t* J = (djob_t*)arg;
  const int D = J->D;
  double* x = malloc(sizeof(double) * (size_t)D);
  double* qr = malloc(sizeof(double) * (size_t)D);
  double* kr = malloc(sizeof(double) * (size_t)D);
  double* scores = malloc(sizeof(double) * (size_t)(J->Smax + 1));
  if (!x || !qr || !kr || !scores) {
    pthread_mutex_lock(&J->mu);
    J->failed = 1;
    pthread_mutex_unlock(&J->mu);
    free(x); free(qr); free(kr); free(scores);
    return NULL;
  }
  const double inv_sqrt_d = 1.0 / sqrt((double)D);
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int64_t item = J->next < J->n_items ? J->next++ : -1;
    pthread_mutex_unlock(&J->mu);
    if (item < 0) break;
    const int64_t b = item / J->H, h = item % J->H;
    const int64_t P = J->pos[b];
    const uint16_t* nq = J->qkv_new + ((b * J->H + h) * 3 + 0) * (int64_t)D;
    for (int d = 0; d < D; ++d) x[d] = bf16_to_f64(nq[d]);
    neox_oracle_rotate(x, D, J->r, J->base, P, qr);
    /* scores of keys 0..P */
    double m = -INFINITY;
    for (int64_t p = 0; p <= P; ++p) {
      const uint16_t* k = p < P ? J->k_cache + ((b * J->H + h) * J->Smax + p) * (int64_t)D
                                : J->qkv_new + ((b * J->H + h) * 3 + 1) * (int64_t)D;
      for (int d = 0; d < D; ++d) x[d] = bf16_to_f64(k[d]);
      neox_oracle_rotate(x, D, J->r, J->base, p, kr);
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qr[d] * kr[d];
      scores[p] = dot * inv_sqrt_d;
      if (scores[p] > m) m = scores[p];
    }
    double l = 0.0;
    for (int64_t p = 0; p <= P; ++p) {
      scores[p] = exp(scores[p] - m);
      l += scores[p];
    }
    double* o = J->out + (b * J->H + h) * (int64_t)D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t p = 0; p <= P; ++p) {
      const uint16_t* v = p < P ? J->v_cache + ((b * J->H + h) * J->Smax + p) * (int64_t)D
                                : J->qkv_new + ((b * J->H + h) * 3 + 2) * (int64_t)D;
      const double w = scores[p] / l;
      for (int d = 0; d < D; ++d) o[d] += w * bf16_to_f64(v[d]);
    }
    J->lse[b * J->H + h] = m + log(l);
  }
  free(x); free(qr); free(kr); free(scores);
  return NULL;
}

int neox_oracle_decode(const uint16_t* qkv_new, const uint16_t* k_cache, const uint16_t* v_cache, const int* pos,
                       int B, int H, int Smax, int D, int r, double base, double* out, double* lse, int threads) {
  if (!qkv_new || !pos || !out || !lse || B < 1 || H < 1 || Smax < 1 || D < 1 || r < 0 || r > D || (r & 1) ||
      !(base > 0.0))
    return ORACLE_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    if (pos[b] < 0 || pos[b] >= Smax) return ORACLE_ERR_ARG;
    if (pos[b] > 0 && (!k_cache || !v_cache)) return ORACLE_ERR_ARG;
  }
  djob_t J;
  memset(&J, 0, sizeof J);
  J.qkv_new = qkv_new; J.k_cache = k_cache; J.v_cache = v_cache; J.pos = pos;
  J.B = B; J.H = H; J.Smax = Smax; J.D = D; J.r = r; J.base = base; J.out = out; J.lse = lse;
  J.n_items = (int64_t)B * H;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  pthread_mutex_init(&J.mu, NULL);
  int started = 0;
  for (int t = 1; t < threads; ++t)
    if (pthread_create(&tid[started], NULL, worker_decode, &J) == 0) ++started;
  worker_decode(&J);
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&J.mu);
  return J.failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ---------------------------------------------------------------- backward ----
 * Gradients of the loss L = sum(dout * out) with respect to the packed qkv, where
 * out is the forward above.  The chain rule through each step of the forward, in
 * its order ("gpt-neox - 模型与框架" page, section "问题二：注意力计算太慢", names the
 * exact attention being differentiated; the rotation is the same rotate-half map):
 *   p_ij = softmax_j(s_ij), s_ij = q'_i.k'_j / sqrt(D)  (j <= i),  o_i = sum_j p_ij v_j
 *   dv_j  = sum_{i >= j} p_ij dout_i
 *   dp_ij = dout_i . v_j,   delta_i = dout_i . o_i = sum_j p_ij dp_ij
 *   ds_ij = p_ij (dp_ij - delta_i)          (softmax Jacobian applied to dp)
 *   dq'_i = sum_j ds_ij k'_j / sqrt(D),   dk'_j = sum_{i >= j} ds_ij q'_i / sqrt(D)
 *   dq_i = R(i)^T dq'_i,  dk_j = R(j)^T dk'_j  (R(p)^T is the rotation by -p theta).
 * o_i and delta_i are recomputed here in fp64, not taken from a forward pass.   */
typedef struct {
  const uint16_t* qkv;
  const uint16_t* dout;
  int B, S, H, D, r;
  double base;
  double* dqkv;
  pthread_mutex_t mu;
  int64_t next, n_items;
  int failed;
} bjob_t;

static void* worker_bwd(void* arg) {
  bjob_t* J = (bjob_t*)arg;
  const int S = J->S, H = J->H, D = J->D;
  const double inv_sqrt_d = 1.0 / sqrt((double)D);
  double* Qr = malloc(sizeof(double) * (size_t)S * D);
  double* Kr = malloc(sizeof(double) * (size_t)S * D);
  double* V = malloc(sizeof(double) * (size_t)S * D);
  double* dO = malloc(sizeof(double) * (size_t)S * D);
  double* dQr = malloc(sizeof(double) * (size_t)S * D);
  double* dKr = malloc(sizeof(double) * (size_t)S * D);
  double* dV = malloc(sizeof(double) * (size_t)S * D);
  double* p = malloc(sizeof(double) * (size_t)S);
  double* dp = malloc(sizeof(double) * (size_t)S);
  double* tmp = malloc(sizeof(double) * (size_t)D);
  double* o = malloc(sizeof(double) * (size_t)D);
  if (!Qr || !Kr || !V || !dO || !dQr || !dKr || !dV || !p || !dp || !tmp || !o) {
    pthread_mutex_lock(&J->mu);
    J->failed = 1;
    pthread_mutex_unlock(&J->mu);
  } else {
    for (;;) {
      pthread_mutex_lock(&J->mu);
      int64_t item = J->next < J->n_items ? J->next++ : -1;
      pthread_mutex_unlock(&J->mu);
      if (item < 0) break;
      const int64_t b = item / H, h = item % H;
      for (int64_t s = 0; s < S; ++s) {
        const uint16_t* qs = J->qkv + qkv_off(b, s, h, 0, S, H, D);
        const uint16_t* ks = J->qkv + qkv_off(b, s, h, 1, S, H, D);
        const uint16_t* vs = J->qkv + qkv_off(b, s, h, 2, S, H, D);
        const uint16_t* g = J->dout + ((b * S + s) * H + h) * (int64_t)D;
        for (int d = 0; d < D; ++d) tmp[d] = bf16_to_f64(qs[d]);
        neox_oracle_rotate(tmp, D, J->r, J->base, s, Qr + s * D);
        for (int d = 0; d < D; ++d) tmp[d] = bf16_to_f64(ks[d]);
        neox_oracle_rotate(tmp, D, J->r, J->base, s, Kr + s * D);
        for (int d = 0; d < D; ++d) {
          V[s * D + d] = bf16_to_f64(vs[d]);
          dO[s * D + d] = bf16_to_f64(g[d]);
        }
      }
      memset(dQr, 0, sizeof(double) * (size_t)S * D);
      memset(dKr, 0, sizeof(double) * (size_t)S * D);
      memset(dV, 0, sizeof(double) * (size_t)S * D);
      for (int64_t i = 0; i < S; ++i) {
        /* forward row i: probabilities and output */
        double m = -INFINITY;
        for (int64_t j = 0; j <= i; ++j) {
          double dot = 0.0;
          for (int d = 0; d < D; ++d) dot += Qr[i * D + d] * Kr[j * D + d];
          p[j] = dot * inv_sqrt_d;
          if (p[j] > m) m = p[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j <= i; ++j) {
          p[j] = exp(p[j] - m);
          l += p[j];
        }
        for (int64_t j = 0; j <= i; ++j) p[j] /= l;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t j = 0; j <= i; ++j)
          for (int d = 0; d < D; ++d) o[d] += p[j] * V[j * D + d];
        /* backward of row i */
        double delta = 0.0;
        for (int d = 0; d < D; ++d) delta += dO[i * D + d] * o[d];
        for (int64_t j = 0; j <= i; ++j) {
          double acc = 0.0;
          for (int d = 0; d < D; ++d) acc += dO[i * D + d] * V[j * D + d];
          dp[j] = acc;
          for (int d = 0; d < D; ++d) dV[j * D + d] += p[j] * dO[i * D + d];
        }
        for (int64_t j = 0; j <= i; ++j) {
          const double ds = p[j] * (dp[j] - delta) * inv_sqrt_d;
          for (int d = 0; d < D; ++d) {
            dQr[i * D + d] += ds * Kr[j * D + d];
            dKr[j * D + d] += ds * Qr[i * D + d];
          }
        }
      }
      /* back through the rotation: R(s)^T = R(-s) */
      for (int64_t s = 0; s < S; ++s) {
        double* gq = J->dqkv + qkv_off(b, s, h, 0, S, H, D);
        double* gk = J->dqkv + qkv_off(b, s, h, 1, S, H, D);
        double* gv = J->dqkv + qkv_off(b, s, h, 2, S, H, D);
        neox_oracle_rotate(dQr + s * D, D, J->r, J->base, -s, gq);
        neox_oracle_rotate(dKr + s * D, D, J->r, J->base, -s, gk);
        for (int d = 0; d < D; ++d) gv[d] = dV[s * D + d];
      }
    }
  }
  free(Qr);
  free(Kr);
  free(V);
  free(dO);
  free(dQr);
  free(dKr);
  free(dV);
  free(p);
  free(dp);
  free(tmp);
  free(o);
  return NULL;
}

/* dqkv: fp64 [B,S,H,3,D], every element written.  dout: bf16 bits [B,S,H,D]. */
int neox_oracle_bwd(const uint16_t* qkv, const uint16_t* dout, int B, int S, int H, int D, int r, double base,
                    double* dqkv, int threads) {
  if (check_args(qkv, B, S, H, D, r, base) != ORACLE_OK || !dout || !dqkv) return ORACLE_ERR_ARG;
  bjob_t J;
  memset(&J, 0, sizeof J);
  J.qkv = qkv;
  J.dout = dout;
  J.B = B;
  J.S = S;
  J.H = H;
  J.D = D;
  J.r = r;
  J.base = base;
  J.dqkv = dqkv;
  J.n_items = (int64_t)B * H;
  pthread_mutex_init(&J.mu, NULL);
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  int started = 0;
  for (int t = 0; t < threads; ++t)
    if (pthread_create(&tid[t], NULL, worker_bwd, &J) == 0) ++started;
  if (started == 0) worker_bwd(&J);
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&J.mu);
  return J.failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ------------------------------------------------------------------ ALiBi ----
 * The pages name ALiBi ("linear bias attention") as GPT-NeoX's other positional scheme
 * ("gpt-neox - 模型与框架" page, section "位置编码"; GPT-NeoX library summary, "Key
 * capabilities") but print no formula.  Reading: the scheme as published with the
 * method (Press et al., "Train Short, Test Long"): no rotation; head h adds
 * -m_h * (i - j) to the score of query i and key j <= i; the slopes form a geometric
 * sequence 2^(-8/n), 2^(-16/n), ... for a power-of-two head count n, and for other head
 * counts the slopes of the largest power of two n below H are followed by every other
 * slope of 2n (the odd-numbered ones), until H slopes are reached.                  */
void neox_oracle_alibi_slopes(int H, double* slopes) {
  int n = 1;
  while (n * 2 <= H) n *= 2;
  for (int k = 0; k < n && k < H; ++k) slopes[k] = pow(2.0, -8.0 * (double)(k + 1) / (double)n);
  for (int k = n, e = 1; k < H; ++k, e += 2) slopes[k] = pow(2.0, -8.0 * (double)e / (double)(2 * n));
}

typedef struct {
  const uint16_t* qkv;
  int B, S, H, D;
  const double* slopes;
  double* out;
  double* lse;
  pthread_mutex_t mu;
  int64_t next, n_items;
  int failed;
} ajob_t;

static void* worker_alibi(void* arg) {
  ajob_t* J = (ajob_t*)arg;
  const int S = J->S, H = J->H, D = J->D;
  const double inv_sqrt_d = 1.0 / sqrt((double)D);
  double* sc = malloc(sizeof(double) * (size_t)S);
  double* q = malloc(sizeof(double) * (size_t)D);
  if (!sc || !q) {
    pthread_mutex_lock(&J->mu);
    J->failed = 1;
    pthread_mutex_unlock(&J->mu);
  } else {
    for (;;) {
      pthread_mutex_lock(&J->mu);
      int64_t item = J->next < J->n_items ? J->next++ : -1;
      pthread_mutex_unlock(&J->mu);
      if (item < 0) break;
      /* item = (b, h, i): one query row */
      const int64_t i = item % S, bh = item / S, h = bh % H, b = bh / H;
      const double m_h = J->slopes[h];
      const uint16_t* qs = J->qkv + qkv_off(b, i, h, 0, S, H, D);
      for (int d = 0; d < D; ++d) q[d] = bf16_to_f64(qs[d]);
      double mx = -INFINITY;
      for (int64_t j = 0; j <= i; ++j) {
        const uint16_t* kj = J->qkv + qkv_off(b, j, h, 1, S, H, D);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * bf16_to_f64(kj[d]);
        sc[j] = dot * inv_sqrt_d - m_h * (double)(i - j);
        if (sc[j] > mx) mx = sc[j];
      }
      double l = 0.0;
      for (int64_t j = 0; j <= i; ++j) {
        sc[j] = exp(sc[j] - mx);
        l += sc[j];
      }
      double* o = J->out + ((b * S + i) * H + h) * (int64_t)D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (int64_t j = 0; j <= i; ++j) {
        const uint16_t* vj = J->qkv + qkv_off(b, j, h, 2, S, H, D);
        for (int d = 0; d < D; ++d) o[d] += sc[j] / l * bf16_to_f64(vj[d]);
      }
      J->lse[(b * H + h) * (int64_t)S + i] = mx + log(l);
    }
  }
  free(sc);
  free(q);
  return NULL;
}

/* Causal attention with the ALiBi bias instead of the rotation.
 * qkv: bf16 bits [B,S,H,3,D]; out fp64 [B,S,H,D]; lse fp64 [B,H,S] (natural log). */
int neox_oracle_fwd_alibi(const uint16_t* qkv, int B, int S, int H, int D, double* out, double* lse, int threads) {
  if (!qkv || !out || !lse || B < 1 || S < 1 || H < 1 || D < 1) return ORACLE_ERR_ARG;
  double* slopes = malloc(sizeof(double) * (size_t)H);
  if (!slopes) return ORACLE_ERR_NOMEM;
  neox_oracle_alibi_slopes(H, slopes);
  ajob_t J;
  memset(&J, 0, sizeof J);
  J.qkv = qkv;
  J.B = B;
  J.S = S;
  J.H = H;
  J.D = D;
  J.slopes = slopes;
  J.out = out;
  J.lse = lse;
  J.n_items = (int64_t)B * H * S;
  pthread_mutex_init(&J.mu, NULL);
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  int started = 0;
  for (int t = 0; t < threads; ++t)
    if (pthread_create(&tid[t], NULL, worker_alibi, &J) == 0) ++started;
  if (started == 0) worker_alibi(&J);
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&J.mu);
  free(slopes);
  return J.failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Fused query_key_value projection (the step just before the attention).
 *
 * "GPT-NeoX on FasterTransformer" guide, section "从 HuggingFace 检查点部署": the
 * HuggingFace checkpoint stores attention.query_key_value.weight as
 * [hidden_size, num_heads, 3, head_hidden], so output feature n = (h*3 + slot)*D + d of
 * token t is sum_k x[t,k] * w[k,n], and the tokens' outputs form the packed qkv
 * [B,S,H,3,D] the attention reads.  The layer list on the same page
 * ("attention.query_key_value.*") includes its bias, added to every token (optional
 * here: bias == NULL means none).
 *
 *   out[t, n] = sum_{k < K} x[t, k] * w[k, n] + bias[n]      (fp64, exact bf16 inputs)
 *
 * x: bf16 bits [M, K] (token-major), w: bf16 bits [K, N], bias: bf16 bits [N] or NULL,
 * out: fp64 [n_rows, N] for the listed token rows (rows == NULL: all M rows in order).
 * ------------------------------------------------------------------------- */
typedef struct {
  const uint16_t* x;
  const uint16_t* w;
  const uint16_t* bias;
  int64_t M;
  int K, N;
  const int64_t* rows;
  int64_t n_rows;
  double* out;
  pthread_mutex_t mu;
  int64_t next;
  int failed;
} pjob_t;

static void* worker_proj(void* arg) {
  pjob_t* J = (pjob_t*)arg;
  const int K = J->K, N = J->N;
  double* xr = malloc(sizeof(double) * (size_t)K);
  if (!xr) {
    pthread_mutex_lock(&J->mu);
    J->failed = 1;
    pthread_mutex_unlock(&J->mu);
    return NULL;
  }
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int64_t it = J->next++;
    pthread_mutex_unlock(&J->mu);
    if (it >= J->n_rows) break;
    const int64_t t = J->rows ? J->rows[it] : it;
    for (int k = 0; k < K; ++k) xr[k] = bf16_to_f64(J->x[t * K + k]);
    double* o = J->out + it * (int64_t)N;
    for (int n = 0; n < N; ++n) o[n] = J->bias ? bf16_to_f64(J->bias[n]) : 0.0;
    for (int k = 0; k < K; ++k) {
      const uint16_t* wk = J->w + (int64_t)k * N;
      const double a = xr[k];
      for (int n = 0; n < N; ++n) o[n] += a * bf16_to_f64(wk[n]);
    }
  }
  free(xr);
  return NULL;
}

int neox_oracle_qkv_proj(const uint16_t* x, const uint16_t* w, const uint16_t* bias, int64_t M, int K, int N,
                         const int64_t* rows, int64_t n_rows, double* out, int threads) {
  if (!x || !w || !out || M < 1 || K < 1 || N < 1) return ORACLE_ERR_ARG;
  if (rows) {
    for (int64_t i = 0; i < n_rows; ++i)
      if (rows[i] < 0 || rows[i] >= M) return ORACLE_ERR_ARG;
  } else {
    n_rows = M;
  }
  pjob_t J;
  memset(&J, 0, sizeof J);
  J.x = x;
  J.w = w;
  J.bias = bias;
  J.M = M;
  J.K = K;
  J.N = N;
  J.rows = rows;
  J.n_rows = n_rows;
  J.out = out;
  pthread_mutex_init(&J.mu, NULL);
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  int started = 0;
  for (int t = 0; t < threads; ++t)
    if (pthread_create(&tid[t], NULL, worker_proj, &J) == 0) ++started;
  if (started == 0) worker_proj(&J);
  for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&J.mu);
  return J.failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}
