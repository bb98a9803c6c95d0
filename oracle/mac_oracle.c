/*
 * mac_oracle.c -- plain, slow, fp64 CPU oracle of MAC-Attention's per-step
 * decode attention (Match -> Complete -> rectify-append, with the exact
 * full-attention fallback on a miss).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path loads, links or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library; both sides read the same raw input buffers and nothing else.
 *
 * Sources (the pages this follows; section names are translated):
 *   [MAC]  "MAC-Attention: Match-Amend-Complete attention reuse, up to 99%
 *          fewer KV reads in long-context decoding (MLSys 2026)",
 *          pinghaoyang.com.cn blog post.
 *   [MACS] "MAC-Attention: A Match-Amend-Complete Scheme for Fast and
 *          Accurate Attention Computation (MLSys 2026)",
 *          awesome-system-papers summary.
 *   [ACSP] "Attention Cache and Sequence Parallelism", shaojiemike.top.
 *
 * Notation: positions are 1-based; m is the current length and the K/V of
 * position m is already in the cache ([ACSP] "Why only K/V are cached":
 * the cache is appended before the new query reads it).  h is a query head,
 * g = h / (Hq/Hkv) its KV head ([ACSP] MHA decode pseudo-code, repeat_kv).
 * A summary is (M, Z, S): running max M, Z = sum exp(l_t - M),
 * S = sum exp(l_t - M) V_t; the empty summary is (-inf, 0, 0)
 * ([MAC] "Decomposable attention": o = S/Z; "Complete": summaries are kept
 * with their running max subtracted).
 *
 * Precision: every arithmetic step is fp64.  Inputs are bf16 (raw 16-bit
 * patterns, the upper half of an IEEE binary32) or fp32; both convert to
 * fp64 exactly.
 *
 * Parity pins (what checks this file against the pages, not against itself)
 * live in tests/test_oracle_pins.py; the hit path's output quality relative
 * to exact attention is an approximation whose error bound the pages lost,
 * so it is reported, not pinned.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OC_BF16 = 0, OC_F32 = 1 };
enum { OC_THR_ONE_MINUS_TAU = 0, OC_THR_TAU = 1 };
enum { OC_ROPE_HALF = 0, OC_ROPE_INTERLEAVED = 1, OC_ROPE_NONE = 2 };

typedef struct {
  int batch, n_q_heads, n_kv_heads, head_dim;
  int ring_k, band_r;
  double tau;
  int thr_mode;
  double rope_base;
  int rope_mode;
  int dtype;        /* element type of the query, ring-query, K and V inputs */
  int page_size;    /* 0 = contiguous [B][Hkv][capacity][d]; else paged */
  int min_context;  /* steps with m < min_context never reuse */
  int front_sink;   /* F: tokens [1, F] kept out of the reused summaries and
                       attended exactly at every step (0 = none) */
} oc_config;

typedef struct {
  const void *k, *v;
  const int32_t *page_table; /* [B][max_pages] for paged caches */
  int64_t capacity;          /* contiguous: tokens per (b, g) block */
  int32_t max_pages;
} oc_kv;

/* Per-request rings of capacity K ([MAC] "Paper version: K1/K2/K3"): one
 * position per slot and request, the stored pre-RoPE query per (b, h, slot)
 * and the rectified summary per (b, h, slot). */
typedef struct {
  int32_t *pos; /* [B][K], 0 = never written */
  double *q;    /* [B][Hq][K][d] */
  double *sM;   /* [B][Hq][K] */
  double *sZ;   /* [B][Hq][K] */
  double *sS;   /* [B][Hq][K][d] */
} oc_ring;

/* ------------------------------------------------------------------ */
/* element access                                                      */
/* ------------------------------------------------------------------ */

static double load_elem(const void *base, int dtype, int64_t i) {
  if (dtype == OC_F32) return (double)((const float *)base)[i];
  uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Offset (in elements) of row t (1-based) of KV head g of request b. */
static int64_t kv_row(const oc_config *c, const oc_kv *kv, int b, int g, int64_t t) {
  int d = c->head_dim;
  if (c->page_size == 0)
    return (((int64_t)b * c->n_kv_heads + g) * kv->capacity + (t - 1)) * d;
  int64_t page = kv->page_table[(int64_t)b * kv->max_pages + (t - 1) / c->page_size];
  return ((page * c->n_kv_heads + g) * c->page_size + (t - 1) % c->page_size) * d;
}

/* ------------------------------------------------------------------ */
/* threshold, RoPE                                                     */
/* ------------------------------------------------------------------ */

/* Squared acceptance threshold ([MAC] "Match (2)": the Gaussian null puts a
 * chance distance at sqrt(2d); accept when the distance is below
 * (1 - tau) sqrt(2d) -- d=128, tau=0.45 gives 8.8, larger tau is stricter,
 * and the K1 pseudo-code misses when d2 >= 2d(1-tau)^2.  The summary page
 * writes tau*sqrt(2d); OC_THR_TAU selects that reading.)  Computed in fp64
 * and rounded once to fp32, the precision the comparison is made in. */
double oc_threshold_sq(int head_dim, double tau, int thr_mode) {
  double f = (thr_mode == OC_THR_TAU) ? tau : (1.0 - tau);
  double thr = f * sqrt(2.0 * (double)head_dim);
  return (double)(float)(thr * thr);
}

/* q = R(pos) x: RoPE as a direct product of 2x2 rotations ([MAC] "Match
 * (1)"), frequency w_j = base^(-2j/d), angle (pos-1) w_j (the first position
 * has angle 0).  HALF pairs (j, j+d/2); INTERLEAVED pairs (2j, 2j+1).  The
 * rotation is [a, b] -> [a cos - b sin, b cos + a sin] (RoFormer). */
void oc_rope(const double *x, int64_t pos, int d, double base, int mode, double *out) {
  if (mode == OC_ROPE_NONE) {
    memcpy(out, x, sizeof(double) * (size_t)d);
    return;
  }
  int half = d / 2;
  for (int j = 0; j < half; ++j) {
    double w = pow(base, -2.0 * (double)j / (double)d);
    double ang = (double)(pos - 1) * w;
    double cs = cos(ang), sn = sin(ang);
    int ia = (mode == OC_ROPE_HALF) ? j : 2 * j;
    int ib = (mode == OC_ROPE_HALF) ? j + half : 2 * j + 1;
    double a = x[ia], b = x[ib];
    out[ia] = a * cs - b * sn;
    out[ib] = b * cs + a * sn;
  }
}

/* ------------------------------------------------------------------ */
/* summaries                                                           */
/* ------------------------------------------------------------------ */

/* Summary of query q (already rotated) over tokens [lo, hi] of KV head g of
 * request b.  l_t = q . K_t / sqrt(d) ([ACSP] MHA decode: scores =
 * q K^T * scale).  M = max l_t, Z = sum exp(l_t - M), S = sum exp(l_t - M) V_t.
 * An empty range gives (-inf, 0, 0). */
void oc_summary(const oc_config *c, const oc_kv *kv, int b, int g, const double *q,
                int64_t lo, int64_t hi, double *M, double *Z, double *S) {
  int d = c->head_dim;
  if (lo < 1) lo = 1;
  *M = -INFINITY;
  *Z = 0.0;
  for (int i = 0; i < d; ++i) S[i] = 0.0;
  if (lo > hi) return;
  int64_t n = hi - lo + 1;
  double *logit = (double *)malloc(sizeof(double) * (size_t)n);
  double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int64_t t = lo; t <= hi; ++t) {
    int64_t row = kv_row(c, kv, b, g, t);
    double dot = 0.0;
    for (int i = 0; i < d; ++i) dot += q[i] * load_elem(kv->k, c->dtype, row + i);
    double l = dot * scale;
    logit[t - lo] = l;
    if (l > mx) mx = l;
  }
  double z = 0.0;
  for (int64_t t = lo; t <= hi; ++t) {
    int64_t row = kv_row(c, kv, b, g, t);
    double e = exp(logit[t - lo] - mx);
    z += e;
    for (int i = 0; i < d; ++i) S[i] += e * load_elem(kv->v, c->dtype, row + i);
  }
  free(logit);
  *M = mx;
  *Z = z;
}

/* acc <- acc (+) x.  Summaries of disjoint sets add once brought to a common
 * max ([MAC] "Decomposable attention" and "Complete"; written out in
 * [ACSP] "MHA decode needs a distributed softmax": m = max m_r,
 * l = sum exp(m_r - m) l_r, u = sum exp(m_r - m) u_r).  The empty summary is
 * the identity. */
void oc_merge(int d, double *accM, double *accZ, double *accS,
              double xM, double xZ, const double *xS) {
  if (xZ == 0.0) return;
  if (*accZ == 0.0) {
    *accM = xM;
    *accZ = xZ;
    for (int i = 0; i < d; ++i) accS[i] = xS[i];
    return;
  }
  double mnew = (*accM > xM) ? *accM : xM;
  double fa = exp(*accM - mnew), fx = exp(xM - mnew);
  *accZ = *accZ * fa + xZ * fx;
  for (int i = 0; i < d; ++i) accS[i] = accS[i] * fa + xS[i] * fx;
  *accM = mnew;
}

/* ------------------------------------------------------------------ */
/* match                                                               */
/* ------------------------------------------------------------------ */

/* Nearest neighbour of the pre-RoPE query qt among the ring entries of
 * (b, h) whose position lies in the recent window [m-K, m-1] ([MAC]
 * "Match (3)": candidates are the last K tokens; the current token is not
 * in the ring yet).  Distance is squared L2 ([MAC] "Match (2)"), ties go to
 * the most recent position (it skips the longest prefix, "Match (3)").
 * Returns the matched position or -1 when no slot is a candidate; *dmin and
 * *dsecond receive the smallest and second-smallest distance. */
static int64_t match_head(const oc_config *c, const oc_ring *ring, int b, int h,
                          const double *qt, int64_t m, double *dmin, double *dsecond) {
  int K = c->ring_k, d = c->head_dim;
  int64_t best = -1;
  double bestD = INFINITY, secondD = INFINITY;
  for (int s = 0; s < K; ++s) {
    int64_t p = ring->pos[(int64_t)b * K + s];
    if (p < 1 || p > m - 1 || p < m - K) continue;
    const double *qc = ring->q + (((int64_t)b * c->n_q_heads + h) * K + s) * d;
    double D = 0.0;
    for (int i = 0; i < d; ++i) {
      double diff = qt[i] - qc[i];
      D += diff * diff;
    }
    if (D < bestD || (D == bestD && p > best)) {
      secondD = bestD;
      bestD = D;
      best = p;
    } else if (D < secondD) {
      secondD = D;
    }
  }
  *dmin = bestD;
  *dsecond = secondD;
  return best;
}

/* ------------------------------------------------------------------ */
/* threads over (b, h)                                                 */
/* ------------------------------------------------------------------ */

typedef struct {
  void (*fn)(void *ctx, int64_t idx);
  void *ctx;
  int64_t n;
  int64_t next;
  pthread_mutex_t mu;
} pool_t;

static void *pool_worker(void *arg) {
  pool_t *p = (pool_t *)arg;
  for (;;) {
    pthread_mutex_lock(&p->mu);
    int64_t i = p->next++;
    pthread_mutex_unlock(&p->mu);
    if (i >= p->n) break;
    p->fn(p->ctx, i);
  }
  return NULL;
}

static void run_parallel(int n_threads, int64_t n, void (*fn)(void *, int64_t), void *ctx) {
  if (n_threads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(ctx, i);
    return;
  }
  if (n_threads > n) n_threads = (int)n;
  pool_t p;
  p.fn = fn;
  p.ctx = ctx;
  p.n = n;
  p.next = 0;
  pthread_mutex_init(&p.mu, NULL);
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  for (int t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, pool_worker, &p);
  for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
  free(th);
  pthread_mutex_destroy(&p.mu);
}

/* ------------------------------------------------------------------ */
/* one decode step                                                     */
/* ------------------------------------------------------------------ */

typedef struct {
  const oc_config *c;
  oc_ring *ring;
  const void *q_pre;
  const int32_t *seq_len;
  const oc_kv *kv;
  const uint8_t *head_mask;
  double thr2;
  double *out;
  int32_t *match_pos;
  double *dmin, *dsecond;
  double *newM, *newZ, *newS; /* AS_{1:m-r} per (b, h), appended in phase 2 */
} step_ctx;

static void step_head(void *vctx, int64_t idx) {
  step_ctx *x = (step_ctx *)vctx;
  const oc_config *c = x->c;
  int Hq = c->n_q_heads, d = c->head_dim, K = c->ring_k, r = c->band_r;
  int G = Hq / c->n_kv_heads;
  int b = (int)(idx / Hq), h = (int)(idx % Hq), g = h / G;
  int64_t m = x->seq_len[b];

  double *qt = (double *)malloc(sizeof(double) * (size_t)d);
  for (int i = 0; i < d; ++i) qt[i] = load_elem(x->q_pre, c->dtype, idx * d + i);

  /* Match ([MAC] K1): nearest ring entry, accepted strictly below thr^2. */
  double dmin, dsecond;
  int64_t p = match_head(c, x->ring, b, h, qt, m, &dmin, &dsecond);
  int hit = (p >= 1) && (dmin < x->thr2) && (m >= c->min_context);
  x->match_pos[idx] = hit ? (int32_t)p : -1;
  x->dmin[idx] = dmin;
  x->dsecond[idx] = dsecond;

  double *nM = x->newM + idx, *nZ = x->newZ + idx, *nS = x->newS + idx * d;
  double *o = x->out + idx * d;
  if (x->head_mask && !x->head_mask[idx]) {
    *nM = NAN;
    *nZ = NAN;
    for (int i = 0; i < d; ++i) nS[i] = NAN, o[i] = NAN;
    free(qt);
    return;
  }

  /* Complete ([MAC] K2): the post-RoPE query attends to the band and tail
   * only.  A hit reuses the cached rectified summary AS_{1:p-r} of slot p;
   * the fresh range starts at p-r+1 (clamped to 1).  A miss has no cached
   * part and attends to [1, m] ([MAC] "Match (1)": fall back to full
   * attention).  With a front sink F ([MAC] "Production version", front
   * sink isolation) the summaries cover [F+1, .] only: the fresh range
   * starts at F+1 at the earliest, and [1, min(F, m)] is attended exactly
   * at every step, joining the output but never a summary. */
  double *q = (double *)malloc(sizeof(double) * (size_t)d);
  oc_rope(qt, m, d, c->rope_base, c->rope_mode, q);
  const int64_t F = c->front_sink;
  int64_t lo = F + 1;
  *nM = -INFINITY;
  *nZ = 0.0;
  for (int i = 0; i < d; ++i) nS[i] = 0.0;
  if (hit) {
    lo = p - r + 1;
    if (lo < F + 1) lo = F + 1;
    int64_t slot = (((int64_t)b * Hq + h) * K + p % K);
    oc_merge(d, nM, nZ, nS, x->ring->sM[slot], x->ring->sZ[slot], x->ring->sS + slot * d);
  }
  /* Split the fresh range at m-r: tokens up to m-r join the cached part to
   * form the new rectified summary AS_{1:m-r} ([MAC] K3: the merged summary
   * minus the last r tokens; accumulating the two parts separately gives it
   * without a log-domain subtraction); the last r tokens complete the
   * output. */
  double bM, bZ, tM, tZ;
  double *bS = (double *)malloc(sizeof(double) * (size_t)d);
  double *tS = (double *)malloc(sizeof(double) * (size_t)d);
  oc_summary(c, x->kv, b, g, q, lo, m - r, &bM, &bZ, bS);
  oc_merge(d, nM, nZ, nS, bM, bZ, bS);
  int64_t tail_lo = m - r + 1;
  if (tail_lo < lo) tail_lo = lo;
  oc_summary(c, x->kv, b, g, q, tail_lo, m, &tM, &tZ, tS);
  double oM = *nM, oZ = *nZ;
  double *oS = (double *)malloc(sizeof(double) * (size_t)d);
  for (int i = 0; i < d; ++i) oS[i] = nS[i];
  oc_merge(d, &oM, &oZ, oS, tM, tZ, tS);
  if (F > 0) {
    /* the sink, exact at this step */
    oc_summary(c, x->kv, b, g, q, 1, F < m ? F : m, &tM, &tZ, tS);
    oc_merge(d, &oM, &oZ, oS, tM, tZ, tS);
  }
  for (int i = 0; i < d; ++i) o[i] = (oZ > 0.0) ? oS[i] / oZ : 0.0;
  free(oS);
  free(bS);
  free(tS);
  free(q);
  free(qt);
}

/* One decode step for every request and query head.  Writes out [B][Hq][d],
 * match_pos [B][Hq] (-1 = miss), dmin/dsecond [B][Hq]; then appends the
 * current position, pre-RoPE query and rectified summary AS_{1:m-r} into
 * ring slot m mod K ([MAC] K3 "rectify-append"; every step appends, hit or
 * miss).  head_mask (optional, [B][Hq]) limits the attention part to the
 * selected heads; the match and the query/position append run for all. */
int oc_decode_step(const oc_config *c, oc_ring *ring, const void *q_pre,
                   const int32_t *seq_len, const oc_kv *kv, const uint8_t *head_mask,
                   double *out, int32_t *match_pos, double *dmin, double *dsecond,
                   int n_threads) {
  int B = c->batch, Hq = c->n_q_heads, d = c->head_dim, K = c->ring_k;
  if (Hq % c->n_kv_heads != 0) return -1;
  for (int b = 0; b < B; ++b)
    if (seq_len[b] < 1) return -2;
  int64_t n = (int64_t)B * Hq;
  step_ctx x;
  x.c = c;
  x.ring = ring;
  x.q_pre = q_pre;
  x.seq_len = seq_len;
  x.kv = kv;
  x.head_mask = head_mask;
  x.thr2 = oc_threshold_sq(d, c->tau, c->thr_mode);
  x.out = out;
  x.match_pos = match_pos;
  x.dmin = dmin;
  x.dsecond = dsecond;
  x.newM = (double *)malloc(sizeof(double) * (size_t)n);
  x.newZ = (double *)malloc(sizeof(double) * (size_t)n);
  x.newS = (double *)malloc(sizeof(double) * (size_t)(n * d));
  run_parallel(n_threads, n, step_head, &x);

  /* Append after every head matched: slot m mod K may hold position m-K,
   * which is still a candidate for this step. */
  for (int64_t idx = 0; idx < n; ++idx) {
    int b = (int)(idx / Hq);
    int64_t m = seq_len[b];
    int64_t slot = idx * K + m % K;
    for (int i = 0; i < d; ++i) ring->q[slot * d + i] = load_elem(q_pre, c->dtype, idx * d + i);
    ring->sM[slot] = x.newM[idx];
    ring->sZ[slot] = x.newZ[idx];
    for (int i = 0; i < d; ++i) ring->sS[slot * d + i] = x.newS[idx * d + i];
  }
  for (int b = 0; b < B; ++b) ring->pos[(int64_t)b * K + seq_len[b] % K] = seq_len[b];
  free(x.newM);
  free(x.newZ);
  free(x.newS);
  return 0;
}

/* ------------------------------------------------------------------ */
/* full attention                                                      */
/* ------------------------------------------------------------------ */

typedef struct {
  const oc_config *c;
  const void *q_pre;
  const int32_t *seq_len;
  const oc_kv *kv;
  const uint8_t *head_mask;
  double *out, *lse;
} full_ctx;

static void full_head(void *vctx, int64_t idx) {
  full_ctx *x = (full_ctx *)vctx;
  const oc_config *c = x->c;
  int Hq = c->n_q_heads, d = c->head_dim, G = Hq / c->n_kv_heads;
  int b = (int)(idx / Hq), h = (int)(idx % Hq);
  double *o = x->out + idx * d;
  if (x->head_mask && !x->head_mask[idx]) {
    for (int i = 0; i < d; ++i) o[i] = NAN;
    if (x->lse) x->lse[idx] = NAN;
    return;
  }
  int64_t m = x->seq_len[b];
  double *qt = (double *)malloc(sizeof(double) * (size_t)d);
  double *q = (double *)malloc(sizeof(double) * (size_t)d);
  double *S = (double *)malloc(sizeof(double) * (size_t)d);
  for (int i = 0; i < d; ++i) qt[i] = load_elem(x->q_pre, c->dtype, idx * d + i);
  oc_rope(qt, m, d, c->rope_base, c->rope_mode, q);
  double M, Z;
  oc_summary(c, x->kv, b, h / G, q, 1, m, &M, &Z, S);
  for (int i = 0; i < d; ++i) o[i] = (Z > 0.0) ? S[i] / Z : 0.0;
  if (x->lse) x->lse[idx] = (Z > 0.0) ? M + log(Z) : -INFINITY;
  free(qt);
  free(q);
  free(S);
}

/* Exact decode attention of every (b, h) over [1, m] ([ACSP] MHA decode:
 * softmax(q K^T / sqrt(d)) V with the GQA head map).  out [B][Hq][d];
 * lse [B][Hq] (natural log of the softmax denominator) or NULL. */
int oc_full_attention(const oc_config *c, const void *q_pre, const int32_t *seq_len,
                      const oc_kv *kv, const uint8_t *head_mask, double *out, double *lse,
                      int n_threads) {
  if (c->n_q_heads % c->n_kv_heads != 0) return -1;
  full_ctx x;
  x.c = c;
  x.q_pre = q_pre;
  x.seq_len = seq_len;
  x.kv = kv;
  x.head_mask = head_mask;
  x.out = out;
  x.lse = lse;
  run_parallel(n_threads, (int64_t)c->batch * c->n_q_heads, full_head, &x);
  return 0;
}

/* ------------------------------------------------------------------ */
/* seeding the rings                                                   */
/* ------------------------------------------------------------------ */

typedef struct {
  const oc_config *c;
  oc_ring *ring;
  const void *q_seed;
  const int32_t *prompt_len;
  int n_seed;
  const oc_kv *kv;
  const uint8_t *head_mask;
} seed_ctx;

static void seed_head(void *vctx, int64_t idx) {
  seed_ctx *x = (seed_ctx *)vctx;
  const oc_config *c = x->c;
  int Hq = c->n_q_heads, d = c->head_dim, K = c->ring_k, G = Hq / c->n_kv_heads;
  int b = (int)(idx / Hq), h = (int)(idx % Hq);
  int64_t L = x->prompt_len[b];
  double *qt = (double *)malloc(sizeof(double) * (size_t)d);
  double *q = (double *)malloc(sizeof(double) * (size_t)d);
  for (int i = 0; i < x->n_seed; ++i) {
    int64_t p = L - x->n_seed + 1 + i;
    if (p < 1) continue;
    int64_t slot = idx * K + p % K;
    for (int j = 0; j < d; ++j)
      qt[j] = load_elem(x->q_seed, c->dtype, (idx * x->n_seed + i) * d + j);
    for (int j = 0; j < d; ++j) x->ring->q[slot * d + j] = qt[j];
    if (x->head_mask && !x->head_mask[idx]) {
      x->ring->sM[slot] = NAN;
      x->ring->sZ[slot] = NAN;
      continue;
    }
    oc_rope(qt, p, d, c->rope_base, c->rope_mode, q);
    /* with a front sink F, the summary leaves out [1, F] */
    oc_summary(c, x->kv, b, h / G, q, (int64_t)c->front_sink + 1, p - c->band_r, &x->ring->sM[slot],
               &x->ring->sZ[slot], x->ring->sS + slot * d);
  }
  free(qt);
  free(q);
}

/* Fill the rings as if positions L-n_seed+1 .. L (L = prompt length) had
 * been decoded with exact attention: slot p mod K holds position p, the
 * seed query and the exact rectified summary AS_{1:p-r} of R(p) q_seed.
 * Slots not seeded are cleared.  (The pages keep prefill on the baseline
 * path and degrade requests whose rings are not ready to exact attention;
 * an all-miss history is what exact attention would have left behind.) */
int oc_seed_rings(const oc_config *c, oc_ring *ring, const void *q_seed,
                  const int32_t *prompt_len, int n_seed, const oc_kv *kv,
                  const uint8_t *head_mask, int n_threads) {
  int B = c->batch, K = c->ring_k;
  if (n_seed > K) return -3;
  for (int64_t i = 0; i < (int64_t)B * K; ++i) ring->pos[i] = 0;
  seed_ctx x;
  x.c = c;
  x.ring = ring;
  x.q_seed = q_seed;
  x.prompt_len = prompt_len;
  x.n_seed = n_seed;
  x.kv = kv;
  x.head_mask = head_mask;
  run_parallel(n_threads, (int64_t)B * c->n_q_heads, seed_head, &x);
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < n_seed; ++i) {
      int64_t p = (int64_t)prompt_len[b] - n_seed + 1 + i;
      if (p >= 1) ring->pos[(int64_t)b * K + p % K] = (int32_t)p;
    }
  return 0;
}

/* The ready gate ([MAC] "Production version": request state that a captured
 * graph can gate).  A request whose flag is set starts over with an empty
 * ring: no slot holds a position, so its next decode step has no candidate,
 * misses on every head and is exact attention, and its appends refill the
 * ring from there.  Other requests are untouched. */
int oc_reset_requests(const oc_config *c, oc_ring *ring, const int32_t *flags) {
  int B = c->batch, K = c->ring_k;
  for (int b = 0; b < B; ++b)
    if (flags[b] != 0)
      for (int s = 0; s < K; ++s) ring->pos[(int64_t)b * K + s] = 0;
  return 0;
}
