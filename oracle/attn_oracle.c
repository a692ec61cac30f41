/*
 * attn_oracle.c -- plain fp64 CPU attention oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load or call this library.  The
 * CUDA product path never links, imports or calls it, and it shares no code
 * with the CUDA kernels.
 *
 * What it computes (the plain definition of the forward pass):
 *
 *   O[b,i,h,:] = sum_j p_j V[b,j,kv,:] / sum_j p_j,
 *   p_j = exp(s_j - max_j s_j),   s_j = scale * sum_d Q[b,i,h,d] K[b,j,kv,d],
 *   kv = floor(h / G),  G = Hq / Hkv,
 *
 * over the visible keys j of row i:
 *   - prefill: j in [0, Sk), and, when causal, j <= i + (Sk - Sq)
 *     (bottom-right alignment);
 *   - decode:  j in [0, L) with L clamped to [0, cap].
 *
 * Sources:
 *   - tessera #90 "compiler-generated flash_attn fwd+bwd", flash_attn
 *     forward commit note: S = scale*Q@K^T, causal/ragged mask, softmax, O = P@V,
 *     runtime Sq/Sk/scale/causal.
 *   - "Dense flash-attention prefill (gfx950 / MI355X)", opening paragraph:
 *     forward only, MHA or GQA, causal.
 *   - rocm-libraries #13108 "minimal single-token attention decode",
 *     interface description: Sq=1 over a contiguous token-major K/V cache with
 *     a device valid length, "unmasked and bottom-right causal".
 *
 * Readings where the pages are silent:
 *   - GQA map kv = floor(h / G) (contiguous groups of query heads);
 *   - a row with no visible key outputs 0;
 *   - decode valid length clamped to [0, cap].
 *
 * Flash attention reaches this same result (up to rounding) by tiling and an
 * online softmax; the oracle does none of that: one row at a time, explicit
 * score vector, max-subtracted exponentials, one normalising division.
 * Cache entries at j >= L are never read, so NaN contents there cannot reach
 * the result.
 *
 * Optional second output, the natural log of the softmax denominator of each
 * row (its log-sum-exp over the visible keys),
 *   lse[b,h,i] = log sum_j exp(s_j) = max_j s_j + log sum_j exp(s_j - max),
 * and -inf for a row that sees no key.  It is the per-row statistic a
 * backward pass recomputes P from (tessera #90, flash-attention backward
 * commit note: the "_pre" kernel's logsumexp L) and the one a split or
 * sequence-parallel combine merges by; rocm-libraries #13108 lists the LSE
 * output among the pieces its first decode milestone leaves out.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* One query row against n_vis visible keys.
 *   q      : D doubles (the query row)
 *   kbase  : K[b, 0, kv, 0]; key j is at kbase + j*kstride
 *   vbase  : V[b, 0, kv, 0]; value j is at vbase + j*kstride
 *   o      : D doubles out
 *   p_out  : optional, n_vis probabilities out (normalised)
 *   lse    : optional, the row's log-sum-exp out
 *   s      : scratch, n_vis doubles
 */
static void attend_row(const double* q, const double* kbase, const double* vbase,
                       int64_t kstride, int64_t n_vis, int D, double scale,
                       double* o, double* p_out, double* lse, double* s) {
  int d;
  int64_t j;
  for (d = 0; d < D; ++d) o[d] = 0.0;
  if (lse) *lse = -INFINITY;
  if (n_vis <= 0) return; /* no visible key: output 0, log-sum-exp -inf */

  /* scores s_j = scale * <q, k_j> */
  double m = -INFINITY;
  for (j = 0; j < n_vis; ++j) {
    const double* kj = kbase + j * kstride;
    double acc = 0.0;
    for (d = 0; d < D; ++d) acc += q[d] * kj[d];
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  /* p_j = exp(s_j - m), l = sum p_j */
  double l = 0.0;
  for (j = 0; j < n_vis; ++j) {
    s[j] = exp(s[j] - m);
    l += s[j];
  }
  /* O = sum_j p_j v_j / l */
  for (j = 0; j < n_vis; ++j) {
    const double* vj = vbase + j * kstride;
    double pj = s[j];
    for (d = 0; d < D; ++d) o[d] += pj * vj[d];
  }
  for (d = 0; d < D; ++d) o[d] /= l;
  if (lse) *lse = m + log(l);
  if (p_out)
    for (j = 0; j < n_vis; ++j) p_out[j] = s[j] / l;
}

/* Number of keys that query row i may see. */
static int64_t visible_keys(int64_t i, int64_t Sq, int64_t Sk, int causal) {
  if (!causal) return Sk;
  int64_t last = i + (Sk - Sq); /* largest visible key index */
  if (last < 0) return 0;
  return last + 1 < Sk ? last + 1 : Sk;
}

typedef struct {
  const double* q_rows; /* [nrows, D] */
  const double* k;      /* [B, Sk, Hkv, D] */
  const double* v;      /* [B, Sk, Hkv, D] */
  double* o_rows;       /* [nrows, D] */
  double* lse_rows;     /* [nrows] or NULL */
  const int64_t* rows;  /* [nrows, 3] = (b, h, i) */
  int64_t nrows;
  int B, Hq, Hkv, D, causal;
  int64_t Sq, Sk;
  double scale;
  int64_t r0, r1; /* this worker's row range */
  int status;
} rows_job_t;

static void* rows_worker(void* arg) {
  rows_job_t* J = (rows_job_t*)arg;
  double* s = (double*)malloc(sizeof(double) * (size_t)(J->Sk > 0 ? J->Sk : 1));
  if (!s) { J->status = 1; return NULL; }
  const int G = J->Hq / J->Hkv;
  const int64_t kstride = (int64_t)J->Hkv * J->D;
  int64_t r;
  for (r = J->r0; r < J->r1; ++r) {
    const int64_t b = J->rows[3 * r + 0];
    const int64_t h = J->rows[3 * r + 1];
    const int64_t i = J->rows[3 * r + 2];
    const int64_t kv = h / G;
    const double* kb = J->k + (b * J->Sk * J->Hkv + kv) * J->D;
    const double* vb = J->v + (b * J->Sk * J->Hkv + kv) * J->D;
    attend_row(J->q_rows + r * J->D, kb, vb, kstride,
               visible_keys(i, J->Sq, J->Sk, J->causal), J->D, J->scale,
               J->o_rows + r * J->D, NULL, J->lse_rows ? J->lse_rows + r : NULL, s);
  }
  free(s);
  J->status = 0;
  return NULL;
}

/* Attention for an explicit list of query rows; lse_rows (nrows doubles) may
 * be NULL.  Returns 0 on success, nonzero on bad arguments or allocation
 * failure. */
int oracle_attention_rows_lse(const double* q_rows, const double* k, const double* v,
                              double* o_rows, double* lse_rows, const int64_t* rows,
                              int64_t nrows, int B, int Hq, int Hkv, int64_t Sq, int64_t Sk,
                              int D, double scale, int causal, int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || Sq < 0 || Sk < 0)
    return 2;
  int64_t r;
  for (r = 0; r < nrows; ++r) {
    if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 ||
        rows[3 * r + 1] >= Hq || rows[3 * r + 2] < 0 || rows[3 * r + 2] >= Sq)
      return 3;
  }
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nrows) nthreads = (int)(nrows > 0 ? nrows : 1);
  rows_job_t* jobs = (rows_job_t*)calloc((size_t)nthreads, sizeof(rows_job_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) { free(jobs); free(th); return 1; }
  int t, rc = 0;
  for (t = 0; t < nthreads; ++t) {
    rows_job_t* J = &jobs[t];
    J->q_rows = q_rows; J->k = k; J->v = v; J->o_rows = o_rows; J->rows = rows;
    J->lse_rows = lse_rows;
    J->nrows = nrows; J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->D = D;
    J->causal = causal; J->Sq = Sq; J->Sk = Sk; J->scale = scale;
    J->r0 = nrows * t / nthreads;
    J->r1 = nrows * (t + 1) / nthreads;
    J->status = 1;
  }
  if (nthreads == 1) {
    rows_worker(&jobs[0]);
  } else {
    for (t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, rows_worker, &jobs[t]);
    for (t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  }
  for (t = 0; t < nthreads; ++t) rc |= jobs[t].status;
  free(jobs);
  free(th);
  return rc;
}

int oracle_attention_rows(const double* q_rows, const double* k, const double* v,
                          double* o_rows, const int64_t* rows, int64_t nrows,
                          int B, int Hq, int Hkv, int64_t Sq, int64_t Sk, int D,
                          double scale, int causal, int nthreads) {
  return oracle_attention_rows_lse(q_rows, k, v, o_rows, NULL, rows, nrows, B, Hq, Hkv, Sq, Sk,
                                   D, scale, causal, nthreads);
}

/* Softmax probabilities of one query row over all Sk keys (masked keys get 0).
 * Exposed so that tests can check that every row sums to one. */
int oracle_attention_probs(const double* q_row, const double* k, const double* v,
                           double* p_out, double* o_out, int b, int h, int64_t i,
                           int B, int Hq, int Hkv, int64_t Sq, int64_t Sk, int D,
                           double scale, int causal) {
  if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Sq || Hkv <= 0 ||
      Hq % Hkv != 0)
    return 2;
  const int G = Hq / Hkv;
  const int64_t kv = h / G;
  const int64_t n_vis = visible_keys(i, Sq, Sk, causal);
  double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
  if (!s) return 1;
  int64_t j;
  for (j = 0; j < Sk; ++j) p_out[j] = 0.0;
  const double* kb = k + ((int64_t)b * Sk * Hkv + kv) * D;
  const double* vb = v + ((int64_t)b * Sk * Hkv + kv) * D;
  attend_row(q_row, kb, vb, (int64_t)Hkv * D, n_vis, D, scale, o_out, p_out, NULL, s);
  free(s);
  return 0;
}

/* Single-token decode: q [B, Hq, D], caches [B, cap, Hkv, D], valid length L
 * shared by the batch and clamped to [0, cap]; o [B, Hq, D]; lse [B, Hq] or
 * NULL. */
int oracle_decode_lse(const double* q, const double* kcache, const double* vcache,
                      double* o, double* lse, int B, int Hq, int Hkv, int64_t cap, int D,
                      int64_t L, double scale) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || cap < 0) return 2;
  if (L < 0) L = 0;
  if (L > cap) L = cap;
  const int G = Hq / Hkv;
  double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  if (!s) return 1;
  int b, h;
  for (b = 0; b < B; ++b) {
    for (h = 0; h < Hq; ++h) {
      const int64_t kv = h / G;
      const double* kb = kcache + ((int64_t)b * cap * Hkv + kv) * D;
      const double* vb = vcache + ((int64_t)b * cap * Hkv + kv) * D;
      attend_row(q + ((int64_t)b * Hq + h) * D, kb, vb, (int64_t)Hkv * D, L, D,
                 scale, o + ((int64_t)b * Hq + h) * D, NULL,
                 lse ? lse + (int64_t)b * Hq + h : NULL, s);
    }
  }
  free(s);
  return 0;
}

int oracle_decode(const double* q, const double* kcache, const double* vcache,
                  double* o, int B, int Hq, int Hkv, int64_t cap, int D,
                  int64_t L, double scale) {
  return oracle_decode_lse(q, kcache, vcache, o, NULL, B, Hq, Hkv, cap, D, L, scale);
}

/*
 * Backward pass: gradients of the loss l = sum_{b,i,h,d} O[b,i,h,d] dO[b,i,h,d]
 * with respect to Q, K and V (tessera #90, flash-attention backward commit
 * note: the "_pre" pass forms Delta_i = sum_d dO_id O_id, then dV += P^T dO,
 * dP = dO V^T, dS = P * (dP - Delta), dK += scale * dS^T Q, dQ += scale * dS K).
 * Written out from the definition of the forward pass, row by row:
 *   p_j    = exp(s_j - m) / sum_k exp(s_k - m)   over the row's visible keys
 *   dV_j  += p_j dO
 *   dp_j   = <dO, V_j>
 *   Delta  = sum_j p_j dp_j                      (= <dO, O>)
 *   ds_j   = p_j (dp_j - Delta)
 *   dQ     = scale * sum_j ds_j K_j
 *   dK_j  += scale * ds_j Q
 * Query heads of a GQA group add into the same dK, dV.  One worker per
 * (b, kv head) owns that head's dK/dV rows, so no two threads add to the same
 * element.
 */
typedef struct {
  const double *q, *k, *v, *dout;
  double *dq, *dk, *dv;
  int B, Hq, Hkv, D, causal;
  int64_t Sq, Sk;
  double scale;
  int64_t u0, u1; /* (b, kv head) units of this worker */
  int status;
} bwd_job_t;

static void* bwd_worker(void* arg) {
  bwd_job_t* J = (bwd_job_t*)arg;
  const int G = J->Hq / J->Hkv, D = J->D;
  double* pr = (double*)malloc(sizeof(double) * (size_t)(J->Sk > 0 ? J->Sk : 1));
  double* dp = (double*)malloc(sizeof(double) * (size_t)(J->Sk > 0 ? J->Sk : 1));
  if (!pr || !dp) { free(pr); free(dp); J->status = 1; return NULL; }
  const int64_t kstride = (int64_t)J->Hkv * D;
  int64_t u, i, j;
  int g, d;
  for (u = J->u0; u < J->u1; ++u) {
    const int64_t b = u / J->Hkv, kv = u % J->Hkv;
    const double* kb = J->k + (b * J->Sk * J->Hkv + kv) * D;
    const double* vb = J->v + (b * J->Sk * J->Hkv + kv) * D;
    double* dkb = J->dk + (b * J->Sk * J->Hkv + kv) * D;
    double* dvb = J->dv + (b * J->Sk * J->Hkv + kv) * D;
    for (g = 0; g < G; ++g) {
      const int64_t h = kv * G + g;
      for (i = 0; i < J->Sq; ++i) {
        const double* qi = J->q + ((b * J->Sq + i) * J->Hq + h) * D;
        const double* doi = J->dout + ((b * J->Sq + i) * J->Hq + h) * D;
        double* dqi = J->dq + ((b * J->Sq + i) * J->Hq + h) * D;
        for (d = 0; d < D; ++d) dqi[d] = 0.0;
        const int64_t n_vis = visible_keys(i, J->Sq, J->Sk, J->causal);
        if (n_vis <= 0) continue;
        /* the row's probabilities pr_j, as in the forward pass */
        double mx = -INFINITY;
        for (j = 0; j < n_vis; ++j) {
          double dot = 0.0;
          for (d = 0; d < D; ++d) dot += qi[d] * kb[j * kstride + d];
          pr[j] = J->scale * dot;
          mx = pr[j] > mx ? pr[j] : mx;
        }
        double den = 0.0;
        for (j = 0; j < n_vis; ++j) {
          pr[j] = exp(pr[j] - mx);
          den += pr[j];
        }
        double delta = 0.0;
        for (j = 0; j < n_vis; ++j) {
          pr[j] /= den;
          double dot = 0.0;
          for (d = 0; d < D; ++d) dot += doi[d] * vb[j * kstride + d];
          dp[j] = dot;
          delta += pr[j] * dp[j];
        }
        for (j = 0; j < n_vis; ++j) {
          const double ds = pr[j] * (dp[j] - delta);
          for (d = 0; d < D; ++d) {
            dvb[j * kstride + d] += pr[j] * doi[d];
            dqi[d] += J->scale * ds * kb[j * kstride + d];
            dkb[j * kstride + d] += J->scale * ds * qi[d];
          }
        }
      }
    }
  }
  free(pr);
  free(dp);
  J->status = 0;
  return NULL;
}

/* dQ [B, Sq, Hq, D], dK / dV [B, Sk, Hkv, D] (overwritten) for the loss
 * sum(O * dO).  Returns 0 on success. */
int oracle_attention_bwd(const double* q, const double* k, const double* v,
                         const double* dout, double* dq, double* dk, double* dv, int B,
                         int Hq, int Hkv, int64_t Sq, int64_t Sk, int D, double scale,
                         int causal, int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || Sq < 0 || Sk < 0) return 2;
  memset(dk, 0, sizeof(double) * (size_t)B * (size_t)Sk * (size_t)Hkv * (size_t)D);
  memset(dv, 0, sizeof(double) * (size_t)B * (size_t)Sk * (size_t)Hkv * (size_t)D);
  memset(dq, 0, sizeof(double) * (size_t)B * (size_t)Sq * (size_t)Hq * (size_t)D);
  const int64_t units = (int64_t)B * Hkv;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > units) nthreads = (int)(units > 0 ? units : 1);
  bwd_job_t* jobs = (bwd_job_t*)calloc((size_t)nthreads, sizeof(bwd_job_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) { free(jobs); free(th); return 1; }
  int t, rc = 0;
  for (t = 0; t < nthreads; ++t) {
    bwd_job_t* J = &jobs[t];
    J->q = q; J->k = k; J->v = v; J->dout = dout; J->dq = dq; J->dk = dk; J->dv = dv;
    J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->D = D; J->causal = causal;
    J->Sq = Sq; J->Sk = Sk; J->scale = scale;
    J->u0 = units * t / nthreads;
    J->u1 = units * (t + 1) / nthreads;
    J->status = 1;
  }
  if (nthreads == 1) {
    bwd_worker(&jobs[0]);
  } else {
    for (t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, bwd_worker, &jobs[t]);
    for (t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  }
  for (t = 0; t < nthreads; ++t) rc |= jobs[t].status;
  free(jobs);
  free(th);
  return rc;
}
