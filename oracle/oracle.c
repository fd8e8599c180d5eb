/*
 * oracle.c -- plain fp64 CPU oracle for attention with an additive relative-position bias.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls this file; only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark do. It shares no code, header,
 * table or constant with the CUDA library.
 *
 * What it computes (FAT5 report, "Noyau CUDA" section, both kernel versions): per document and head,
 *     S = Q K^T,   S' = S + B,   P = softmax(S'),   O = P V,
 * with B built from relative positions instead of being passed in. The pages print no formulas, so
 * each reading below is stated where it is used:
 *   - The softmax scale multiplies Q K^T only; the bias is added unscaled (the section lists
 *     S = Q K^T first, then S' = S + B).
 *   - T5 bias (RelativePositionalEncoding, named in the same section; T5 is the cited model):
 *     B[p, r] = table[bucket(r - p), h] with the T5 log-bucket function, evaluated exactly
 *     (real-valued floor, ties decided by integer arithmetic).
 *   - ALiBi bias (ALiBiPositionalEncoding, same section): B[p, r] = -slope_h * |r - p|.
 *   - Both may be present; they add.
 *   - Causal: S'[p, r] = -inf for r > p. Positions restart at 0 in every document of a packed
 *     batch (padding-free packing page: examples concatenated with per-example boundaries).
 *   - Backward: the loss is sum(out * dout); the gradients are the standard softmax-attention
 *     calculus (the pages only benchmark the backward and give no derivation). The row statistic
 *     D = sum_r P dP is either exact, or (on request) formed from the output rounded to bf16,
 *     which is what a backward pass that receives the stored bf16 output computes.
 * All arithmetic is fp64. Inputs arrive as fp64 arrays; the Python wrapper widens the exact bf16
 * and fp32 values the GPU path receives, so both sides start from identical numbers.
 *
 * The bias matrix is built element by element from its definition (the "first version" of the
 * kernel in the report passes the full bias matrix); rows are processed one at a time so that
 * long documents fit in memory. Bucket ids are cached per distinct distance within a document.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#include "oracle.h"

/* ------------------------------------------------------------------------------------------ */
/* small unsigned big integers, base 10^9 (used only to settle near-ties of the bucket floor)   */
/* ------------------------------------------------------------------------------------------ */
#define ORACLE_BIG_DIGITS 400 /* 3600 decimal digits: enough for n^E with n < 2^31, E <= 128 */
typedef struct {
  int len;
  uint32_t d[ORACLE_BIG_DIGITS];
} big_t;

static void big_set(big_t *a, uint32_t v) {
  a->len = 0;
  while (v) {
    a->d[a->len++] = v % 1000000000u;
    v /= 1000000000u;
  }
}

static int big_mul_small(big_t *a, uint32_t m) {
  uint64_t carry = 0;
  for (int i = 0; i < a->len; ++i) {
    uint64_t cur = (uint64_t)a->d[i] * m + carry;
    a->d[i] = (uint32_t)(cur % 1000000000u);
    carry = cur / 1000000000u;
  }
  while (carry) {
    if (a->len >= ORACLE_BIG_DIGITS) return -1;
    a->d[a->len++] = (uint32_t)(carry % 1000000000u);
    carry /= 1000000000u;
  }
  return 0;
}

static int big_cmp(const big_t *a, const big_t *b) {
  if (a->len != b->len) return a->len < b->len ? -1 : 1;
  for (int i = a->len - 1; i >= 0; --i)
    if (a->d[i] != b->d[i]) return a->d[i] < b->d[i] ? -1 : 1;
  return 0;
}

/* Is n^E * me^t >= md^t * me^E ?  (equivalently  E*ln(n/me) >= t*ln(md/me)) */
static int exact_at_least(int64_t n, int me, int md, int E, int t) {
  big_t lhs, rhs;
  big_set(&lhs, 1);
  big_set(&rhs, 1);
  for (int i = 0; i < E; ++i) big_mul_small(&lhs, (uint32_t)n);
  for (int i = 0; i < t; ++i) big_mul_small(&lhs, (uint32_t)me);
  for (int i = 0; i < t; ++i) big_mul_small(&rhs, (uint32_t)md);
  for (int i = 0; i < E; ++i) big_mul_small(&rhs, (uint32_t)me);
  return big_cmp(&lhs, &rhs) >= 0;
}

/* ------------------------------------------------------------------------------------------ */
/* T5 relative-position bucket (the T5 paper's scheme; the report cites T5 and names the class) */
/* ------------------------------------------------------------------------------------------ */
int oracle_t5_bucket(long long delta, int num_buckets, int max_distance, int bidirectional) {
  /* delta = key position - query position */
  int nbh = num_buckets;
  int offset = 0;
  long long n;
  if (bidirectional) {
    nbh = num_buckets / 2;
    if (delta > 0) offset = nbh;
    n = delta < 0 ? -delta : delta;
  } else {
    n = delta < 0 ? -delta : 0;
  }
  int me = nbh / 2;     /* distances below this each get their own bucket */
  int E = nbh - me;     /* number of logarithmic buckets */
  if (n < me) return offset + (int)n;
  /* t = floor( ln(n/me) / ln(md/me) * E ), capped at E-1 so that the bucket stays below nbh */
  double x = log((double)n / (double)me) / log((double)max_distance / (double)me) * (double)E;
  long long t;
  if (x >= (double)E) {
    t = E - 1;
  } else {
    t = (long long)floor(x);
    /* fp64 is far more precise than the distance to the next integer unless x is (nearly)
       an integer; there, decide the floor exactly */
    double frac = x - floor(x);
    if (frac < 1e-9 || frac > 1.0 - 1e-9) {
      long long guess = (long long)floor(x + 0.5);
      if (guess > E) guess = E;
      /* largest t' in {guess-1, guess} that satisfies the exact inequality */
      if (guess >= 0 && exact_at_least(n, me, max_distance, E, (int)guess))
        t = guess;
      else
        t = guess - 1;
    }
    if (t > E - 1) t = E - 1;
    if (t < 0) t = 0;
  }
  return offset + me + (int)t;
}

double oracle_alibi_bias(long long delta, double slope) {
  long long a = delta < 0 ? -delta : delta;
  return -slope * (double)a;
}

/* ------------------------------------------------------------------------------------------ */
/* argument checks (same conventions as the library: bidirectional T5 needs an even count)      */
/* ------------------------------------------------------------------------------------------ */
static int check_args(const oracle_problem_t *pb) {
  if (!pb || !pb->q || !pb->k || !pb->v || !pb->cu_seqlens) return -1;
  if (pb->num_heads <= 0 || pb->head_dim <= 0 || pb->num_seqs < 0 || pb->total_tokens < 0) return -2;
  if (pb->cu_seqlens[0] != 0 || pb->cu_seqlens[pb->num_seqs] != pb->total_tokens) return -2;
  for (int i = 0; i < pb->num_seqs; ++i)
    if (pb->cu_seqlens[i + 1] < pb->cu_seqlens[i]) return -2;
  if (pb->bias_table) {
    int nbh = pb->bidirectional ? pb->num_buckets / 2 : pb->num_buckets;
    if (pb->bidirectional && (pb->num_buckets % 2)) return -3;
    if (nbh < 2 || nbh > 128) return -3;
    if (pb->max_distance <= nbh / 2) return -3;
  }
  return 0;
}

/* bias of one (query, key) pair for head h, from the definitions above */
static double pair_bias(const oracle_problem_t *pb, const int *bucket_of_delta, int L, int h,
                        int p, int r) {
  double b = 0.0;
  long long delta = (long long)r - (long long)p;
  if (pb->bias_table) {
    int bk = bucket_of_delta[delta + (L - 1)];
    b += pb->bias_table[(size_t)bk * pb->num_heads + h];
  }
  if (pb->alibi_slopes) b += oracle_alibi_bias(delta, pb->alibi_slopes[h]);
  return b;
}

static int *bucket_cache(const oracle_problem_t *pb, int L) {
  if (!pb->bias_table || L <= 0) return NULL;
  int *c = (int *)malloc(sizeof(int) * (size_t)(2 * L - 1));
  for (int dd = -(L - 1); dd <= L - 1; ++dd)
    c[dd + L - 1] = oracle_t5_bucket(dd, pb->num_buckets, pb->max_distance, pb->bidirectional);
  return c;
}

/* round to bf16, nearest-even, via fp32 (NaN/Inf not expected here) */
static double round_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  u &= 0xFFFF0000u;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* D of one row: either the exact sum_r P dP, or from the bf16-rounded output row */
static double row_D(const oracle_problem_t *pb, const double *P, const double *dP,
                    const double *dop, int s, int L, int h) {
  double D = 0.0;
  if (!pb->d_from_bf16_out) {
    for (int r = 0; r < L; ++r) D += P[r] * dP[r];
    return D;
  }
  const int H = pb->num_heads, d = pb->head_dim;
  for (int c = 0; c < d; ++c) {
    double o = 0.0;
    for (int r = 0; r < L; ++r)
      if (P[r] != 0.0) o += P[r] * pb->v[((size_t)(s + r) * H + h) * d + c];
    D += dop[c] * round_bf16(o);
  }
  return D;
}

static double dotd(const double *a, const double *b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

/* row p of S' for (doc starting at token s, length L, head h); masked entries are -inf */
static void logits_row(const oracle_problem_t *pb, const int *bk, int s, int L, int h, int p,
                       double *row) {
  const int H = pb->num_heads, d = pb->head_dim;
  const double *qp = pb->q + ((size_t)(s + p) * H + h) * d;
  for (int r = 0; r < L; ++r) {
    if (pb->causal && r > p) {
      row[r] = -INFINITY;
      continue;
    }
    const double *kr = pb->k + ((size_t)(s + r) * H + h) * d;
    row[r] = pb->softmax_scale * dotd(qp, kr, d) + pair_bias(pb, bk, L, h, p, r);
  }
}

/* softmax of one row in place: returns lse, leaves P in row */
static double softmax_row(double *row, int L) {
  double m = -INFINITY;
  for (int r = 0; r < L; ++r)
    if (row[r] > m) m = row[r];
  if (m == -INFINITY) { /* fully masked row (cannot happen for causal self-attention) */
    for (int r = 0; r < L; ++r) row[r] = 0.0;
    return -INFINITY;
  }
  double sum = 0.0;
  for (int r = 0; r < L; ++r) sum += exp(row[r] - m);
  double lse = m + log(sum);
  for (int r = 0; r < L; ++r) row[r] = exp(row[r] - lse);
  return lse;
}

/* ------------------------------------------------------------------------------------------ */
/* forward                                                                                      */
/* ------------------------------------------------------------------------------------------ */
int oracle_attn_fwd(const oracle_problem_t *pb, double *out, double *lse) {
  int rc = check_args(pb);
  if (rc) return rc;
  const int H = pb->num_heads, d = pb->head_dim, T = pb->total_tokens;
  const int npairs = pb->num_seqs * H;
#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < npairs; ++w) {
    int i = w / H, h = w % H;
    int s = pb->cu_seqlens[i], L = pb->cu_seqlens[i + 1] - s;
    if (L <= 0) continue;
    int *bk = bucket_cache(pb, L);
    double *row = (double *)malloc(sizeof(double) * (size_t)L);
    for (int p = 0; p < L; ++p) {
      logits_row(pb, bk, s, L, h, p, row);
      double l = softmax_row(row, L);
      if (lse) lse[(size_t)h * T + s + p] = l;
      double *o = out + ((size_t)(s + p) * H + h) * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int r = 0; r < L; ++r) {
        if (row[r] == 0.0) continue;
        const double *vr = pb->v + ((size_t)(s + r) * H + h) * d;
        for (int c = 0; c < d; ++c) o[c] += row[r] * (vr[c]);
      }
    }
    free(row);
    free(bk);
  }
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* backward: loss = sum(out * dout)                                                             */
/*   dV = P^T dO;  dP = dO V^T;  D_p = sum_r P dP;  dS = P (dP - D);                            */
/*   dQ = scale dS K;  dK = scale dS^T Q;  dtable[bucket(r-p), h] += dS[p, r]                   */
/* ------------------------------------------------------------------------------------------ */
static void bwd_pair(const oracle_problem_t *pb, const double *dout, int s, int L, int h,
                     double *dq, double *dk, double *dv, double *dtab_col /* [nb] or NULL */) {
  const int H = pb->num_heads, d = pb->head_dim;
  int *bk = bucket_cache(pb, L);
  double *P = (double *)malloc(sizeof(double) * (size_t)L);
  double *dP = (double *)malloc(sizeof(double) * (size_t)L);
  for (int p = 0; p < L; ++p) {
    logits_row(pb, bk, s, L, h, p, P);
    softmax_row(P, L);
    const double *dop = dout + ((size_t)(s + p) * H + h) * d;
    for (int r = 0; r < L; ++r) {
      const double *vr = pb->v + ((size_t)(s + r) * H + h) * d;
      dP[r] = dotd(dop, vr, d);
    }
    const double D = row_D(pb, P, dP, dop, s, L, h);
    const double *qp = pb->q + ((size_t)(s + p) * H + h) * d;
    double *dqp = dq ? dq + ((size_t)(s + p) * H + h) * d : NULL;
    for (int r = 0; r < L; ++r) {
      double ds = P[r] * (dP[r] - D);
      const double *kr = pb->k + ((size_t)(s + r) * H + h) * d;
      if (dqp)
        for (int c = 0; c < d; ++c) dqp[c] += pb->softmax_scale * ds * (kr[c]);
      if (dk) {
        double *dkr = dk + ((size_t)(s + r) * H + h) * d;
        for (int c = 0; c < d; ++c) dkr[c] += pb->softmax_scale * ds * (qp[c]);
      }
      if (dv && P[r] != 0.0) {
        double *dvr = dv + ((size_t)(s + r) * H + h) * d;
        for (int c = 0; c < d; ++c) dvr[c] += P[r] * (dop[c]);
      }
      if (dtab_col && bk) dtab_col[bk[r - p + L - 1]] += ds;
    }
  }
  free(P);
  free(dP);
  free(bk);
}

int oracle_attn_bwd(const oracle_problem_t *pb, const double *dout, double *dq, double *dk,
                    double *dv, double *dtable) {
  int rc = check_args(pb);
  if (rc) return rc;
  if (!dout) return -1;
  const int H = pb->num_heads, d = pb->head_dim, T = pb->total_tokens;
  const int nb = pb->bias_table ? pb->num_buckets : 0;
  memset(dq, 0, sizeof(double) * (size_t)T * H * d);
  memset(dk, 0, sizeof(double) * (size_t)T * H * d);
  memset(dv, 0, sizeof(double) * (size_t)T * H * d);
  const int npairs = pb->num_seqs * H;
  /* per (doc, head) bucket-gradient columns, summed afterwards in a fixed order */
  double *cols = (dtable && nb) ? (double *)calloc((size_t)npairs * nb, sizeof(double)) : NULL;
#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < npairs; ++w) {
    int i = w / H, h = w % H;
    int s = pb->cu_seqlens[i], L = pb->cu_seqlens[i + 1] - s;
    if (L <= 0) continue;
    bwd_pair(pb, dout, s, L, h, dq, dk, dv, cols ? cols + (size_t)w * nb : NULL);
  }
  if (dtable && nb) {
    memset(dtable, 0, sizeof(double) * (size_t)nb * H);
    for (int w = 0; w < npairs; ++w) {
      int h = w % H;
      for (int b = 0; b < nb; ++b) dtable[(size_t)b * H + h] += cols[(size_t)w * nb + b];
    }
  }
  free(cols);
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* sampled rows of one (doc, head): the same definitions, restricted to the requested rows      */
/* ------------------------------------------------------------------------------------------ */
int oracle_attn_fwd_rows(const oracle_problem_t *pb, int doc, int head, const int *rows, int nrows,
                         double *out_rows, double *lse_rows) {
  int rc = check_args(pb);
  if (rc) return rc;
  if (doc < 0 || doc >= pb->num_seqs || head < 0 || head >= pb->num_heads) return -2;
  const int H = pb->num_heads, d = pb->head_dim;
  int s = pb->cu_seqlens[doc], L = pb->cu_seqlens[doc + 1] - s;
  for (int j = 0; j < nrows; ++j)
    if (rows[j] < 0 || rows[j] >= L) return -2;
  int *bk = bucket_cache(pb, L);
#pragma omp parallel for schedule(dynamic, 1)
  for (int j = 0; j < nrows; ++j) {
    int p = rows[j];
    double *row = (double *)malloc(sizeof(double) * (size_t)L);
    logits_row(pb, bk, s, L, head, p, row);
    double l = softmax_row(row, L);
    if (lse_rows) lse_rows[j] = l;
    double *o = out_rows + (size_t)j * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int r = 0; r < L; ++r) {
      if (row[r] == 0.0) continue;
      const double *vr = pb->v + ((size_t)(s + r) * H + head) * d;
      for (int c = 0; c < d; ++c) o[c] += row[r] * (vr[c]);
    }
    free(row);
  }
  free(bk);
  return 0;
}

/*
 * Gradients for sampled rows of one (doc, head): dq for query rows qrows, dk and dv for key rows
 * krows, and (optionally) this (doc, head)'s full contribution to the bucket gradient. Every
 * query row of the document enters dk, dv and the bucket gradient, so each row's softmax
 * statistics are recomputed from the definition.
 */
int oracle_attn_bwd_rows(const oracle_problem_t *pb, const double *dout, int doc, int head,
                         const int *qrows, int nq, const int *krows, int nk, double *dq_rows,
                         double *dk_rows, double *dv_rows, double *dtable_col) {
  int rc = check_args(pb);
  if (rc) return rc;
  if (!dout) return -1;
  if (doc < 0 || doc >= pb->num_seqs || head < 0 || head >= pb->num_heads) return -2;
  const int H = pb->num_heads, d = pb->head_dim;
  const int nb = pb->bias_table ? pb->num_buckets : 0;
  int s = pb->cu_seqlens[doc], L = pb->cu_seqlens[doc + 1] - s;
  for (int j = 0; j < nq; ++j)
    if (qrows[j] < 0 || qrows[j] >= L) return -2;
  for (int j = 0; j < nk; ++j)
    if (krows[j] < 0 || krows[j] >= L) return -2;
  int *bk = bucket_cache(pb, L);
  int *qpos = (int *)malloc(sizeof(int) * (size_t)(L > 0 ? L : 1));
  for (int p = 0; p < L; ++p) qpos[p] = -1;
  for (int j = 0; j < nq; ++j) qpos[qrows[j]] = j;
  if (dq_rows) memset(dq_rows, 0, sizeof(double) * (size_t)nq * d);
  if (dk_rows) memset(dk_rows, 0, sizeof(double) * (size_t)nk * d);
  if (dv_rows) memset(dv_rows, 0, sizeof(double) * (size_t)nk * d);
  if (dtable_col && nb) memset(dtable_col, 0, sizeof(double) * (size_t)nb);
  int nthreads = 1;
#ifdef _OPENMP
  nthreads = omp_get_max_threads();
#endif
  /* per-thread partial sums over query rows, added in thread order at the end */
  double *pdk = (double *)calloc((size_t)nthreads * (nk * d + 1), sizeof(double));
  double *pdv = (double *)calloc((size_t)nthreads * (nk * d + 1), sizeof(double));
  double *pdt = (double *)calloc((size_t)nthreads * (nb + 1), sizeof(double));
#pragma omp parallel
  {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    double *P = (double *)malloc(sizeof(double) * (size_t)L);
    double *dP = (double *)malloc(sizeof(double) * (size_t)L);
    double *mydk = pdk + (size_t)tid * (nk * d + 1);
    double *mydv = pdv + (size_t)tid * (nk * d + 1);
    double *mydt = pdt + (size_t)tid * (nb + 1);
#pragma omp for schedule(dynamic, 4)
    for (int p = 0; p < L; ++p) {
      logits_row(pb, bk, s, L, head, p, P);
      softmax_row(P, L);
      const double *dop = dout + ((size_t)(s + p) * H + head) * d;
      for (int r = 0; r < L; ++r)
        dP[r] = (P[r] == 0.0) ? 0.0 : dotd(dop, pb->v + ((size_t)(s + r) * H + head) * d, d);
      const double D = row_D(pb, P, dP, dop, s, L, head);
      const double *qp = pb->q + ((size_t)(s + p) * H + head) * d;
      if (qpos[p] >= 0 && dq_rows) {
        double *o = dq_rows + (size_t)qpos[p] * d;
        for (int r = 0; r < L; ++r) {
          double ds = P[r] * (dP[r] - D);
          if (ds == 0.0) continue;
          const double *kr = pb->k + ((size_t)(s + r) * H + head) * d;
          for (int c = 0; c < d; ++c) o[c] += pb->softmax_scale * ds * (kr[c]);
        }
      }
      for (int j = 0; j < nk; ++j) {
        int r = krows[j];
        double ds = P[r] * (dP[r] - D);
        for (int c = 0; c < d; ++c) {
          mydk[(size_t)j * d + c] += pb->softmax_scale * ds * (qp[c]);
          mydv[(size_t)j * d + c] += P[r] * (dop[c]);
        }
      }
      if (dtable_col && bk)
        for (int r = 0; r < L; ++r) mydt[bk[r - p + L - 1]] += P[r] * (dP[r] - D);
    }
    free(P);
    free(dP);
  }
  for (int t = 0; t < nthreads; ++t) {
    for (int x = 0; x < nk * d; ++x) {
      if (dk_rows) dk_rows[x] += pdk[(size_t)t * (nk * d + 1) + x];
      if (dv_rows) dv_rows[x] += pdv[(size_t)t * (nk * d + 1) + x];
    }
    if (dtable_col && nb)
      for (int b = 0; b < nb; ++b) dtable_col[b] += pdt[(size_t)t * (nb + 1) + b];
  }
  free(pdk);
  free(pdv);
  free(pdt);
  free(qpos);
  free(bk);
  return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
