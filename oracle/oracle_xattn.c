/*
 * oracle_xattn.c -- plain fp64 CPU oracle for the generalised problem of oracle_xattn.h.
 *
 * TEST INFRASTRUCTURE ONLY, like oracle.c, and independent of the CUDA library.
 *
 * Scope: the T5 encoder-decoder architecture the FAT5 report keeps ("Motivation" section). Its
 * decoder attends over the encoder's output (cross-attention: Lq != Lk, no positional bias in
 * T5), and its decoder self-attention at inference runs over a key cache longer than the new
 * queries. Grouped-query heads let several query heads share one key/value head.
 *
 * Definitions (per document with Lq queries and Lk keys, query head h, key/value head
 * g(h) = h / (Hq / Hkv)); the pages print no formulas, so each reading is stated here:
 *   - Positions: query p sits at key position a(p) = p + (Lk - Lq), i.e. the last query lines up
 *     with the last key (bottom-right alignment). For Lq = Lk this is the self-attention case.
 *   - Relative position delta = r - a(p) (key minus query), as in oracle.c.
 *   - S'[p, r] = scale * q_p . k_r + B[p, r], B from the T5 table column h and/or the ALiBi slope
 *     of h at that delta (the same scalar functions as oracle.c).
 *   - Causal: S'[p, r] = -inf for r > a(p). A query row with no allowed key (a(p) < 0) has
 *     out = 0, lse = -inf and contributes no gradient.
 *   - P = softmax(S') per row, out = P V; the backward of sum(out * dout) is the usual calculus,
 *     with dK and dV of a key/value head summed over the query heads that read it.
 * All arithmetic is fp64, one row at a time.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"
#include "oracle_xattn.h"

static int xcheck(const oracle_xproblem_t *pb) {
  if (!pb || !pb->q || !pb->k || !pb->v || !pb->cu_seqlens_q || !pb->cu_seqlens_k) return -1;
  if (pb->num_heads_q <= 0 || pb->num_heads_kv <= 0 || pb->head_dim <= 0 || pb->num_seqs < 0)
    return -2;
  if (pb->num_heads_q % pb->num_heads_kv) return -2;
  if (pb->cu_seqlens_q[0] != 0 || pb->cu_seqlens_q[pb->num_seqs] != pb->total_q) return -2;
  if (pb->cu_seqlens_k[0] != 0 || pb->cu_seqlens_k[pb->num_seqs] != pb->total_k) return -2;
  for (int i = 0; i < pb->num_seqs; ++i)
    if (pb->cu_seqlens_q[i + 1] < pb->cu_seqlens_q[i] ||
        pb->cu_seqlens_k[i + 1] < pb->cu_seqlens_k[i])
      return -2;
  if (pb->bias_table) {
    int nbh = pb->bidirectional ? pb->num_buckets / 2 : pb->num_buckets;
    if (pb->bidirectional && (pb->num_buckets % 2)) return -3;
    if (nbh < 2 || nbh > 128) return -3;
    if (pb->max_distance <= nbh / 2) return -3;
  }
  return 0;
}

/* geometry of one document */
typedef struct {
  int sq, lq, sk, lk, shift; /* shift = Lk - Lq: query p sits at key position p + shift */
} xdoc_t;

static xdoc_t xdoc(const oracle_xproblem_t *pb, int i) {
  xdoc_t g;
  g.sq = pb->cu_seqlens_q[i];
  g.lq = pb->cu_seqlens_q[i + 1] - g.sq;
  g.sk = pb->cu_seqlens_k[i];
  g.lk = pb->cu_seqlens_k[i + 1] - g.sk;
  g.shift = g.lk - g.lq;
  return g;
}

static double xdot(const double *a, const double *b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

/* row p of S' (masked entries -inf) for query head h; *bucket_row receives the bucket of each
   key when a table is given */
static void xlogits_row(const oracle_xproblem_t *pb, const xdoc_t *g, int h, int p, double *row,
                        int *bucket_row) {
  const int Hq = pb->num_heads_q, Hkv = pb->num_heads_kv, d = pb->head_dim;
  const int hk = h / (Hq / Hkv);
  const double *qp = pb->q + ((size_t)(g->sq + p) * Hq + h) * d;
  const long long a = (long long)p + g->shift;
  for (int r = 0; r < g->lk; ++r) {
    const long long delta = (long long)r - a;
    if (bucket_row)
      bucket_row[r] = pb->bias_table ? oracle_t5_bucket(delta, pb->num_buckets, pb->max_distance,
                                                        pb->bidirectional)
                                     : -1;
    if (pb->causal && delta > 0) {
      row[r] = -INFINITY;
      continue;
    }
    const double *kr = pb->k + ((size_t)(g->sk + r) * Hkv + hk) * d;
    double s = pb->softmax_scale * xdot(qp, kr, d);
    if (pb->bias_table) s += pb->bias_table[(size_t)bucket_row[r] * Hq + h];
    if (pb->alibi_slopes) s += oracle_alibi_bias(delta, pb->alibi_slopes[h]);
    row[r] = s;
  }
}

/* softmax in place; returns lse (-inf and an all-zero row when nothing is allowed) */
static double xsoftmax(double *row, int n) {
  double m = -INFINITY;
  for (int r = 0; r < n; ++r)
    if (row[r] > m) m = row[r];
  if (m == -INFINITY) {
    for (int r = 0; r < n; ++r) row[r] = 0.0;
    return -INFINITY;
  }
  double sum = 0.0;
  for (int r = 0; r < n; ++r) sum += exp(row[r] - m);
  const double lse = m + log(sum);
  for (int r = 0; r < n; ++r) row[r] = exp(row[r] - lse);
  return lse;
}

int oracle_xattn_fwd(const oracle_xproblem_t *pb, double *out, double *lse) {
  int rc = xcheck(pb);
  if (rc) return rc;
  if (!out) return -1;
  const int Hq = pb->num_heads_q, Hkv = pb->num_heads_kv, d = pb->head_dim;
  const int n = pb->num_seqs * Hq;
#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < n; ++w) {
    const int i = w / Hq, h = w % Hq, hk = h / (Hq / Hkv);
    const xdoc_t g = xdoc(pb, i);
    double *row = (double *)malloc(sizeof(double) * (size_t)(g.lk > 0 ? g.lk : 1));
    int *bkt = (int *)malloc(sizeof(int) * (size_t)(g.lk > 0 ? g.lk : 1));
    for (int p = 0; p < g.lq; ++p) {
      xlogits_row(pb, &g, h, p, row, bkt);
      const double l = xsoftmax(row, g.lk);
      if (lse) lse[(size_t)h * pb->total_q + g.sq + p] = l;
      double *o = out + ((size_t)(g.sq + p) * Hq + h) * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int r = 0; r < g.lk; ++r) {
        if (row[r] == 0.0) continue;
        const double *vr = pb->v + ((size_t)(g.sk + r) * Hkv + hk) * d;
        for (int c = 0; c < d; ++c) o[c] += row[r] * vr[c];
      }
    }
    free(row);
    free(bkt);
  }
  return 0;
}

/* one (document, key/value head): every query head of the group, so that the dK and dV sums of
   the group stay inside one task */
static void xbwd_group(const oracle_xproblem_t *pb, const double *dout, int i, int hk, double *dq,
                       double *dk, double *dv, double *dtab /* [nb, Hq] slice owner: caller */) {
  const int Hq = pb->num_heads_q, Hkv = pb->num_heads_kv, d = pb->head_dim;
  const int grp = Hq / Hkv;
  const xdoc_t g = xdoc(pb, i);
  const int nk = g.lk > 0 ? g.lk : 1;
  double *P = (double *)malloc(sizeof(double) * (size_t)nk);
  double *dP = (double *)malloc(sizeof(double) * (size_t)nk);
  int *bkt = (int *)malloc(sizeof(int) * (size_t)nk);
  for (int h = hk * grp; h < (hk + 1) * grp; ++h) {
    for (int p = 0; p < g.lq; ++p) {
      xlogits_row(pb, &g, h, p, P, bkt);
      xsoftmax(P, g.lk);
      const double *dop = dout + ((size_t)(g.sq + p) * Hq + h) * d;
      const double *qp = pb->q + ((size_t)(g.sq + p) * Hq + h) * d;
      double D = 0.0;
      for (int r = 0; r < g.lk; ++r) {
        const double *vr = pb->v + ((size_t)(g.sk + r) * Hkv + hk) * d;
        dP[r] = xdot(dop, vr, d);
        D += P[r] * dP[r];
      }
      double *dqp = dq + ((size_t)(g.sq + p) * Hq + h) * d;
      for (int r = 0; r < g.lk; ++r) {
        if (P[r] == 0.0) continue; /* masked (or underflowed): no contribution */
        const double ds = P[r] * (dP[r] - D);
        const double *kr = pb->k + ((size_t)(g.sk + r) * Hkv + hk) * d;
        double *dkr = dk + ((size_t)(g.sk + r) * Hkv + hk) * d;
        double *dvr = dv + ((size_t)(g.sk + r) * Hkv + hk) * d;
        for (int c = 0; c < d; ++c) {
          dqp[c] += pb->softmax_scale * ds * kr[c];
          dkr[c] += pb->softmax_scale * ds * qp[c];
          dvr[c] += P[r] * dop[c];
        }
        if (dtab && pb->bias_table) dtab[(size_t)bkt[r] * Hq + h] += ds;
      }
    }
  }
  free(P);
  free(dP);
  free(bkt);
}

int oracle_xattn_bwd(const oracle_xproblem_t *pb, const double *dout, double *dq, double *dk,
                     double *dv, double *dtable) {
  int rc = xcheck(pb);
  if (rc) return rc;
  if (!dout || !dq || !dk || !dv) return -1;
  const int Hq = pb->num_heads_q, Hkv = pb->num_heads_kv, d = pb->head_dim;
  const int nb = pb->bias_table ? pb->num_buckets : 0;
  memset(dq, 0, sizeof(double) * (size_t)pb->total_q * Hq * d);
  memset(dk, 0, sizeof(double) * (size_t)pb->total_k * Hkv * d);
  memset(dv, 0, sizeof(double) * (size_t)pb->total_k * Hkv * d);
  const int n = pb->num_seqs * Hkv;
  /* one table-gradient slice per task, summed afterwards in a fixed order */
  double *parts = (dtable && nb) ? (double *)calloc((size_t)n * nb * Hq, sizeof(double)) : NULL;
#pragma omp parallel for schedule(dynamic, 1)
  for (int w = 0; w < n; ++w)
    xbwd_group(pb, dout, w / Hkv, w % Hkv, dq, dk, dv, parts ? parts + (size_t)w * nb * Hq : NULL);
  if (dtable && nb) {
    memset(dtable, 0, sizeof(double) * (size_t)nb * Hq);
    for (int w = 0; w < n; ++w)
      for (size_t e = 0; e < (size_t)nb * Hq; ++e) dtable[e] += parts[(size_t)w * nb * Hq + e];
  }
  free(parts);
  return 0;
}
