/*
 * oracle.h -- fp64 CPU oracle for attention with an in-kernel relative-position bias.
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the benchmark's CPU-baseline
 * leg. Independent of the CUDA library (no shared code or headers).
 *
 * Layouts: q, k, v, dout are fp64 [total_tokens, num_heads, head_dim], token major. cu_seqlens is a HOST int32 array of num_seqs+1 offsets (cu[0] = 0, cu[n] = total).
 * bias_table is fp64 [num_buckets, num_heads] (T5) or NULL; alibi_slopes is fp64 [num_heads]
 * or NULL. Outputs are fp64: out/dq/dk/dv [total_tokens, num_heads, head_dim], lse
 * [num_heads, total_tokens] (natural log), dtable [num_buckets, num_heads].
 * Return codes: 0 ok, -1 null pointer, -2 bad shape / index, -3 bad bucket arguments.
 */
#ifndef ATTN_RELPOS_ORACLE_H
#define ATTN_RELPOS_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int total_tokens;
  int num_seqs;
  int num_heads;
  int head_dim;
  const int32_t *cu_seqlens;
  const double *q, *k, *v;
  const double *bias_table;
  int num_buckets, max_distance, bidirectional;
  const double *alibi_slopes;
  int causal;
  double softmax_scale;
  /* 0: D_p = sum_r P[p,r] dP[p,r] (exact calculus). 1: D_p = sum_c dO[p,c] * bf16(O[p,c]), the
     row statistic formed from the forward output as stored in bf16 (the backward's inputs are
     the bf16 output, as in FlashAttention-style backward passes). */
  int d_from_bf16_out;
} oracle_problem_t;

int oracle_t5_bucket(long long delta, int num_buckets, int max_distance, int bidirectional);
double oracle_alibi_bias(long long delta, double slope);
int oracle_attn_fwd(const oracle_problem_t *pb, double *out, double *lse);
int oracle_attn_bwd(const oracle_problem_t *pb, const double *dout, double *dq, double *dk,
                    double *dv, double *dtable);
int oracle_attn_fwd_rows(const oracle_problem_t *pb, int doc, int head, const int *rows, int nrows,
                         double *out_rows, double *lse_rows);
int oracle_attn_bwd_rows(const oracle_problem_t *pb, const double *dout, int doc, int head,
                         const int *qrows, int nq, const int *krows, int nk, double *dq_rows,
                         double *dk_rows, double *dv_rows, double *dtable_col);
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
