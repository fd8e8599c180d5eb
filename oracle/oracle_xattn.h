/*
 * oracle_xattn.h -- fp64 CPU oracle for the generalised attention problem: per document a query
 * sequence and a key/value sequence of their own lengths (cross-attention, or self-attention
 * over a longer key cache), grouped-query heads, and causal masking aligned at the bottom right.
 * TEST INFRASTRUCTURE ONLY (same callers as oracle.h). Not yet matched by a CUDA path.
 *
 * Layouts: q and dout fp64 [total_q, num_heads_q, head_dim]; k and v fp64
 * [total_k, num_heads_kv, head_dim]; cu_seqlens_q / cu_seqlens_k HOST int32 [num_seqs + 1].
 * Query head h reads key/value head h / (num_heads_q / num_heads_kv). bias_table fp64
 * [num_buckets, num_heads_q] or NULL; alibi_slopes fp64 [num_heads_q] or NULL.
 * Outputs fp64: out/dq like q, dk/dv like k, lse [num_heads_q, total_q] (natural log; -inf for a
 * row with no allowed key, whose out is 0), dtable [num_buckets, num_heads_q].
 * Return codes: 0 ok, -1 null pointer, -2 bad shape / index, -3 bad bucket arguments.
 */
#ifndef ATTN_RELPOS_ORACLE_XATTN_H
#define ATTN_RELPOS_ORACLE_XATTN_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int num_seqs;
  int total_q, total_k;
  int num_heads_q, num_heads_kv, head_dim;
  const int32_t *cu_seqlens_q, *cu_seqlens_k;
  const double *q, *k, *v;
  const double *bias_table;
  int num_buckets, max_distance, bidirectional;
  const double *alibi_slopes;
  int causal; /* key r is allowed for query p iff r <= p + (Lk - Lq) */
  double softmax_scale;
} oracle_xproblem_t;

int oracle_xattn_fwd(const oracle_xproblem_t *pb, double *out, double *lse);
int oracle_xattn_bwd(const oracle_xproblem_t *pb, const double *dout, double *dq, double *dk,
                     double *dv, double *dtable);

#ifdef __cplusplus
}
#endif
#endif
