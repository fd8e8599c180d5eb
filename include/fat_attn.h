/*
 * fat_attn.h -- C ABI of the GB300 (sm_103a) fused attention library with an in-kernel
 * relative-position bias (T5 log-bucket table and/or ALiBi), padding-free varlen packing,
 * forward and backward.
 *
 * What is computed. FAT5 report, "Noyau CUDA" section (second kernel version, "Flash Attention
 * RPE"): per document and head, S = Q K^T, S' = S + B, P = softmax(S'), O = P V, where B is not
 * passed in but built inside the kernel from the relative position of each (query, key) pair, so
 * that memory stays linear in the sequence length. Readings of points the pages leave open:
 *   - scale: S' = softmax_scale * (Q K^T) + B (the scale does not multiply the bias);
 *   - relative position: delta = key_position - query_position, positions local to each
 *     document (they restart at 0 at every cu_seqlens boundary: padding-free packing page);
 *   - T5 bias: B = bias_table[bucket(delta), head] with the T5 paper's log-bucket function
 *     (exact real floor; bidirectional: negative deltas use buckets [0, nb/2), positive ones
 *     [nb/2, nb); causal/unidirectional: only delta <= 0 is distinguished);
 *   - ALiBi bias: B = -alibi_slopes[head] * |delta|; T5 and ALiBi may be combined (they add);
 *   - causal: keys with delta > 0 are masked (top-left aligned, self-attention per document);
 *   - backward: gradients of sum(out * dout) with the standard softmax-attention calculus
 *     (the pages benchmark the backward, "Benchmark / TFLOPS" section, but give no derivation);
 *     the bias-table gradient sums dS over all (query, key) pairs that share a bucket.
 *
 * Layout (all row-major, contiguous, device memory unless stated):
 *   q, k, v, out, dout, dq, dk, dv : bf16 [total_tokens, num_heads, head_dim]
 *   lse                            : fp32 [num_heads, total_tokens], natural-log logsumexp of S'
 *   cu_seqlens                     : int32 [num_seqs + 1], cu[0] = 0, non-decreasing,
 *                                    cu[num_seqs] = total_tokens (read on the device only)
 *   bias_table, dbias_table        : fp32 [num_buckets, num_heads]
 *   alibi_slopes                   : fp32 [num_heads]
 * Every pointer must be 16-byte aligned. head_dim must be 64 or 128.
 *
 * Ownership and execution. The caller allocates every buffer, including the backward
 * workspace; no call allocates device memory. Calls are asynchronous on shape->stream (a
 * cudaStream_t; NULL = legacy default stream) and return after enqueueing. Global state: a
 * device error word per GPU (see fat_attn_get_device_error) and the scratch array of
 * fat_attn_bwd_noalloc (FAT_NOALLOC_SCRATCH_BYTES per GPU), both file-scope device variables
 * that every GPU on which the library's module is loaded holds until the process exits, whether
 * or not those calls are made; and a host-side cache of encoded TMA tensor maps, keyed by every
 * field they encode (address, sizes, tile box, element type), so that a cached map is identical
 * to a fresh one.
 *
 * Errors. Every call returns 0 on success or a negative FAT_E* code; nothing throws, exits or
 * traps. Argument errors are detected on the host before anything is enqueued. Device-side
 * problems (a pipeline wait that exceeded its time limit, a cu_seqlens entry outside
 * [0, total_tokens]) make the kernel skip the remaining work of that block and set a bit in the
 * device error word, which fat_attn_get_device_error reports.
 */
#ifndef FAT_ATTN_H
#define FAT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FAT_OK 0
#define FAT_EINVAL_NULL (-1)    /* a required pointer is NULL */
#define FAT_EINVAL_SHAPE (-2)   /* bad size, head_dim not 64/128, misaligned pointer */
#define FAT_EINVAL_BUCKETS (-3) /* bad num_buckets / max_distance / bidirectional */
#define FAT_ECUDA (-4)          /* a CUDA runtime/driver call failed (launch, tensor map, ...) */
#define FAT_EUNSUPPORTED (-5)   /* valid but unsupported combination (see each call) */
#define FAT_EDEVICE (-6)        /* the device error word was set (see below) */

/* bits of the device error word */
#define FAT_DEVERR_TIMEOUT_FWD 1 /* a forward pipeline wait exceeded its time limit */
#define FAT_DEVERR_TIMEOUT_BWD 2 /* a backward pipeline wait exceeded its time limit */
#define FAT_DEVERR_INDEX 8       /* fat_cross_entropy: a target at or beyond the vocabulary */
#define FAT_DEVERR_SEQLENS 4     /* cu_seqlens had an entry outside [0, total_tokens] or out of
                                    order, or a document longer than max_seqlen (its rows beyond
                                    the grid were not computed) */

typedef struct {
  int32_t total_tokens; /* T: sum of document lengths (rows of q, k, v) */
  int32_t num_seqs;     /* n: number of documents; cu_seqlens has n + 1 entries */
  int32_t max_seqlen;   /* upper bound on every document length (sizes the grid; must not be
                           smaller than the longest document: the host cannot check it, the
                           kernels report a longer one as FAT_DEVERR_SEQLENS) */
  int32_t num_heads;    /* H (q, k and v share the head count) */
  int32_t head_dim;     /* d: 64 or 128 */
  void *stream;         /* cudaStream_t the work is enqueued on */
} fat_shape_t;

/*
 * Forward. out = softmax(softmax_scale * Q K^T + B) V per document and head; lse = logsumexp
 * of the same logits (natural log). The bias B is the sum of the T5 term (when bias_table is
 * not NULL: num_buckets, max_distance, bidirectional describe the bucket function; bidirectional
 * needs an even num_buckets; the buckets per direction nbh must satisfy 2 <= nbh <= 128 and
 * max_distance > nbh/2) and the ALiBi term (when alibi_slopes is not NULL). Both NULL gives
 * plain attention. lse may be NULL if the caller does not need it (the backward needs it).
 * FAT_EUNSUPPORTED: the bucket layout needs a larger in-kernel lookup table than shared memory
 * holds. The table has sat_pos + sat_neg + 507 entries (sat_neg = the saturation distance of
 * fat_attn_bucket_thresholds, sat_pos = the same when bidirectional, else 0); the forward takes
 * up to 24687 entries at head_dim 64 and 8303 at head_dim 128 (32 buckets, bidirectional:
 * max_distance up to 34404 / 9436).
 */
int fat_attn_fwd(const fat_shape_t *shape, const void *q, const void *k, const void *v,
                 const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                 const float *alibi_slopes, const int32_t *cu_seqlens, int causal,
                 float softmax_scale, void *out, float *lse);

/*
 * fat_attn_fwd with a caller-owned device workspace (may be NULL). When every document has
 * length max_seqlen (total_tokens = num_seqs * max_seqlen), there is no causal mask, and the
 * forward grid (one CTA per 256 query rows x head x document, one per SM) ends in a partial
 * wave, a workspace of at least fat_attn_fwd_workspace_size(shape) bytes (256-byte aligned;
 * contents need not be initialised) lets the library split that wave's CTAs along the keys
 * and merge their partial rows in a second pass, so the last wave no longer leaves most SMs
 * idle. A smaller workspace (or NULL) gives the fat_attn_fwd schedule; results agree up to the
 * rounding of the merge. Errors as fat_attn_fwd; a misaligned workspace: FAT_EINVAL_SHAPE.
 */
int fat_attn_fwd_ws(const fat_shape_t *shape, const void *q, const void *k, const void *v,
                    const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                    const float *alibi_slopes, const int32_t *cu_seqlens, int causal,
                    float softmax_scale, void *out, float *lse, void *workspace,
                    size_t workspace_bytes);
/* Bytes fat_attn_fwd_ws uses for this shape on the current device (its SM count sets the
   waves): 0 when the shape has no split last wave. */
size_t fat_attn_fwd_workspace_size(const fat_shape_t *shape);

/* Bytes of device workspace for fat_attn_bwd at its fastest. The layout starts with an fp32 dQ
   accumulator [T, H, d] and the fp32 row statistics D = rowsum(dout * out) [H, T], each
   256-byte aligned: that prefix is the minimum every backward call accepts. Shapes whose
   documents all have length max_seqlen (total_tokens = num_seqs * max_seqlen) and whose
   one-CTA-per-key-tile backward grid ends in a partial wave (head_dim 128, or more than 8192
   keys at head_dim 64) add fp32 dK/dV rows for splitting that wave along the queries, which
   fat_attn_bwd uses without the causal mask when the workspace holds them (the dK/dV of those
   rows are then summed with fp32 atomics: order-dependent rounding). The size depends on the
   current device's SM count. */
size_t fat_attn_bwd_workspace_size(const fat_shape_t *shape);

/*
 * Backward of sum(out * dout) for the forward above (same bias, mask and scale arguments).
 * Inputs: q, k, v, out and lse from the forward, dout. Outputs dq, dk, dv (bf16) and, when
 * dbias_table is not NULL (requires bias_table), the T5 table gradient, which is OVERWRITTEN
 * (zeroed by the library, then accumulated with fp32 atomics: bit-exact bucket assignment,
 * order-dependent rounding). ALiBi slopes receive no gradient. workspace must hold
 * fat_attn_bwd_workspace_size(shape) bytes; its contents need not be initialised.
 * It enqueues the three stages below; the second and third are launched as programmatic
 * dependents of the grid before them (each is scheduled while that grid drains and waits for
 * its outputs inside the kernel), which the stage-by-stage calls do not do.
 * FAT_EUNSUPPORTED: the lookup table (entries as for the forward), with its per-delta gradient
 * sums, does not fit next to the backward's tiles: up to 3083 entries at head_dim 64 and 6951
 * at head_dim 128 (32 buckets, bidirectional: max_distance up to 2661 / 7590).
 */
int fat_attn_bwd(const fat_shape_t *shape, const void *q, const void *k, const void *v,
                 const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                 const float *alibi_slopes, const int32_t *cu_seqlens, int causal,
                 float softmax_scale, const void *out, const float *lse, const void *dout,
                 void *workspace, size_t workspace_bytes, void *dq, void *dk, void *dv,
                 float *dbias_table);

/*
 * The three stages fat_attn_bwd runs, in order, on the same stream and workspace (exposed so
 * that callers can schedule or time them separately):
 *   preprocess: D = rowsum(dout * out) (fp32, into the workspace), zero the fp32 dQ
 *               accumulator, zero dbias_table when given (num_buckets rows);
 *   main:       dK, dV (written), dQ (accumulated into the workspace) and the table gradient
 *               (accumulated into dbias_table), one CTA per (document, head, 128-key tile);
 *   finalize:   dq = bf16(softmax_scale * dQ accumulator).
 * Arguments mean what they mean for fat_attn_bwd; the same errors apply.
 */
int fat_attn_bwd_preprocess(const fat_shape_t *shape, const void *out, const void *dout,
                            void *workspace, size_t workspace_bytes, float *dbias_table,
                            int num_buckets);
int fat_attn_bwd_main(const fat_shape_t *shape, const void *q, const void *k, const void *v,
                      const float *bias_table, int num_buckets, int max_distance,
                      int bidirectional, const float *alibi_slopes, const int32_t *cu_seqlens,
                      int causal, float softmax_scale, const float *lse, const void *dout,
                      void *workspace, size_t workspace_bytes, void *dk, void *dv,
                      float *dbias_table);
int fat_attn_bwd_finalize(const fat_shape_t *shape, const void *workspace,
                          size_t workspace_bytes, float softmax_scale, void *dq);

/*
 * Backward for callers that cannot allocate device memory (no counterpart in the paper; an
 * addition of this library). Examples: an application that owns every allocation on the GPU and
 * hands libraries only fixed, caller-owned buffers, or a plug-in inside a framework whose
 * allocator must not be bypassed and which offers no way to request scratch space. Such a caller
 * cannot provide the workspace fat_attn_bwd needs, so this entry point uses a scratch array of
 * FAT_NOALLOC_SCRATCH_BYTES that the library keeps in device memory: every GPU that loads the
 * library holds it until the process exits. Otherwise it is fat_attn_bwd (same arguments minus
 * the workspace, same results, same errors); it allocates nothing and calls nothing that does.
 *   - Limit: problems whose fat_attn_bwd_workspace_size() exceeds FAT_NOALLOC_SCRATCH_BYTES are
 *     rejected with FAT_EUNSUPPORTED before any work is enqueued (fat_attn_last_error_message
 *     says why); e.g. T * H * (d + 1) * 4 bytes must fit, about 8 M elements of q at d = 64.
 *   - The first call on a device looks up the array's device address with that device current;
 *     make that first call before any stream capture. Make the device of shape->stream current
 *     for every call (as for any kernel launch); resetting a device after its first call is not
 *     supported (the looked-up address is kept for the life of the process).
 *   - Argument errors are reported exactly as fat_attn_bwd reports them, before the size test.
 *   - All calls on a device share the one array, which keeps whatever the last call left there
 *     (each call zeroes the part that must start at zero). Calls whose work overlaps on the GPU
 *     (other streams, other host threads) race on it and must be serialised by the caller.
 */
#define FAT_NOALLOC_SCRATCH_BYTES (32u << 20)
int fat_attn_bwd_noalloc(const fat_shape_t *shape, const void *q, const void *k, const void *v,
                         const float *bias_table, int num_buckets, int max_distance,
                         int bidirectional, const float *alibi_slopes, const int32_t *cu_seqlens,
                         int causal, float softmax_scale, const void *out, const float *lse,
                         const void *dout, void *dq, void *dk, void *dv, float *dbias_table);

/*
 * Cross-attention, grouped-query heads and decode (own query and key lengths per document).
 *
 * What is computed. The FAT5 report keeps T5's encoder-decoder architecture ("Motivation"
 * section): the decoder attends over the encoder's output (cross-attention, query and key
 * sequences of different lengths; T5 puts no positional bias there) and, when generating, over
 * a key/value cache longer than the new queries; the report's plans for linear-cost inference
 * ("La suite" section) rest on that decode step. The pages give no formulas for these; the
 * readings, which reduce exactly to the self-attention calls above when every document has
 * Lq = Lk and num_heads_kv = num_heads_q:
 *   - per document, query p sits at key position p + (Lk - Lq): the last query lines up with
 *     the last key (bottom-right alignment); the relative position of the bias is
 *     delta = key_position - (p + Lk - Lq), and causal masks delta > 0;
 *   - query head h reads key/value head h / (num_heads_q / num_heads_kv) (grouped-query heads);
 *     the bias table and slopes are indexed by the query head;
 *   - a query row that sees no key (causal with Lk < Lq, or Lk = 0) has out = 0, lse = -inf and
 *     contributes no gradient;
 *   - the backward sums dK, dV of a key/value head over the query heads that read it.
 * Layout: q, out, dout, dq bf16 [total_q, num_heads_q, head_dim]; k, v, dk, dv bf16
 * [total_k, num_heads_kv, head_dim]; lse fp32 [num_heads_q, total_q]; cu_seqlens_q and
 * cu_seqlens_k int32 [num_seqs + 1] (device); bias_table / dbias_table fp32
 * [num_buckets, num_heads_q]; alibi_slopes fp32 [num_heads_q]. Ownership, alignment, errors and
 * streams as above; num_heads_q must be a multiple of num_heads_kv.
 */
typedef struct {
  int32_t total_q;      /* rows of q, out, dout, dq */
  int32_t total_k;      /* rows of k, v, dk, dv */
  int32_t num_seqs;     /* documents; both cu_seqlens arrays have num_seqs + 1 entries */
  int32_t max_seqlen_q; /* bound on every document's query count (a longer one is reported as
                           FAT_DEVERR_SEQLENS) */
  int32_t max_seqlen_k; /* bound on every document's key count (likewise) */
  int32_t num_heads_q;
  int32_t num_heads_kv; /* divides num_heads_q */
  int32_t head_dim;     /* 64 or 128 */
  void *stream;         /* cudaStream_t */
} fat_xshape_t;

/* Forward of the generalised problem (arguments as fat_attn_fwd, with both cu_seqlens). */
int fat_xattn_fwd(const fat_xshape_t *shape, const void *q, const void *k, const void *v,
                  const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                  const float *alibi_slopes, const int32_t *cu_seqlens_q,
                  const int32_t *cu_seqlens_k, int causal, float softmax_scale, void *out,
                  float *lse);

/*
 * The same forward with the keys of every document split into num_splits ranges, each range
 * computed by blocks of its own, and the partial results merged by a second grid
 * (out = sum_s exp(lse_s - lse) out_s, lse = log sum_s exp(lse_s)). For decode steps and other
 * problems with few query rows and long key sequences, where whole rows alone would occupy only
 * a few SMs. num_splits in [1, 64] (1 = fat_xattn_fwd); fat_xattn_splitkv_num_splits suggests
 * one (about two blocks per SM). The workspace (256-byte aligned, contents need not be
 * initialised) holds the partial outputs: fat_xattn_splitkv_workspace_size bytes (0 for one
 * split). num_seqs * num_splits must not exceed 65535 (FAT_EUNSUPPORTED).
 */
int fat_xattn_splitkv_num_splits(const fat_xshape_t *shape);
size_t fat_xattn_splitkv_workspace_size(const fat_xshape_t *shape, int num_splits);
int fat_xattn_fwd_splitkv(const fat_xshape_t *shape, const void *q, const void *k, const void *v,
                          const float *bias_table, int num_buckets, int max_distance,
                          int bidirectional, const float *alibi_slopes,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int causal,
                          float softmax_scale, int num_splits, void *workspace,
                          size_t workspace_bytes, void *out, float *lse);

/* Backward workspace of the generalised problem: the fp32 dQ accumulator [total_q, Hq, d];
   when num_heads_kv < num_heads_q also fp32 dK and dV accumulators [total_k, Hkv, d]; then D
   [Hq, total_q]; each 256-byte aligned (the minimum a call accepts); then, as for
   fat_attn_bwd_workspace_size, the rows of a split last wave when the shape has one (own
   key/value heads; with grouped heads the split wave adds into the dK/dV accumulators). */
size_t fat_xattn_bwd_workspace_size(const fat_xshape_t *shape);

/* Backward of the generalised problem (arguments as fat_attn_bwd, with both cu_seqlens). */
int fat_xattn_bwd(const fat_xshape_t *shape, const void *q, const void *k, const void *v,
                  const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                  const float *alibi_slopes, const int32_t *cu_seqlens_q,
                  const int32_t *cu_seqlens_k, int causal, float softmax_scale, const void *out,
                  const float *lse, const void *dout, void *workspace, size_t workspace_bytes,
                  void *dq, void *dk, void *dv, float *dbias_table);

/*
 * Rotary position embedding (RoPE). The FAT5 report lists RoFormer's rotary embedding among the
 * positional encodings its attention kernels take ("Noyau CUDA" section); it prints no formula,
 * and the plainest reading is RoFormer's: channel pair (2i, 2i + 1) of a row at position m turns
 * by the angle m * base^(-2i/d) (base 10000 in RoFormer), positions local to each document
 * (restarting at every cu_seqlens boundary). Unlike the T5 and ALiBi biases it acts on Q and K
 * rather than on the logits: rotate q and k with this call, run fat_attn_fwd / fat_attn_bwd on
 * the rotated tensors (no bias), and turn dq and dk back with inverse = 1 (the rotation is
 * orthogonal, so the gradient of the unrotated input is the transposed rotation of the
 * rotated one's).
 *   x, y: bf16 [total_tokens, num_heads, head_dim] (y may equal x: in place); head_dim 64/128;
 *   cu_seqlens as for the attention calls; base > 1; inverse: 0 rotates, 1 turns back.
 * Angles are reduced exactly modulo one turn (64-bit fixed-point turns per position), so cosine
 * and sine carry fp32 accuracy at any position; the result is rounded to bf16.
 * A document longer than max_seqlen, or a corrupt cu_seqlens entry, sets FAT_DEVERR_SEQLENS.
 */
int fat_rope_apply(const fat_shape_t *shape, const void *x, void *y, const int32_t *cu_seqlens,
                   double base, int inverse);

/*
 * The FAT5 report's two other fused kernels ("Noyau Triton" section; their speed and memory are
 * compared with PyTorch in "Torch vs Triton"). The pages print no formulas; the readings:
 *
 * RMSNorm, the T5 layer norm (no mean subtraction, no bias):
 *   rstd = 1 / sqrt(mean_j x_j^2 + eps),  y = weight * x * rstd.
 * fat_rmsnorm_fwd: x, y bf16 [rows, dim]; weight fp32 [dim]; rstd fp32 [rows] (may be NULL; the
 *   backward needs it). dim a multiple of 256, at most 2048.
 * fat_rmsnorm_bwd: gradients of sum(y * dy): dx bf16 [rows, dim] and dweight fp32 [dim], which is
 *   OVERWRITTEN (zeroed by the call, then accumulated with fp32 atomics: order-dependent
 *   rounding). x, weight and rstd as given to / returned by the forward.
 *
 * Cross-entropy with a z-loss term (the auxiliary loss that keeps the log-partition near 0):
 *   lse = log sum_v exp(z_v),  loss = lse - z_target + z_loss * lse^2;
 *   rows with a negative target are ignored (loss 0, gradient 0).
 * fat_cross_entropy: logits bf16 [rows, vocab] (vocab a multiple of 8, at most 65536); target
 *   int32 [rows]; loss and lse fp32 [rows] (either may be NULL). When dlogits (bf16
 *   [rows, vocab]) is not NULL, the gradient of grad_scale * sum(loss) is written there in the
 *   same pass (grad_scale = 1 / number of counted rows gives the mean's gradient):
 *   dz_v = grad_scale * (softmax_v * (1 + 2 z_loss lse) - [v == target]).
 *   A target at or beyond vocab sets FAT_DEVERR_INDEX (that row: loss 0, gradient 0).
 * All three are asynchronous on `stream` (a cudaStream_t), allocate nothing and return FAT_*.
 */
int fat_rmsnorm_fwd(long long rows, int dim, const void *x, const float *weight, float eps,
                    void *y, float *rstd, void *stream);
int fat_rmsnorm_bwd(long long rows, int dim, const void *x, const float *weight,
                    const float *rstd, const void *dy, void *dx, float *dweight, void *stream);
int fat_cross_entropy(long long rows, int vocab, const void *logits, const int32_t *target,
                      float z_loss, float grad_scale, float *loss, float *lse, void *dlogits,
                      void *stream);

/* Synchronises `stream`, reads the current GPU's device error word, clears it, and returns
   FAT_OK if it was zero, else FAT_EDEVICE with the word's bits stored in *bits (if not NULL). */
int fat_attn_get_device_error(void *stream, int *bits);

/* Static English description of a FAT_* return code. */
const char *fat_attn_strerror(int code);

/* Description of the last CUDA call that failed in this thread (which call, its error code and
   text); empty if none has. The string stays valid until the next failing call of the thread. */
const char *fat_attn_last_error_message(void);

/*
 * Host-only helper (no GPU needed): the integer thresholds the kernels compare distances with.
 * For t = 1 .. E-1 (E = nbh - nbh/2 log buckets per direction), thresholds[t-1] is the smallest
 * distance n with bucket_offset(n) >= nbh/2 + t. *count receives E - 1 and *saturation the
 * distance from which the bucket no longer changes. `thresholds` needs room for 63 entries.
 */
int fat_attn_bucket_thresholds(int num_buckets, int max_distance, int bidirectional,
                               int32_t *thresholds, int *count, int *saturation);

#ifdef __cplusplus
}
#endif
#endif /* FAT_ATTN_H */
