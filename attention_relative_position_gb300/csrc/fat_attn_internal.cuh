// fat_attn_internal.cuh -- parameter blocks and device helpers shared by the forward and
// backward kernels of the relative-position attention library (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fat_attn.h"
#include "sm103_ptx.cuh"

namespace fat {

constexpr int kMaxThresholds = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kSmemLimit = 232448;           // 227 KB of dynamic shared memory per block
constexpr long long kDefaultTimeoutNs = 4000000000LL;
constexpr long long kTeardownNs = 200000000LL;
constexpr long long kTurnNs = 20000LL;  // bound of a wait that only orders work

// How the additive bias of relative position delta = k - q is formed.
//   T5 part: table[bucket(delta), h]; the bucket is a pure integer function of delta: exact
//            region n < me, then the number of host-computed thresholds <= n.
//   ALiBi part: -slope_h * |delta|.
// Tiles whose deltas all lie at or beyond the saturation distance on one side get the bias in
// closed form (constant T5 part + linear ALiBi part); the other tiles read a per-block lookup
// table over delta in [lut_lo, lut_lo + lut_len).
struct BiasParams {
  const float *table;   // [nb, H] fp32 or nullptr
  const float *slopes;  // [H] fp32 or nullptr
  int nb, bidir, nbh, me;
  int n_thr;
  int thr[kMaxThresholds];
  int sat_pos;  // every delta >= sat_pos has the same T5 bucket (and |delta| = delta)
  int sat_neg;  // every delta <= -sat_neg has the same T5 bucket (and |delta| = -delta)
  int lut_lo, lut_len;
  int has_bias;
};

// Packed documents. Every document has a query sequence and a key/value sequence of its own
// lengths (the same array for self-attention); query p of a document sits at key position
// p + (Lk - Lq) (bottom-right alignment: the last query lines up with the last key), which is
// what the relative position and the causal mask are measured from. Query head h reads
// key/value head h / group.
struct SeqParams {
  const int32_t *cu_seqlens;    // query side [num_seqs + 1]
  const int32_t *cu_seqlens_k;  // key/value side [num_seqs + 1]
  int num_seqs, num_heads, total_tokens;  // query heads and query rows
  int max_seqlen;    // the caller's bound on every query length (sizes the grids)
  int num_heads_kv, total_k;
  int max_seqlen_k;  // the caller's bound on every key length
  int group;         // num_heads / num_heads_kv
};

// One document's spans, read from both cu_seqlens arrays; ok = false for a corrupt entry.
struct DocSpan {
  int sq, lq, sk, lk, shift;  // shift = lk - lq
  bool ok;
};
__device__ __forceinline__ DocSpan doc_span(const SeqParams &s, int doc) {
  DocSpan d;
  d.sq = __ldg(s.cu_seqlens + doc);
  const int eq = __ldg(s.cu_seqlens + doc + 1);
  d.sk = __ldg(s.cu_seqlens_k + doc);
  const int ek = __ldg(s.cu_seqlens_k + doc + 1);
  d.ok = d.sq >= 0 && eq <= s.total_tokens && eq >= d.sq && d.sk >= 0 && ek <= s.total_k &&
         ek >= d.sk;
  d.lq = eq - d.sq;
  d.lk = ek - d.sk;
  d.shift = d.lk - d.lq;
  return d;
}
// ---- longest-first work order for the persistent kernels ----------------------------------------
// Work order by decreasing cost (documents of different lengths): at most kLptGroups groups are
// sorted, and each CTA keeps at most kLptRounds item ranks.
constexpr int kLptGroups = 8192;
constexpr int kLptRounds = 128;
// shared-memory scratch lpt_order needs for a block of nthreads threads
__host__ __device__ constexpr int lpt_scratch_bytes(int nthreads) {
  return kLptGroups + 4 * (68 + 68 * (nthreads / 32) + kLptGroups);
}

// The item ranks this CTA walks (all threads of the block call it; it synchronises the block).
// Items are ranked r = a * (nseq * H) + doc * H + h for a group g = a * nseq + doc (a is the key
// tile of the backward, the reversed query block of the forward) and head h; bucket(g) gives
// 0..63 (lower costs more) or 64 (a group without items). A plain round-robin over the rank
// order balances the CTAs only when the documents have one length; otherwise a CTA's share
// depends on which documents its rounds happen to hit. Here the groups are sorted by bucket with
// a stable counting sort (so that the H heads of a group stay adjacent: the two CTAs of a pair
// keep walking neighbouring heads) and their items dealt in alternating rounds (round v of CTA
// c takes position v G + c, or v G + G - 1 - c when v is odd, G CTAs): the longest-processing-
// time-first rule. Returns the number of ranks written to list, or -1 when the CTAs would need
// more than max_rounds rounds (every CTA reaches the same answer). scratch: shared memory the
// block does not use yet, lpt_scratch_bytes(blockDim.x) bytes; ng <= kLptGroups.
template <typename BucketFn>
__device__ int lpt_order(int ng, int nseq, int H, int max_rounds, BucketFn bucket,
                         uint8_t *scratch, int *list) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  uint8_t *key = scratch;  // bucket of each group
  int *hist = reinterpret_cast<int *>(scratch + ((ng + 15) & ~15));  // [68]
  int *wcnt = hist + 68;                                              // [warps][68]
  int *sorted = wcnt + nwarps * 68;                                   // [groups with items]
  for (int i = tid; i < 68; i += nthreads) hist[i] = 0;
  __syncthreads();
  for (int g = tid; g < ng; g += nthreads) {
    const int b = bucket(g);
    key[g] = static_cast<uint8_t>(b);
    atomicAdd(hist + b, 1);
  }
  __syncthreads();
  if (warp == 0) {  // bucket starts (exclusive scan of the 65 counts)
    int run = 0;
    for (int b0 = 0; b0 < 65; b0 += 32) {
      const int b = b0 + lane;
      const int c = b < 65 ? hist[b] : 0;
      int x = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (b < 65) hist[b] = run + x - c;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  __syncthreads();
  const int n_valid = hist[64];
  // stable scatter, one group per thread and chunk: rank within the warp by matching buckets,
  // warp offsets per bucket from the chunk's counts
  for (int base = 0; base < ng; base += nthreads) {
    for (int i = tid; i < nwarps * 68; i += nthreads) wcnt[i] = 0;
    __syncthreads();
    const int g = base + tid;
    const int b = g < ng ? key[g] : 255;
    const unsigned peers = __match_any_sync(0xffffffffu, b);
    const int rank_w = __popc(peers & ((1u << lane) - 1u));
    if (b < 64 && rank_w == 0) wcnt[warp * 68 + b] = __popc(peers);
    __syncthreads();
    if (tid < 64) {
      int run = hist[tid];
      for (int w = 0; w < nwarps; ++w) {
        const int c = wcnt[w * 68 + tid];
        wcnt[w * 68 + tid] = run;
        run += c;
      }
      hist[tid] = run;
    }
    __syncthreads();
    if (b < 64) sorted[wcnt[warp * 68 + b] + rank_w] = g;
    __syncthreads();
  }
  const long long total = (long long)n_valid * H;
  const long long G = gridDim.x, c = blockIdx.x;
  const long long rounds = (total + G - 1) / G;
  if (rounds > max_rounds) return -1;
  // rounds before the last are full; the last holds this CTA's position if it is < total
  const long long last = (rounds - 1) * G + (((rounds - 1) & 1) ? G - 1 - c : c);
  const int n = rounds == 0 ? 0 : (int)(rounds - 1) + (last < total ? 1 : 0);
  const long long n_dh = (long long)H * nseq;
  for (int v = tid; v < n; v += nthreads) {
    const long long pos = (long long)v * G + ((v & 1) ? G - 1 - c : c);
    const int g = sorted[pos / H];
    const int h = (int)(pos % H);
    const int a = g / nseq, doc = g - a * nseq;
    list[v] = (int)(a * n_dh + (long long)doc * H + h);
  }
  __syncthreads();
  return n;
}

// natural-log lse of a row -> the log2 statistic the backward subtracts; a row that saw no key
// (lse = -inf) gets +inf, so that every P of the row is 2^-inf = 0
__device__ __forceinline__ float lse_to_log2_stat(float lse) {
  return lse == -INFINITY ? INFINITY : lse * 1.4426950408889634f;
}

__device__ __forceinline__ int t5_bucket_dev(int delta, const BiasParams &b) {
  int off = 0, n;
  if (b.bidir) {
    off = delta > 0 ? b.nbh : 0;
    n = delta < 0 ? -delta : delta;
  } else {
    n = delta < 0 ? -delta : 0;
  }
  if (n < b.me) return off + n;
  int t = 0;
#pragma unroll
  for (int i = 0; i < kMaxThresholds; ++i) t += (i < b.n_thr && n >= b.thr[i]) ? 1 : 0;
  return off + b.me + t;
}

// Building a block's bias table over delta without a global load per entry: the thresholds and
// head h's table column are first staged in shared memory (bias_stage, one load per value, all
// in flight together), then each entry's bucket is a binary search over the staged thresholds
// (the same integer function as t5_bucket_dev: the count of thresholds <= n) and its bias, in
// log2 units, (table[bucket, h] - slope_h |delta|) log2(e) (bias_log2_staged).
__device__ __forceinline__ void bias_stage(const BiasParams &b, int h, int H, int *thr_s,
                                           float *col_s, int tid, int nthreads) {
  for (int i = tid; i < b.n_thr; i += nthreads) thr_s[i] = b.thr[i];
  if (b.table)
    for (int i = tid; i < b.nb; i += nthreads) col_s[i] = __ldg(b.table + (size_t)i * H + h);
}
__device__ __forceinline__ int t5_bucket_staged(int delta, const BiasParams &b,
                                                const int *thr_s) {
  int off = 0, n;
  if (b.bidir) {
    off = delta > 0 ? b.nbh : 0;
    n = delta < 0 ? -delta : delta;
  } else {
    n = delta < 0 ? -delta : 0;
  }
  if (n < b.me) return off + n;
  int lo = 0, hi = b.n_thr;  // thresholds ascend: the first index whose threshold exceeds n
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (thr_s[mid] <= n)
      lo = mid + 1;
    else
      hi = mid;
  }
  return off + b.me + lo;
}
__device__ __forceinline__ float bias_log2_staged(int bucket, int delta, float slope,
                                                  const BiasParams &b, const float *col_s) {
  float v = 0.f;
  if (b.table) v += col_s[bucket];
  if (b.slopes) v -= slope * (float)(delta < 0 ? -delta : delta);
  return v * kLog2e;
}

// Closed-form bias on the far sides, in log2 units: bias(delta) = c + k * delta.
struct FarBias {
  float c_pos, k_pos, c_neg, k_neg;
};

// Each side's constant (the table entry of the saturated bucket) and slope term, from the staged
// thresholds and table column (no global load but the slope's)
__device__ __forceinline__ FarBias far_bias_staged(const BiasParams &b, const int *thr_s,
                                                   const float *col_s, float slope) {
  FarBias f{0.f, 0.f, 0.f, 0.f};
  if (b.table) {
    f.c_pos = col_s[t5_bucket_staged(b.sat_pos, b, thr_s)] * kLog2e;
    f.c_neg = col_s[t5_bucket_staged(-b.sat_neg, b, thr_s)] * kLog2e;
  }
  if (b.slopes) {
    const float s = slope * kLog2e;
    f.k_pos = -s;
    f.k_neg = s;
  }
  return f;
}

// ---------------------------------------------------------------------------------------------
// host-side launch descriptors (filled by the API layer)
// ---------------------------------------------------------------------------------------------
struct FwdParams {
  SeqParams seq;
  BiasParams bias;
  int causal;
  float scale_log2;
  __nv_bfloat16 *out;
  float *lse;
  int *err;
  long long timeout_ns;
  int debug_flags;
  // split along keys: blockIdx.z = document * kv_splits + split; split s takes the key tiles
  // [s * split_tiles, (s + 1) * split_tiles) and writes its normalised partial output (fp32,
  // o_part [kv_splits, T, H, d]) and partial lse (lse_part [kv_splits, H, T]); a combine pass
  // merges them. kv_splits = 1: whole rows, out and lse written directly.
  int kv_splits, split_tiles;
  float *o_part, *lse_part;
  // Balanced last wave (documents of equal length, no causal mask, kv_splits = 1): the CTAs
  // from linear id tail_first on (x fastest in the (tail_gx, H, documents) grid) run as a second
  // launch in which CTA t takes key-tile share t % tail_splits of CTA tail_first +
  // t / tail_splits, writing its normalised partial rows to tail_o [t][256][d] and partial lse
  // to tail_lse [t][256]; a merge pass writes out and lse. tail_splits = 0: no split.
  long long tail_first;
  int tail_splits, tail_gx, tail_ntail;
  float *tail_o, *tail_lse;
  // One-tile CTAs over documents of different lengths (kv_splits = 1): blockIdx.x enumerates the
  // 128-row blocks of all documents, document i owning ids [cu[i] / 128 + i, cu[i + 1] / 128 +
  // i + 1) (at least its ceil(L_i / 128) blocks; an extra id exits at once), so no CTA is spent
  // on rows a short document does not have. 0: the (block, head, document) grid.
  int flat;
  // Persistent one-tile forward: walk the items longest-first (filled by the launcher).
  int lpt;
};

struct BwdParams {
  SeqParams seq;
  BiasParams bias;
  int causal;
  float scale_log2;
  float scale;
  const float *lse;   // [H, T]
  const float *dvec;  // [H, T]: rowsum(dout * out)
  float *dq_acc;      // [T, H, d] fp32
  __nv_bfloat16 *dk, *dv;
  float *dk_acc, *dv_acc;  // [Tk, Hkv, d] fp32 when several query heads share a key/value head
                           // (group > 1): dK, dV accumulate there; else nullptr
  float *dbias;       // [nb, H] or nullptr
  int *err;
  int nkb;            // key tiles of the longest document (filled by the launcher)
  int lpt;            // persistent kernel: walk the items longest-first (filled by the launcher)
  long long timeout_ns;
  int debug_flags;
  // Balanced last wave of the one-CTA-per-key-tile grid (documents of equal length, no causal
  // mask, so every CTA carries the same work): CTA ids >= tail_first come in groups of
  // tail_splits, each group sharing the query tiles of key tile tail_first + (id - tail_first) /
  // tail_splits. Their dK, dV rows are added into tail_acc [tail CTA][dK, dV][128 keys][d] fp32
  // (or into dk_acc / dv_acc when those exist). tail_splits = 0: no split.
  long long tail_first;
  int tail_splits;
  float *tail_acc;
};

// Launchers (defined next to their kernels). Return a cudaError_t value.
int launch_fwd(const FwdParams &p, int head_dim, const void *q, const void *k, const void *v,
               cudaStream_t stream);
// merge the kv_splits partial results of a split forward into out (bf16) and lse
int launch_fwd_combine(const FwdParams &p, int head_dim, cudaStream_t stream);
// Forward CTAs take two 128-row Q tiles (one CTA per SM), or, at d = 64 when no document is
// longer than kFwdOneTileMaxRows, one tile (two CTAs per SM: short documents are bound by each
// CTA's fixed costs, which a second resident CTA overlaps).
constexpr int kFwdOneTileMaxRows = 2048;
int fwd_tiles_per_cta(int head_dim, int max_seqlen);
size_t fwd_smem_bytes(int head_dim, int lut_len, int nt);
// Few-row forward (decode steps, short query chunks): taken when max_seqlen * group rows fit
// the kernel's row tile and its bias lookup table fits shared memory. Same FwdParams contract
// as launch_fwd (kv_splits = 1: out and lse; more: the partials launch_fwd_combine merges).
bool decode_eligible(int head_dim, int max_rows, int group, const BiasParams &b);
int decode_rows(int head_dim, int rows);  // the kernel's row tile for `rows` rows (0: too many)
size_t decode_smem_bytes(int head_dim, int R, int group, const BiasParams &b);
int decode_blocks_per_sm();
int launch_decode(const FwdParams &p, int head_dim, const void *q, const void *k, const void *v,
                  cudaStream_t stream);
// overlap_previous: launch as a programmatic dependent of the previous grid in the stream (only
// when that grid is this library's preprocessing grid, which itself waited for its inputs).
int launch_bwd(const BwdParams &p, int head_dim, const void *q, const void *k, const void *v,
               const void *dout, cudaStream_t stream, bool overlap_previous);
size_t bwd_smem_bytes(int head_dim, int lut_len);
// Whether the backward of this head dimension and key bound runs one CTA per key tile (the grid
// whose last wave can be split), and that grid's query-tile height.
bool bwd_uses_tiles(int head_dim, int max_seqlen_k);
int bwd_query_tile(int head_dim);
int launch_debug_buckets(const BiasParams &b, long long lo, int n, int32_t *out,
                         cudaStream_t stream);

// The host-side argument checks of the backward (everything but the workspace): FAT_OK or the
// FAT_E* code fat_attn_bwd would return for these arguments.
int check_bwd_args(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                   const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                   const float *alibi_slopes, const int32_t *cu_seqlens, const void *out,
                   const float *lse, const void *dout, const void *dq, const void *dk,
                   const void *dv, const float *dbias_table);

// Address of the current device's error word (FAT_OK, or FAT_ECUDA with the reason recorded).
int device_error_address(int **out);

// Before a launch: allow `smem` bytes of dynamic shared memory for kernel `fn` and check that its
// compiled register count times nthreads holds regs_needed (0: no re-balancing), once per
// (kernel, device, size). Returns a cudaError_t value (the reason recorded on failure).
int prepare_kernel(const void *fn, size_t smem, int nthreads, int regs_needed);

// Number of SMs of the current device (cached per device; 0 if the query fails).
int sm_count();

// How many CTAs of kernel `fn` (nthreads threads, smem bytes of dynamic shared memory, set up by
// prepare_kernel) can be resident at once when launched as clusters of two: twice the number of
// co-resident two-CTA clusters, cached per (kernel, device, size); 0 if the query fails.
int max_pair_ctas(const void *fn, size_t smem, int nthreads);

// Record a description of the last failing CUDA call of this thread (read by the C ABI).
void set_last_error(const char *what, int code, const char *text);

// Tensor map over a [T, H, d] bf16 tensor, box = 64 channels x 1 head x box_rows tokens,
// 128-byte swizzle (the shared-memory layout the tcgen05 descriptors expect).
int make_tmap_thd(CUtensorMap *map, const void *ptr, int T, int H, int d, int box_rows);
// Tensor map over a [T, H, d] fp32 tensor, box = box_c channels x 1 head x box_rows tokens (for
// bulk reductions from a shared-memory tile): 64-byte swizzle when a box row is 64 bytes (16-byte
// chunk c of row r at c ^ ((r / 2) % 4)), else row-major without swizzle.
int make_tmap_thd_f32(CUtensorMap *map, const void *ptr, int T, int H, int d, int box_c,
                      int box_rows);

}  // namespace fat
