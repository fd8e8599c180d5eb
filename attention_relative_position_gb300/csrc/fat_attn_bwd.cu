// fat_attn_bwd.cu -- backward kernel of the fused relative-position attention.
//
// The FAT5 report benchmarks the backward of its bias kernel ("Benchmark / TFLOPS" section)
// without describing it; this is the standard softmax-attention backward of loss = sum(O * dO):
//   P = exp(S' - lse), dV = P^T dO, dP = dO V^T, dS = P * (dP - D) with D = rowsum(dO * O),
//   dK = scale * dS^T Q, dQ = scale * dS K, dTable[b, h] = sum of dS over pairs in bucket b.
//
// GB300 design: the unit of work is a (document, head, 128-key tile) item; its CTA walks the
// query tiles of the document (only those at or after the key tile when causal). Two launch
// shapes: fat_bwd_kernel is persistent (one CTA per SM walks several items; used for d = 64 and
// short documents, where one item's set-up and tail overlap the next item), fat_bwd_tiles_kernel
// has one CTA per item. Everything is computed in the key-major frame (TMEM lane = key row).
// Five warpgroups, one warp of each per SM sub-partition:
//   warps 0-15   four P/dS warpgroups, each owning a quarter of the query columns of a tile.
//                One pass per 16 columns reads S^T and dP^T from TMEM (the next tile's
//                products may then be issued), forms P^T = 2^(x - lse) (bf16 to TMEM: the A
//                operand of dV) and dS^T = P^T (dP^T - D) in fp32 from the same registers
//                (bf16, 128-byte swizzled, to shared memory for the dK / dQ products), and
//                keeps table-gradient partial sums; then a quarter of each dQ tile goes from
//                TMEM into the fp32 dQ accumulator, and at the end a quarter of dK, dV.
//   warp 16      TMA producer: K, V once; Q_i, dO_i (and lse_i, D_i) through a 2-3 stage ring.
//   warps 17-19  MMA issuers (whole warps, one elected lane issues): C = dK += dS^T Q_i,
//                B = dQ_i = dS K (d = 64) or dQ_i^T = K^T dS^T (d = 128), A = S^T = K Q_i^T,
//                dP^T = V dO_i^T and dV += P^T dO_i (P^T from TMEM); fp32 accumulators in
//                TMEM, dK and dV for the whole walk.
// Bias gradient: tiles beyond the T5 saturation distance add dS into one register per side;
// the other tiles reduce each 32-row block along its diagonals with warp shuffles and add the
// sums into a shared-memory array indexed by delta; at the end of each item the CTA folds
// deltas into buckets (segmented warp scan) and adds each run once into the global table
// gradient.
// Query tiles are 128 wide for d = 64 and 64 wide for d = 128 so that S, dP, dQ, P, dK and dV
// fit the 512 TMEM columns together.
#include <algorithm>
#include <cstdio>
#include <type_traits>

#include "fat_attn_internal.cuh"

namespace fat {

template <int D, int NSTAGES>
struct BwdCfg {
  static constexpr int BQ = (D == 64) ? 128 : 64;
  static constexpr int QW = BQ / 4;             // query columns per P/dS warpgroup
  static constexpr int DB = D / 64;
  static constexpr int KBLK = 128 * 128;        // 128 rows x 64 bf16
  static constexpr int KTILE = DB * KBLK;       // K or V tile: 128 keys x D
  static constexpr int QBLK = BQ * 128;         // BQ rows x 64 bf16
  static constexpr int QTILE = DB * QBLK;       // Q_i or dO_i tile
  static constexpr int NS = NSTAGES;            // Q/dO ring depth
  static constexpr int DSBLK = 128 * 128;       // 128 keys x 64 queries bf16
  static constexpr int DSTILE = (BQ / 64) * DSBLK;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KTILE;
  static constexpr int OFF_Q = OFF_V + KTILE;
  static constexpr int OFF_DO = OFF_Q + NS * QTILE;
  static constexpr int OFF_DS = OFF_DO + NS * QTILE;
  // d = 64: each warpgroup stages its 16-channel slice of a dQ tile (128 rows x 64 bytes) here
  // and hands it to the TMA engine as one bulk reduction.
  static constexpr bool DQ_TMA = (D == 64);
  static constexpr int DQS_SLICE = 32 * 16 * 4;  // one warp: 32 rows x 16 channels fp32
  static constexpr int OFF_DQS = OFF_DS + 2 * DSTILE;
  // per Q/dO stage: lse2, dvec, and (one-CTA-per-key-tile kernel) the column terms of linear
  // far-side tiles, -k * j - lse2 for each side's slope term
  static constexpr int OFF_STAT = OFF_DQS + (DQ_TMA ? 16 * DQS_SLICE : 0);
  static constexpr int OFF_BAR = OFF_STAT + NS * 4 * BQ * 4;
  // lut[lut_len] (bias, log2 units), diag[lut_len] (bias-gradient sums per delta), then the
  // bucket of each delta as bytes
  static constexpr int OFF_LUT = OFF_BAR + 256;
  static constexpr int NTHREADS = 640;
  static constexpr int NCOMP = 512;                     // threads of the P/dS warpgroups
  // MMA issuers, one thread each, on three schedulers: S, dP, dV / dQ / dK
  static constexpr int WARP_A = 19, WARP_B = 18, WARP_C = 17;
  // TMEM columns: S^T and dP^T (BQ each), dQ (64), P^T as packed bf16 pairs (BQ/2), dK, dV.
  // P has its own columns so that the next S^T product cannot overwrite it while the dV
  // product may still read it.
  static constexpr int COL_S = 0, COL_DP = BQ, COL_DQ = 2 * BQ, COL_P = 2 * BQ + 64;
  static constexpr int COL_DK = 512 - 2 * D, COL_DV = 512 - D;
  static_assert(COL_P + BQ / 2 <= COL_DK, "TMEM column budget");
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BQ, 0, 0);
  static constexpr uint32_t IDESC_DKV = idesc_bf16_f32(128, D, 0, 1);
  static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, 64, 1, 1);
};

// One unit of work of the persistent backward: a 128-key tile of one (document, head).
struct WorkItem {
  int kb, h, seq_start, L;  // key tile, query head, first query row and query count
  int hk, seq_start_k, Lk;  // key/value head, first key row and key count
  int shift;                // query p sits at key position p + shift (= Lk - L)
  int ks;    // first key of the tile (document-local)
  int i0;    // first query tile walked (causal: the first that sees the key tile)
  int nq;    // number of query tiles walked
  int qrot;  // walk offset
};
// Item ring in shared memory: the producer publishes, with the first Q/dO tile of item i,
// which item follows it, so the P/dS warpgroups need no global loads between items.
struct ItemSlot {
  WorkItem next;
  int more;
  int pad[7];
};
constexpr int kItemSlots = 8;

template <int D, int NS>
size_t bwd_smem_bytes_t(int lut_len) {
  // lut, diag (fp32), bucket ids (bytes), one table column (256 fp32), the staged thresholds
  // (64 int), the item ring
  return 1024 + (size_t)BwdCfg<D, NS>::OFF_LUT + (size_t)lut_len * 9 + 16 + 1024 +
         kMaxThresholds * 4 + kItemSlots * sizeof(ItemSlot) + 16 * sizeof(int4) + kLptRounds * 4;
}
// Three Q/dO stages when they fit next to the bias table, else two.
int bwd_stages(int head_dim, int lut_len) {
  const size_t three = head_dim == 64 ? bwd_smem_bytes_t<64, 3>(lut_len)
                                      : bwd_smem_bytes_t<128, 3>(lut_len);
  return three <= (size_t)kSmemLimit ? 3 : 2;
}
bool bwd_uses_tiles(int head_dim, int max_seqlen_k) {
  return !(head_dim == 64 && (max_seqlen_k + 127) / 128 <= 64);
}
int bwd_query_tile(int head_dim) { return head_dim == 64 ? BwdCfg<64, 2>::BQ : BwdCfg<128, 2>::BQ; }

size_t bwd_smem_bytes(int head_dim, int lut_len) {
  const int ns = bwd_stages(head_dim, lut_len);
  if (head_dim == 64)
    return ns == 3 ? bwd_smem_bytes_t<64, 3>(lut_len) : bwd_smem_bytes_t<64, 2>(lut_len);
  return ns == 3 ? bwd_smem_bytes_t<128, 3>(lut_len) : bwd_smem_bytes_t<128, 2>(lut_len);
}

// TMEM <-> registers for W columns (W = 16 or 32) of this warp's 32 lanes.
template <int W>
__device__ __forceinline__ void tmem_ldw(uint32_t taddr, uint32_t (&r)[W]) {
  if constexpr (W == 32)
    tmem_ld32(taddr, r);
  else
    tmem_ld16(taddr, r);
}
template <int W>
__device__ __forceinline__ void tmem_stw(uint32_t taddr, const uint32_t (&r)[W]) {
  if constexpr (W == 32)
    tmem_st32(taddr, r);
  else if constexpr (W == 16)
    tmem_st16(taddr, r);
  else
    tmem_st8(taddr, r);
}

// 16 channels of one key row of dK (times the softmax scale) and dV, fp32 from TMEM: stored as
// bf16 when every query head has its own key/value head, else added into the fp32 accumulators
// that the query heads of a group share (finished to bf16 by the finishing grid).
__device__ __forceinline__ void store_dkdv_row(const BwdParams &p, size_t off,
                                               const uint32_t (&a)[16], const uint32_t (&b)[16]) {
  if (p.dk_acc == nullptr) {
    uint32_t pa[8], pb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      pa[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * p.scale,
                          __uint_as_float(a[2 * i + 1]) * p.scale);
      pb[i] = pack_bf16x2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
    }
    uint4 *dk4 = reinterpret_cast<uint4 *>(p.dk + off);
    dk4[0] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
    dk4[1] = make_uint4(pa[4], pa[5], pa[6], pa[7]);
    uint4 *dv4 = reinterpret_cast<uint4 *>(p.dv + off);
    dv4[0] = make_uint4(pb[0], pb[1], pb[2], pb[3]);
    dv4[1] = make_uint4(pb[4], pb[5], pb[6], pb[7]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      red_add_v4(p.dk_acc + off + 4 * i, __uint_as_float(a[4 * i]) * p.scale,
                 __uint_as_float(a[4 * i + 1]) * p.scale, __uint_as_float(a[4 * i + 2]) * p.scale,
                 __uint_as_float(a[4 * i + 3]) * p.scale);
      red_add_v4(p.dv_acc + off + 4 * i, __uint_as_float(b[4 * i]), __uint_as_float(b[4 * i + 1]),
                 __uint_as_float(b[4 * i + 2]), __uint_as_float(b[4 * i + 3]));
    }
  }
}

// 16 channels of key row r of a split last-wave CTA's dK and dV (partial sums over its share of
// the query tiles), added into that key tile's fp32 rows of tail_acc (dK scaled here, as above).
template <int D>
__device__ __forceinline__ void add_dkdv_tail(const BwdParams &p, long long tail_cta, int r,
                                              int col, const uint32_t (&a)[16],
                                              const uint32_t (&b)[16]) {
  float *dk = p.tail_acc + ((size_t)tail_cta * 2 * 128 + r) * D + col;
  float *dv = dk + (size_t)128 * D;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    red_add_v4(dk + 4 * i, __uint_as_float(a[4 * i]) * p.scale,
               __uint_as_float(a[4 * i + 1]) * p.scale, __uint_as_float(a[4 * i + 2]) * p.scale,
               __uint_as_float(a[4 * i + 3]) * p.scale);
    red_add_v4(dv + 4 * i, __uint_as_float(b[4 * i]), __uint_as_float(b[4 * i + 1]),
               __uint_as_float(b[4 * i + 2]), __uint_as_float(b[4 * i + 3]));
  }
}

// P^T of one W-column chunk: x = S^T * scale_log2 + bias (log2 units), masked, P = 2^(x - lse2).
// Writes fp32 P into raw (in place of S) and bf16 pairs into pk. Works on column pairs with
// packed fp32x2 arithmetic. Bias forms are compile-time so the unrolled loop carries no
// branches: BIAS 0 = lookup table (lut_row[-j]), 1 = constant rowc, 2 = rowc + kq * j, 3 = the
// same linear form with c + kq * j - lse2 staged per column (lse4 then points at those terms,
// rowc holds the row's part, and x = S^T * scale_log2 + (rowc + term) needs no separate
// subtraction), 4 = a constant bias with c - lse2 staged per column (x = S^T * scale_log2 +
// term).
template <int W, int BIAS, bool MASK>
__device__ __forceinline__ void bwd_p_chunk(uint32_t (&raw)[W], uint32_t (&pk)[W / 2],
                                            const float4 *lse4, const float *lut_row, int jc,
                                            float rowc, float kq, float scale_log2, int lo_j,
                                            int hi_j) {
  const uint64_t sl2 = f2_pack(scale_log2, scale_log2);
  const uint64_t rc2 = f2_pack(rowc, rowc);
  const uint64_t kq2 = f2_pack(kq, kq);
  const float jcf = (float)jc;
#pragma unroll
  for (int g = 0; g < W / 4; ++g) {
    const float4 l4 = lse4[g];
    const uint64_t lv2[2] = {f2_pack(l4.x, l4.y), f2_pack(l4.z, l4.w)};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = 4 * g + 2 * h;
      const int j = jc + t;
      uint64_t b2;
      if (BIAS == 0)
        b2 = f2_pack(lut_row[-j], lut_row[-j - 1]);
      else if (BIAS == 1)
        b2 = rc2;
      else if (BIAS == 2)
        b2 = f2_fma(kq2, f2_pack(jcf + (float)t, jcf + (float)(t + 1)), rc2);
      else if (BIAS == 3)
        b2 = f2_add(rc2, lv2[h]);
      else
        b2 = lv2[h];
      const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(raw[t]), __uint_as_float(raw[t + 1])),
                                 sl2, b2);
      float x0, x1;
      if (BIAS >= 3)
        f2_unpack(x2, x0, x1);
      else
        f2_unpack(f2_sub(x2, lv2[h]), x0, x1);
      if (MASK) {
        x0 = (j >= lo_j && j < hi_j) ? x0 : -INFINITY;
        x1 = (j + 1 >= lo_j && j + 1 < hi_j) ? x1 : -INFINITY;
      }
      const float p0 = ex2(x0), p1 = ex2(x1);
      pk[t / 2] = pack_bf16x2(p0, p1);
      raw[t] = __float_as_uint(p0);
      raw[t + 1] = __float_as_uint(p1);
    }
  }
}

// dS^T of one W-column chunk (columns T0 .. T0+W-1 of a 32-column group): ds = P (dP - D),
// packed to bf16 pairs; returns the chunk's sum. NEAR also reduces the 32-row block along its
// diagonals: lane m accumulates the sum over delta = base + m in acc_a and over
// delta = base + m - 32 in acc_b (base = delta of lane 0, column 0 of the group).
// SUM = false: the chunk's sum is not wanted (no far-side table gradient), so not formed.
template <int W, bool NEAR, int T0, bool SUM = true>
__device__ __forceinline__ float bwd_ds_chunk(const uint32_t (&pf)[W], const uint32_t (&dp)[W],
                                              const float4 *dvs4, uint32_t (&pk)[W / 2],
                                              int lane, float &acc_a, float &acc_b) {
  uint64_t part2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
  float a[2] = {0.f, 0.f}, b[2] = {0.f, 0.f};  // two short dependency chains each
#pragma unroll
  for (int g = 0; g < W / 4; ++g) {
    const float4 d4 = dvs4[g];
    const uint64_t dv2[2] = {f2_pack(d4.x, d4.y), f2_pack(d4.z, d4.w)};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = 4 * g + 2 * h;
      const uint64_t p2 = f2_pack(__uint_as_float(pf[t]), __uint_as_float(pf[t + 1]));
      const uint64_t dp2 = f2_pack(__uint_as_float(dp[t]), __uint_as_float(dp[t + 1]));
      const uint64_t ds2 = f2_mul(p2, f2_sub(dp2, dv2[h]));
      if (SUM) part2[h] = f2_add(part2[h], ds2);
      float ds[2];
      f2_unpack(ds2, ds[0], ds[1]);
      pk[t / 2] = pack_bf16x2(ds[0], ds[1]);
      if (NEAR) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          // the source lane index is taken modulo 32 by the shuffle
          const float y = __shfl_sync(0xffffffffu, ds[e], lane + T0 + t + e);
          if (lane + T0 + t + e < 32)  // one predicated add per element
            a[e] += y;
          else
            b[e] += y;
        }
      }
    }
  }
  if (NEAR) {
    acc_a += a[0] + a[1];
    acc_b += b[0] + b[1];
  }
  if (!SUM) return 0.f;
  float p0, p1;
  f2_unpack(f2_add(part2[0], part2[1]), p0, p1);
  return p0 + p1;
}


// Bucket of key-tile group g = kb * nseq + doc for lpt_order: 64 - the query tiles each of its
// items walks (1..64; longer first), 64 when the group has no item. Corrupt or out-of-bound
// cu_seqlens entries are reported as the rank walk reports them.
template <int BQ>
struct BwdLptBucket {
  const BwdParams &p;
  __device__ int operator()(int g) const {
    const int nseq = p.seq.num_seqs;
    const int kb = g / nseq, doc = g - kb * nseq;
    const DocSpan sp = doc_span(p.seq, doc);
    if (!sp.ok) {
      if (kb == 0) atomicOr(p.err, FAT_DEVERR_SEQLENS);
      return 64;
    }
    if (kb == 0 && (sp.lq > p.seq.max_seqlen || sp.lk > p.seq.max_seqlen_k))
      atomicOr(p.err, FAT_DEVERR_SEQLENS);
    if (kb * 128 >= sp.lk) return 64;
    const int i0 = p.causal ? max(0, kb * 128 - sp.shift) / BQ : 0;
    const int nq = (sp.lq + BQ - 1) / BQ - i0;
    return nq > 0 ? 64 - min(nq, 64) : 64;
  }
};

template <int D, int NSTAGES>
__global__ void __launch_bounds__(640, 1)
    fat_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D, NSTAGES>;
  constexpr int QW = C::QW;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (the 128-byte swizzle atoms need it), reached by indexing the
  // shared array itself so every derived pointer stays a shared-memory pointer
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.seq.total_tokens, H = p.seq.num_heads;

  // Work items: (document, head, 128-key tile), ranked with the key tile slowest (when causal,
  // the first key tiles walk the most query tiles: longest first). Round k of CTA c takes rank
  // k G + c on even rounds and k G + G - 1 - c on odd ones (G CTAs), which evens out the work
  // per CTA; every role walks the same sequence. Items past a document's end are skipped; a
  // corrupt cu_seqlens entry is reported and its items skipped. Documents of different lengths
  // (p.lpt): the ranks come sorted longest-first from lpt_order instead.
  const long long n_virtual = (long long)p.nkb * H * p.seq.num_seqs;
  const long long n_dh = (long long)H * p.seq.num_seqs;
  // documents of different lengths: this CTA's ranks in longest-first order (lpt_order)
  int *lpt_list = reinterpret_cast<int *>(
      sm + C::OFF_LUT + ((p.bias.lut_len * 9 + 15) & ~15) + 1024 + kMaxThresholds * 4 +
      kItemSlots * sizeof(ItemSlot) + 16 * sizeof(int4));
  static_assert(D != 64 || 2 * C::DSTILE >= lpt_scratch_bytes(C::NTHREADS),
                "the ordering scratch fits the dS tiles");
  const int lpt_n = (D == 64 && p.lpt)
                        ? lpt_order(p.nkb * p.seq.num_seqs, p.seq.num_seqs, H, kLptRounds,
                                    BwdLptBucket<C::BQ>{p}, sm + C::OFF_DS, lpt_list)
                        : -1;
  auto next_item = [&](long long &v, WorkItem &w) -> bool {
    for (;; ++v) {
      long long rank;
      if (lpt_n >= 0) {
        if (v >= lpt_n) return false;
        rank = lpt_list[v];
      } else {
        rank = v * gridDim.x +
               ((v & 1) ? (long long)gridDim.x - 1 - blockIdx.x : (long long)blockIdx.x);
        if (rank >= n_virtual) return false;
      }
      const int kb = (int)(rank / n_dh);
      const long long rest = rank % n_dh;
      const int h = (int)(rest % H), doc = (int)(rest / H);
      const DocSpan sp = doc_span(p.seq, doc);
      if (!sp.ok) {  // reported by whichever thread decodes the item
        atomicOr(p.err, FAT_DEVERR_SEQLENS);
        continue;
      }
      // key tiles or query rows of a document longer than the bounds lie beyond the item
      // space: reported
      if (kb == 0 && (sp.lq > p.seq.max_seqlen || sp.lk > p.seq.max_seqlen_k))
        atomicOr(p.err, FAT_DEVERR_SEQLENS);
      if (kb * 128 >= sp.lk) continue;
      w.kb = kb;
      w.h = h;
      w.seq_start = sp.sq;
      w.L = sp.lq;
      w.hk = h / p.seq.group;
      w.seq_start_k = sp.sk;
      w.Lk = sp.lk;
      w.shift = sp.shift;
      w.ks = kb * 128;
      // causal: query p sees key r iff r <= p + shift, so the first query of the tile's
      // walk is ks - shift
      w.i0 = p.causal ? max(0, w.ks - w.shift) / C::BQ : 0;
      w.nq = (w.L + C::BQ - 1) / C::BQ - w.i0;
      if (w.nq <= 0) continue;  // no query of the document sees this key tile
      // query tiles are walked from a per-key-tile offset, so the key-tile CTAs of one head do
      // not all add into the same dQ rows at the same time
      w.qrot = w.nq > 0 ? kb % w.nq : 0;
      return true;
    }
  };
  auto qtile_start = [](const WorkItem &w, int it) {
    const int k = it + w.qrot;
    return (w.i0 + (k >= w.nq ? k - w.nq : k)) * C::BQ;
  };
  long long v_first = 0;  // round index
  WorkItem first;
  if (!next_item(v_first, first)) return;  // nothing to do: before any barrier or allocation
  const bool do_dbias = p.dbias != nullptr && p.bias.table != nullptr;

  uint8_t *sK = sm + C::OFF_K, *sV = sm + C::OFF_V, *sQ = sm + C::OFF_Q, *sDO = sm + C::OFF_DO;
  uint8_t *sDS = sm + C::OFF_DS;
  uint8_t *sDQS = sm + C::OFF_DQS;
  float *s_lse2 = reinterpret_cast<float *>(sm + C::OFF_STAT);
  float *s_dvec = s_lse2 + C::NS * C::BQ;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
  uint64_t *kv_full = bars;
  uint64_t *qd_full = kv_full + 1;       // [NS]
  uint64_t *qd_empty = qd_full + C::NS;  // [NS]
  // (one slot unused: the P/dS warpgroups wait for dP^T only, whose commit follows S^T's
  // products, so its completion covers both)
  uint64_t *dp_full = qd_empty + C::NS + 1;
  uint64_t *p_ready = dp_full + 1;
  uint64_t *ds_ready = p_ready + 1;
  uint64_t *ds_empty = ds_ready + 1;     // [2]
  uint64_t *dq_full = ds_empty + 2;
  uint64_t *dq_empty = dq_full + 1;
  uint64_t *dkdv_done = dq_empty + 1;    // dK, dV of the item complete in TMEM
  uint64_t *mma_done = dkdv_done + 1;    // [3], one per issuer
  uint64_t *s_consumed = mma_done + 3;   // S^T and dP^T of the tile are in registers
  uint64_t *p_free = s_consumed + 1;     // the dV product has read P^T
  uint64_t *kv_empty = p_free + 1;       // the item's last products reading K, V completed
  uint64_t *dkdv_free = kv_empty + 1;    // dK, dV of the item have been read out of TMEM
  uint64_t *comp_sync = dkdv_free + 1;   // P/dS warpgroups: between items
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(comp_sync + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *lut = reinterpret_cast<float *>(sm + C::OFF_LUT);
  float *diag = lut + p.bias.lut_len;
  uint8_t *lbk = reinterpret_cast<uint8_t *>(diag + p.bias.lut_len);
  float *tcol_s = reinterpret_cast<float *>(sm + C::OFF_LUT + ((p.bias.lut_len * 9 + 15) & ~15));
  int *thr_s = reinterpret_cast<int *>(tcol_s + 256);
  ItemSlot *slots = reinterpret_cast<ItemSlot *>(thr_s + kMaxThresholds);
  int4 *last_dq = reinterpret_cast<int4 *>(slots + kItemSlots);  // [16], one per P/dS warp

  // The producer warp sets up the barriers and starts the first item's first step (K, V, the
  // first Q/dO tile and the loads of its lse) before the rest of the block builds its tables, so
  // the load latency overlaps them. The statistics are stored and announced after the block
  // sync (D comes from the preprocessing grid).
  const bool early_q = !(p.debug_flags & 2);
  float lv0[C::BQ / 32];
  if (warp == 16) {
    if (lane == 0) {
      mbar_init(kv_full, 1);
      for (int s = 0; s < C::NS; ++s) {
        mbar_init(qd_full + s, 32);
        mbar_init(qd_empty + s, 2);  // the dV and dK issuers release a stage
      }
      mbar_init(dp_full, 1);
      mbar_init(p_ready, C::NCOMP);
      mbar_init(ds_ready, C::NCOMP);
      mbar_init(ds_empty, 2);  // the dQ and dK products both read dS
      mbar_init(ds_empty + 1, 2);
      mbar_init(dq_full, 1);
      mbar_init(dq_empty, C::NCOMP);
      mbar_init(dkdv_done, 2);
      for (int i = 0; i < 3; ++i) mbar_init(mma_done + i, 1);
      mbar_init(s_consumed, C::NCOMP);
      mbar_init(p_free, 1);
      mbar_init(kv_empty, 2);  // the S/dP and dQ issuers both read K
      mbar_init(dkdv_free, C::NCOMP);
      mbar_init(comp_sync, C::NCOMP);
      *abort_flag = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
    }
    __syncwarp();
    if (early_q) {
      const int qs0 = qtile_start(first, 0);
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, 2 * C::KTILE);
        for (int b = 0; b < C::DB; ++b) {
          tma_load_3d(&tm_k, kv_full, sK + b * C::KBLK, 64 * b, first.hk,
                      first.seq_start_k + first.ks);
          tma_load_3d(&tm_v, kv_full, sV + b * C::KBLK, 64 * b, first.hk,
                      first.seq_start_k + first.ks);
        }
      }
#pragma unroll
      for (int k = 0; k < C::BQ / 32; ++k) {
        const int q = qs0 + lane + 32 * k;
        const size_t idx = (size_t)first.h * T + first.seq_start + q;
        lv0[k] = q < first.L ? __ldg(p.lse + idx) : 0.f;
      }
      if (lane == 0) {
        mbar_expect_tx(qd_full, 2 * C::QTILE);  // the warp's 32 arrivals follow the block sync
        for (int b = 0; b < C::DB; ++b) {
          tma_load_3d(&tm_q, qd_full, sQ + b * C::QBLK, 64 * b, first.h, first.seq_start + qs0);
          tma_load_3d(&tm_do, qd_full, sDO + b * C::QBLK, 64 * b, first.h, first.seq_start + qs0);
        }
      }
    }
  }
  if (warp == 17) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  // bias table of the first item's head; bucket ids (head-independent) for the table gradient
  // and for rebuilding the table when the head changes
  const bool has_table = p.bias.table != nullptr;
  bias_stage(p.bias, first.h, H, thr_s, tcol_s, tid, C::NTHREADS);
  {
    const float slope = p.bias.slopes != nullptr ? __ldg(p.bias.slopes + first.h) : 0.f;
    __syncthreads();
    for (int i = tid; i < p.bias.lut_len; i += C::NTHREADS) {
      const int delta = p.bias.lut_lo + i;
      const int b = has_table ? t5_bucket_staged(delta, p.bias, thr_s) : 0;
      lut[i] = bias_log2_staged(b, delta, slope, p.bias, tcol_s);
      diag[i] = 0.f;
      lbk[i] = static_cast<uint8_t>(b);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Everything above reads only inputs of the backward. D, the zeroed dQ accumulator and the
  // zeroed table gradient come from the preprocessing grid, which this launch may overlap.
  grid_dep_wait();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{abort_flag, p.err, FAT_DEVERR_TIMEOUT_BWD, p.timeout_ns};

  if (warp == 16) {
    // ------------------------------------------------------------------ producer
    int last_q[C::NS];
#pragma unroll
    for (int x = 0; x < C::NS; ++x) last_q[x] = -1;
    int last_kv = -1;
    if (early_q) {
      bool ok = true;
      long long v = v_first;
      int ii = 0, gs = 0;
      WorkItem w = first;
      do {
        long long vnext = v + 1;
        WorkItem wnext;
        const bool more = next_item(vnext, wnext);
        auto publish = [&]() {  // before the arrival on this item's first Q/dO stage
          if (lane == 0) {
            ItemSlot &sl = slots[ii % kItemSlots];
            if (more) sl.next = wnext;
            sl.more = more ? 1 : 0;
          }
        };
        for (int it = 0; it < w.nq; ++it) {
          const int g = gs + it, st = g % C::NS, u = g / C::NS;
          const int qs = qtile_start(w, it);
          if (it == 0) publish();
          if (g == 0) {  // copies started with the block set-up; store its statistics, arrive
#pragma unroll
            for (int k = 0; k < C::BQ / 32; ++k) {
              const int q = qs + lane + 32 * k;
              s_lse2[lane + 32 * k] = lse_to_log2_stat(lv0[k]);
              s_dvec[lane + 32 * k] =
                  q < w.L ? __ldg(p.dvec + (size_t)w.h * T + w.seq_start + q) : 0.f;
            }
            mbar_arrive(qd_full);
            if (lane == 0) last_q[0] = 0;
            continue;
          }
          // fetch this tile's row statistics before waiting for the stage to be free
          float lv[C::BQ / 32], dv[C::BQ / 32];
#pragma unroll
          for (int k = 0; k < C::BQ / 32; ++k) {
            const int q = qs + lane + 32 * k;
            const size_t idx = (size_t)w.h * T + w.seq_start + q;
            lv[k] = q < w.L ? lse_to_log2_stat(__ldg(p.lse + idx)) : 0.f;
            dv[k] = q < w.L ? __ldg(p.dvec + idx) : 0.f;
          }
          if (u > 0 && !warp_wait(qd_empty + st, (u - 1) & 1, wd)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int k = 0; k < C::BQ / 32; ++k) {
            s_lse2[st * C::BQ + lane + 32 * k] = lv[k];
            s_dvec[st * C::BQ + lane + 32 * k] = dv[k];
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(qd_full + st, 2 * C::QTILE);
            for (int b = 0; b < C::DB; ++b) {
              tma_load_3d(&tm_q, qd_full + st, sQ + st * C::QTILE + b * C::QBLK, 64 * b, w.h,
                          w.seq_start + qs);
              tma_load_3d(&tm_do, qd_full + st, sDO + st * C::QTILE + b * C::QBLK, 64 * b, w.h,
                          w.seq_start + qs);
            }
#pragma unroll
            for (int x = 0; x < C::NS; ++x)
              if (x == st) last_q[x] = u;
          } else {
            mbar_arrive(qd_full + st);
          }
          if (it == 0 && ii > 0) {
            // K, V of this item (after its first Q/dO tile), once the previous item's products
            // are done with them
            if (!warp_wait(kv_empty, (ii - 1) & 1, wd)) {
              ok = false;
              break;
            }
            if (lane == 0) {
              mbar_arrive_expect_tx(kv_full, 2 * C::KTILE);
              for (int b = 0; b < C::DB; ++b) {
                tma_load_3d(&tm_k, kv_full, sK + b * C::KBLK, 64 * b, w.hk,
                            w.seq_start_k + w.ks);
                tma_load_3d(&tm_v, kv_full, sV + b * C::KBLK, 64 * b, w.hk,
                            w.seq_start_k + w.ks);
              }
            }
            last_kv = ii;
          }
        }
        if (ii == 0) last_kv = 0;
        gs += w.nq;
        ++ii;
        v = vnext;
        w = wnext;
        if (!more) break;
      } while (ok);
    }
    if (lane == 0) {  // teardown: every copy this thread issued has landed
      if (last_kv >= 0) mbar_wait_teardown(kv_full, last_kv & 1, kTeardownNs);
#pragma unroll
      for (int x = 0; x < C::NS; ++x)
        if (last_q[x] >= 0) mbar_wait_teardown(qd_full + x, last_q[x] & 1, kTeardownNs);
    }
  } else if (warp == C::WARP_A || warp == C::WARP_B || warp == C::WARP_C) {
    // ------------------------------------------------------------------ MMA issuers
    // Three warps on three schedulers: A issues the products that feed and consume P (S^T,
    // dP^T, dV), B the dQ product and C the dK product, so that no chain of hand-offs waits
    // behind another and the issue cost is spread; each Q/dO stage is released by A and C, each
    // dS buffer by B and C, K and V by A and B, and TMEM dK, dV are reused once the P/dS
    // warpgroups have read the previous item's.
    {  // the whole warp runs the loop; one elected lane issues each instruction
      auto issue_qk = [&](uint64_t a0, uint64_t b0, uint32_t dcol) {
        // D[key][q] = sum_c A[key][c] * B[q][c]; A, B K-major
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss_e(tmem + dcol, a0 + (((kk >> 2) * C::KBLK + (kk & 3) * 32) >> 4),
                        b0 + (((kk >> 2) * C::QBLK + (kk & 3) * 32) >> 4), C::IDESC_S, kk > 0);
      };
      bool ok = true;
      long long v = v_first;
      int ii = 0, gs = 0;
      WorkItem w = first;
      if (warp == C::WARP_A) {
        // descriptors built once; moving the start address by b bytes adds b >> 4
        const uint64_t dKk = sw128_desc(smem_u32(sK), 16, 1024);         // K, K-major
        const uint64_t dVk = sw128_desc(smem_u32(sV), 16, 1024);         // V, K-major
        const uint64_t dQk = sw128_desc(smem_u32(sQ), 16, 1024);         // Q_i, K-major
        const uint64_t dDOk = sw128_desc(smem_u32(sDO), 16, 1024);       // dO_i, K-major
        const uint64_t dDOm = sw128_desc(smem_u32(sDO), C::QBLK, 1024);  // dO_i, MN-major
        auto issue_dv = [&](int st, bool acc) {
          // dV[key][c] += sum_q P^T[key][q] dO[q][c]; A = P^T in TMEM, B = dO MN-major
          const uint64_t b0 = dDOm + ((st * C::QTILE) >> 4);
#pragma unroll
          for (int k16 = 0; k16 < C::BQ / 16; ++k16)
            mma_bf16_ts_e(tmem + C::COL_DV, tmem + C::COL_P + 8 * k16, b0 + ((k16 * 2048) >> 4),
                          C::IDESC_DKV, (acc || k16 > 0) ? 1u : 0u);
        };
        auto issue_sdp = [&](int st) {
          issue_qk(dKk, dQk + ((st * C::QTILE) >> 4), C::COL_S);
          issue_qk(dVk, dDOk + ((st * C::QTILE) >> 4), C::COL_DP);
          mma_commit_e(dp_full);
        };
        do {
          if (!warp_wait(kv_full, ii & 1, wd)) { ok = false; break; }
          for (int it = 0; ok && it < w.nq; ++it) {
            const int g = gs + it, st = g % C::NS;
            if (it == 0) {  // the first tile's S^T, dP^T once the previous ones have been read
              if ((g >= 1 && !warp_wait(s_consumed, (g - 1) & 1, wd)) ||
                  !warp_wait(qd_full + st, (g / C::NS) & 1, wd)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_sdp(st);
            }
            // the next tile's S^T and dP^T as soon as this tile's have been read into registers
            // (they run while the P/dS pass computes); after the item's last, K and V are free
            // once these complete
            if (it + 1 < w.nq) {
              const int gn = g + 1;
              if (!warp_wait2(s_consumed, g & 1, qd_full + gn % C::NS, (gn / C::NS) & 1, wd)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_sdp(gn % C::NS);
            } else {
              mma_commit_e(kv_empty);
            }
            if (!warp_wait(p_ready, g & 1, wd)) { ok = false; break; }
            tc_fence_after();
            if (it == 0 && ii > 0) {  // dV in TMEM is reused once the previous item's was read
              if (!warp_wait(dkdv_free, (ii - 1) & 1, wd)) { ok = false; break; }
              tc_fence_after();
            }
            issue_dv(st, it > 0);
            mma_commit_e(p_free);
            mma_commit_e(qd_empty + st);  // this issuer is done with Q_i / dO_i
          }
          if (!ok) break;
          mma_commit_e(dkdv_done);
          gs += w.nq;
          ++ii;
          ++v;
        } while (next_item(v, w));
      } else if (warp == C::WARP_B) {
        const uint64_t dDSm = sw128_desc(smem_u32(sDS), C::DSBLK, 1024);  // dS^T, MN-major
        const uint64_t dKm = sw128_desc(smem_u32(sK), C::KBLK, 1024);     // K, MN-major
        auto issue_dq = [&](int buf) {
          const uint64_t ds0 = dDSm + ((buf * C::DSTILE) >> 4);
#pragma unroll
          for (int k16 = 0; k16 < 8; ++k16) {  // 128 keys
            if (D == 64)  // dQ[q][c] = sum_key dS[q][key] K[key][c]
              mma_bf16_ss_e(tmem + C::COL_DQ, ds0 + ((k16 * 2048) >> 4),
                            dKm + ((k16 * 2048) >> 4), C::IDESC_DQ, k16 > 0);
            else          // dQ^T[c][q] = sum_key K[key][c] dS^T[key][q]
              mma_bf16_ss_e(tmem + C::COL_DQ, dKm + ((k16 * 2048) >> 4),
                            ds0 + ((k16 * 2048) >> 4), C::IDESC_DQ, k16 > 0);
          }
        };
        do {
          for (int it = 0; ok && it < w.nq; ++it) {
            const int g = gs + it;
            if (g >= 1 ? !warp_wait2(ds_ready, g & 1, dq_empty, (g - 1) & 1, wd)
                       : !warp_wait(ds_ready, g & 1, wd)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_dq(g & 1);
            mma_commit_e(dq_full);
            mma_commit_e(ds_empty + (g & 1));
          }
          if (!ok) break;
          mma_commit_e(kv_empty);  // K is free once this item's dQ products complete
          gs += w.nq;
          ++ii;
          ++v;
        } while (next_item(v, w));
      } else {
        const uint64_t dDSk = sw128_desc(smem_u32(sDS), 16, 1024);     // dS^T, K-major
        const uint64_t dQm = sw128_desc(smem_u32(sQ), C::QBLK, 1024);  // Q_i, MN-major
        auto issue_dk = [&](int buf, int st, bool acc) {
          // dK[key][c] += sum_q dS^T[key][q] Q[q][c]; A = dS^T K-major, B = Q MN-major
          const uint64_t a0 = dDSk + ((buf * C::DSTILE) >> 4);
          const uint64_t b0 = dQm + ((st * C::QTILE) >> 4);
#pragma unroll
          for (int k16 = 0; k16 < C::BQ / 16; ++k16)
            mma_bf16_ss_e(tmem + C::COL_DK,
                          a0 + ((((16 * k16) >> 6) * C::DSBLK + (((16 * k16) & 63) >> 4) * 32) >> 4),
                          b0 + ((k16 * 2048) >> 4), C::IDESC_DKV, (acc || k16 > 0) ? 1u : 0u);
        };
        do {
          for (int it = 0; ok && it < w.nq; ++it) {
            const int g = gs + it, st = g % C::NS;
            if (!warp_wait(ds_ready, g & 1, wd)) { ok = false; break; }
            tc_fence_after();
            if (it == 0 && ii > 0) {  // dK in TMEM is reused once the previous item's was read
              if (!warp_wait(dkdv_free, (ii - 1) & 1, wd)) { ok = false; break; }
              tc_fence_after();
            }
            issue_dk(g & 1, st, it > 0);
            mma_commit_e(ds_empty + (g & 1));
            mma_commit_e(qd_empty + st);  // this issuer is done with Q_i
          }
          if (!ok) break;
          mma_commit_e(dkdv_done);
          gs += w.nq;
          ++ii;
          ++v;
        } while (next_item(v, w));
      }
      const int who = warp == C::WARP_A ? 0 : (warp == C::WARP_B ? 1 : 2);
      mma_commit_e(mma_done + who);
      mbar_wait_teardown(mma_done + who, 0, kTeardownNs);
    }
  } else if (warp < 16) {
    // ------------------------------------------------------------------ P / dS warpgroups
    const int wg = warp >> 2;
    const int r = tid & 127;
    const int c0 = wg * QW;  // this warpgroup's first query column
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::COL_S + c0;
    const uint32_t tP = tmem + lane_off + C::COL_P + c0 / 2;
    const uint32_t tDP = tmem + lane_off + C::COL_DP + c0;
    // dS^T store addresses: row r of the 128-byte swizzled tile; the 16-byte group 2 sub + gg of
    // this warpgroup's columns sits at chunk ((c0 & 63) / 8 + 2 sub + gg) ^ (r & 7) (the two
    // terms of the sum have no bit in common)
    const uint32_t ds_row = smem_u32(sDS) + (c0 >> 6) * C::DSBLK + r * 128;
    const uint32_t ds_x = static_cast<uint32_t>((((c0 & 63) >> 3) ^ (r & 7)) << 4);
    const uint32_t tDQ = tmem + lane_off + C::COL_DQ + 16 * wg;  // this warpgroup's dQ quarter
    const bool has_slopes = p.bias.slopes != nullptr;
    bool dq_staged = false;  // this warp has a bulk reduction in flight from its staging slice

    // dQ of global step g into the fp32 accumulator: the tile's first token row0, its head h and
    // the rows left in its document from row0
    auto drain_dq = [&](int g, int row0, int h, int rows) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(dq_full, g & 1, wd))) return false;
      tc_fence_after();
      uint32_t vq[16];
      tmem_ld16(tDQ, vq);
      tc_fence_before();
      mbar_arrive(dq_empty);
      if (C::DQ_TMA) {
        // lane = query row, columns = channels 16*wg ..: each warp stages its 32 x 16 block and
        // lane 0 adds it with one bulk tensor reduction (no synchronisation beyond the warp).
        uint8_t *slice = sDQS + warp * C::DQS_SLICE;
        if (dq_staged) {  // the previous reduction of this slice has finished reading it
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        }
        // 64-byte swizzle (the tensor map's): chunk c of row `lane` sits at c ^ ((lane / 2) % 4),
        // so that the eight rows a store wavefront serves hit eight different bank groups
        uint4 *dst = reinterpret_cast<uint4 *>(slice + lane * 64);
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dst[c ^ sw] = make_uint4(vq[4 * c], vq[4 * c + 1], vq[4 * c + 2], vq[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        // rows past the document end carry zeros (their dS is masked), rows past T are clipped
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, slice, 16 * wg, h, row0 + 32 * (warp & 3));
          bulk_commit_group();
        }
        dq_staged = true;
      } else {  // lane = channel, columns = query rows 16*wg ..
        float *dst = p.dq_acc + ((size_t)(row0 + 16 * wg) * H + h) * D + r;
        const size_t step = (size_t)H * D;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (16 * wg + j < rows) red_add(dst + j * step, __uint_as_float(vq[j]));
      }
      return true;
    };

    bool ok = true;
    int ii = 0, gs = 0;
    WorkItem w = first;
    FarBias fb = far_bias_staged(p.bias, thr_s, tcol_s,
                                 has_slopes ? __ldg(p.bias.slopes + w.h) : 0.f);
    do {
      const int krow = w.ks + r;
      const bool row_valid = krow < w.Lk;
      float acc_pos = 0.f, acc_neg = 0.f;  // table-gradient sums of far tiles, this item
      bool new_head = false;
      float tcol_next = 0.f, slope_next = 0.f;
      for (int it = 0; it < w.nq; ++it) {
        const int g = gs + it, st = g % C::NS;
        const int qs = qtile_start(w, it);
        {  // the three phases tested at once (usually all complete), else waited for in turn
          const uint32_t pq = (g / C::NS) & 1, pd = g & 1, pe = ((g >> 1) - 1) & 1;
          const bool all = g >= 2 ? mbar_try_wait3(qd_full + st, pq, dp_full, pd, ds_empty + (g & 1), pe)
                                  : mbar_try_wait2(qd_full + st, pq, dp_full, pd);
          ok = __all_sync(0xffffffffu, all) ||
               (__all_sync(0xffffffffu, mbar_wait(qd_full + st, pq, wd)) &&
                __all_sync(0xffffffffu, mbar_wait(dp_full, pd, wd)) &&
                (g < 2 || __all_sync(0xffffffffu, mbar_wait(ds_empty + (g & 1), pe, wd))));
        }
        if (!ok) break;
        tc_fence_after();
        if (it == 0) {
          // The next item (published by the producer with this item's first Q/dO tile) and,
          // when its head differs, its head's table column and slope, fetched now so that the
          // switch between items reads shared memory only.
          const ItemSlot &sl = slots[ii % kItemSlots];
          const int hn = sl.next.h;
          new_head = sl.more != 0 && hn != w.h && p.bias.has_bias;
          if (new_head) {
            if (has_table && tid < p.bias.nb)
              tcol_next = __ldg(p.bias.table + (size_t)tid * H + hn);
            if (has_slopes) slope_next = __ldg(p.bias.slopes + hn);
          }
        }
        const int d0 = w.ks - qs - w.shift;  // delta of (key row 0, query column 0)
        const bool need_mask =
            (w.ks + 128 > w.Lk) || (qs + C::BQ > w.L) || (p.causal && d0 + 127 > 0);
        const int lo_j = p.causal ? krow - w.shift - qs : -1;  // first query column that sees it
        const int hi_j = row_valid ? w.L - qs : 0;
        // side: 0 = lookup table, 1 = positive far side, 2 = negative far side, 3 = no bias
        int side;
        float rowc = 0.f, kq = 0.f;  // bias = rowc + kq * j
        if (!p.bias.has_bias) {
          side = 3;
        } else if (d0 - (C::BQ - 1) >= p.bias.sat_pos) {
          side = 1;
          rowc = fmaf(fb.k_pos, (float)(d0 + r), fb.c_pos);
          kq = -fb.k_pos;
        } else if (d0 + 127 <= -p.bias.sat_neg) {
          side = 2;
          rowc = fmaf(fb.k_neg, (float)(d0 + r), fb.c_neg);
          kq = -fb.k_neg;
        } else {
          side = 0;
        }
        const bool linear = has_slopes && (side == 1 || side == 2);
        const int lut_base = d0 + r - p.bias.lut_lo;  // index of (r, j) is lut_base - j
        const float4 *lse4 = reinterpret_cast<const float4 *>(s_lse2 + st * C::BQ + c0);
        const float4 *dvs4 = reinterpret_cast<const float4 *>(s_dvec + st * C::BQ + c0);
        // ---- one pass per 16 query columns: P^T = 2^(x - lse2) (bf16 to TMEM for the dV
        // product), dS^T = P^T (dP^T - D) in fp32 from the same registers (bf16, swizzled, to
        // shared memory for the dK / dQ products). Table gradient: far tiles add into one
        // register per side; near tiles sum each 32-row block along its diagonals with warp
        // shuffles (lane m collects deltas base + m and base + m - 32) and add two values per
        // lane into the per-delta array.
        {
          const float *lut_row = lut + lut_base;
          const float sl = p.scale_log2;
          const uint32_t dsb = ds_row + (g & 1) * C::DSTILE;
          const bool near_db = do_dbias && side == 0;
          float acc_a = 0.f, acc_b = 0.f, part = 0.f;
          // The whole pass is instantiated per (bias form, mask, diagonal reduction) and chosen
          // once per tile, so no chunk carries the other forms' instructions.
          auto pass = [&](auto bias_c, auto mask_c, auto near_c, auto sum_c) -> bool {
            constexpr int BIAS = decltype(bias_c)::value;
            constexpr bool MASK = decltype(mask_c)::value;
            constexpr bool NEAR = decltype(near_c)::value;
            constexpr bool SUM = decltype(sum_c)::value;  // far-side table-gradient sum wanted
#pragma unroll
            for (int sub = 0; sub < QW / 16; ++sub) {
              uint32_t raw[16], dp[16], pk[8];
              tmem_ld16_issue(tS + 16 * sub, raw);
              tmem_ld16_issue(tDP + 16 * sub, dp);
              tmem_ld16_fence(raw);
              tmem_ld16_fence(dp);
              if (sub == QW / 16 - 1) {  // S^T, dP^T fully read: the next ones may be computed
                tc_fence_before();
                mbar_arrive(s_consumed);
              }
              bwd_p_chunk<16, BIAS, MASK>(raw, pk, lse4 + 4 * sub, lut_row, c0 + 16 * sub, rowc,
                                          kq, sl, lo_j, hi_j);
              if (sub == 0 && g >= 1) {  // the previous tile's dV product has read P^T
                if (!__all_sync(0xffffffffu, mbar_wait(p_free, (g - 1) & 1, wd))) return false;
                tc_fence_after();
              }
              tmem_st8(tP + 8 * sub, pk);  // bf16 P^T: A operand of the dV product
              const float4 *d4 = dvs4 + 4 * sub;
              if (sub == 0)
                part += bwd_ds_chunk<16, NEAR, 0, SUM>(raw, dp, d4, pk, lane, acc_a, acc_b);
              else
                part += bwd_ds_chunk<16, NEAR, 16, SUM>(raw, dp, d4, pk, lane, acc_a, acc_b);
#pragma unroll
              for (int gg = 0; gg < 2; ++gg)  // groups of 8 queries = 16 bytes each
                st_shared_v4(dsb + (ds_x ^ ((2 * sub + gg) << 4)), pk[4 * gg], pk[4 * gg + 1],
                             pk[4 * gg + 2], pk[4 * gg + 3]);
            }
            return true;
          };
          using B0 = std::integral_constant<int, 0>;
          using B1 = std::integral_constant<int, 1>;
          using B2 = std::integral_constant<int, 2>;
          using Y = std::true_type;
          using N = std::false_type;
          // the far sides' sums feed only the table gradient
          if (side == 0) {  // lookup table
            if (near_db)
              ok = need_mask ? pass(B0{}, Y{}, Y{}, N{}) : pass(B0{}, N{}, Y{}, N{});
            else
              ok = need_mask ? pass(B0{}, Y{}, N{}, N{}) : pass(B0{}, N{}, N{}, N{});
          } else if (!linear) {  // constant over the tile
            if (do_dbias)
              ok = need_mask ? pass(B1{}, Y{}, N{}, Y{}) : pass(B1{}, N{}, N{}, Y{});
            else
              ok = need_mask ? pass(B1{}, Y{}, N{}, N{}) : pass(B1{}, N{}, N{}, N{});
          } else {  // linear in the query index
            if (do_dbias)
              ok = need_mask ? pass(B2{}, Y{}, N{}, Y{}) : pass(B2{}, N{}, N{}, Y{});
            else
              ok = need_mask ? pass(B2{}, Y{}, N{}, N{}) : pass(B2{}, N{}, N{}, N{});
          }
          if (!ok) break;
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(p_ready);
          if (near_db) {
            // delta of (row of lane m, column t) = base + m - t
            const int base = d0 + 32 * (warp & 3) - c0 - p.bias.lut_lo;
            red_add_shared(diag + base + lane, acc_a);
            if (lane > 0) red_add_shared(diag + base + lane - 32, acc_b);
          } else if (side == 1) {
            acc_pos += part;
          } else if (side == 2) {
            acc_neg += part;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(ds_ready);
        // ---- the previous step's dQ (its product was issued after that step's dS); an item's
        // last one is read after the next item's first dS, so that the wait for it overlaps the
        // dK/dV epilogue and the switch between items
        bool drained;
        if (it >= 1) {
          const int qp = qtile_start(w, it - 1);
          drained = drain_dq(g - 1, w.seq_start + qp, w.h, w.L - qp);
        } else if (g >= 1) {
          const int4 l = last_dq[warp];
          drained = drain_dq(g - 1, l.x, l.y, l.z);
        } else {
          drained = true;
        }
        if (!drained) {
          ok = false;
          break;
        }
      }
      if (ok && w.nq >= 1) {  // where the item's last dQ goes, for the step that drains it
        const int qp = qtile_start(w, w.nq - 1);
        if (lane == 0) last_dq[warp] = make_int4(w.seq_start + qp, w.h, w.L - qp, 0);
        __syncwarp();
      }
      // ---- dK, dV of the item: this warpgroup's quarter of the channels
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(dkdv_done, ii & 1, wd));
      if (!ok) break;
      tc_fence_after();
      // Own key/value heads, d = 64: the item's dK and dV rows go through shared memory, so that
      // the global stores write whole 128-byte rows (a thread holds 16 channels of one row, and
      // rows of one head lie H d 2 bytes apart: stored from registers, every store instruction
      // touched 32 lines, about 2 us per item). The staging area is the dS buffer the item's
      // last step did not use: its products (and the previous step's dQ) have completed.
      const bool stage = D == 64 && p.dk_acc == nullptr;
      const uint32_t stg = smem_u32(sDS) + ((gs + w.nq) & 1) * C::DSTILE;  // dK [128][64], dV
      {
        const int cb = wg * (D / 4);
        const size_t kvrow = ((size_t)(w.seq_start_k + krow) * p.seq.num_heads_kv + w.hk) * D + cb;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t a[16], b[16];
          tmem_ld16_issue(tmem + lane_off + C::COL_DK + cb + 16 * c, a);
          tmem_ld16_issue(tmem + lane_off + C::COL_DV + cb + 16 * c, b);
          tmem_ld16_fence(a);
          tmem_ld16_fence(b);
          if (c == D / 64 - 1) {  // dK, dV read: the next item's products may overwrite them
            tc_fence_before();
            mbar_arrive(dkdv_free);
          }
          if (stage) {
            // row r (128 bytes) at 128 r, its 16-byte chunk j at (j ^ (r & 7)) 16: this
            // warpgroup's chunks 2 wg, 2 wg + 1 land in different bank groups across a warp
            uint32_t pa[8], pb[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              pa[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * p.scale,
                                  __uint_as_float(a[2 * i + 1]) * p.scale);
              pb[i] = pack_bf16x2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
            }
            const uint32_t row = stg + r * 128;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const uint32_t off = static_cast<uint32_t>(((2 * wg + h2) ^ (r & 7)) << 4);
              st_shared_v4(row + off, pa[4 * h2], pa[4 * h2 + 1], pa[4 * h2 + 2], pa[4 * h2 + 3]);
              st_shared_v4(row + 128 * 128 + off, pb[4 * h2], pb[4 * h2 + 1], pb[4 * h2 + 2],
                           pb[4 * h2 + 3]);
            }
          } else if (row_valid) {
            store_dkdv_row(p, kvrow + 16 * c, a, b);
          }
        }
      }

      // ---- table gradient of the item, then the next item's bias table, and the staged dK, dV
      // rows written back (between two syncs of the P/dS warpgroups: bounded waits, so that a
      // warp leaving on a timeout cannot hold the others)
      const bool more = slots[ii % kItemSlots].more != 0;
      if (do_dbias || new_head || stage) {
        if (do_dbias) {  // far sides: one bucket each, added at the saturation deltas
          float a = acc_pos, b = acc_neg;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, off);
            b += __shfl_xor_sync(0xffffffffu, b, off);
          }
          if (lane == 0) {
            if (a != 0.f) red_add_shared(diag + p.bias.sat_pos - p.bias.lut_lo, a);
            if (b != 0.f) red_add_shared(diag - p.bias.sat_neg - p.bias.lut_lo, b);
          }
        }
        if (new_head && tid < p.bias.nb) tcol_s[tid] = tcol_next;
        mbar_arrive(comp_sync);
        if (!__all_sync(0xffffffffu, mbar_wait(comp_sync, 0, wd))) { ok = false; break; }
        if (stage) {  // 2 tensors x 128 rows x 8 chunks, eight threads per row
          const int nvalid = min(128, w.Lk - w.ks);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int idx = tid + C::NCOMP * k;
            const int t = idx >> 10, rr = (idx >> 3) & 127, ch = idx & 7;
            const uint4 val =
                ld_shared_v4(stg + t * (128 * 128) + rr * 128 + ((ch ^ (rr & 7)) << 4));
            if (rr < nvalid) {
              __nv_bfloat16 *dst =
                  (t == 0 ? p.dk : p.dv) +
                  ((size_t)(w.seq_start_k + w.ks + rr) * p.seq.num_heads_kv + w.hk) * D + 8 * ch;
              *reinterpret_cast<uint4 *>(dst) = val;
            }
          }
        }
        if (do_dbias) {
          // per-delta sums to per-bucket sums: each warp takes 32 consecutive deltas, runs of
          // equal buckets are summed with a segmented scan and each run adds once
          for (int base = warp * 32; base < p.bias.lut_len; base += C::NCOMP) {
            const int i = base + lane;
            const bool in = i < p.bias.lut_len;
            float x = in ? diag[i] : 0.f;
            if (in) diag[i] = 0.f;
            const int b = in ? static_cast<int>(lbk[i]) : -1;
            const int b_prev = __shfl_up_sync(0xffffffffu, b, 1);
            const uint32_t heads = __ballot_sync(0xffffffffu, lane == 0 || b_prev != b);
            const int seg = __popc(heads & (0xffffffffu >> (31 - lane)));  // run index
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
              const float xo = __shfl_up_sync(0xffffffffu, x, off);
              const int so = __shfl_up_sync(0xffffffffu, seg, off);
              if (lane >= off && so == seg) x += xo;
            }
            const int seg_next = __shfl_down_sync(0xffffffffu, seg, 1);
            if (in && (lane == 31 || seg_next != seg) && x != 0.f)
              red_add(p.dbias + (size_t)b * H + w.h, x);
          }
        }
        if (new_head) {  // same arithmetic as the set-up's table (bias_log2_staged)
          for (int i = tid; i < p.bias.lut_len; i += C::NCOMP) {
            const int delta = p.bias.lut_lo + i;
            float x = 0.f;
            if (has_table) x += tcol_s[lbk[i]];
            if (has_slopes) x -= slope_next * (float)(delta < 0 ? -delta : delta);
            lut[i] = x * kLog2e;
          }
          fb.c_pos = has_table ? tcol_s[lbk[p.bias.sat_pos - p.bias.lut_lo]] * kLog2e : 0.f;
          fb.c_neg = has_table ? tcol_s[lbk[-p.bias.sat_neg - p.bias.lut_lo]] * kLog2e : 0.f;
          fb.k_pos = has_slopes ? -(slope_next * kLog2e) : 0.f;
          fb.k_neg = has_slopes ? slope_next * kLog2e : 0.f;
        }
        mbar_arrive(comp_sync);
        if (!__all_sync(0xffffffffu, mbar_wait(comp_sync, 1, wd))) { ok = false; break; }
      }
      if (!more) {
        gs += w.nq;
        break;
      }
      gs += w.nq;
      w = slots[ii % kItemSlots].next;
      ++ii;
    } while (true);
    if (ok && gs >= 1) {  // the last item's last dQ
      const int4 l = last_dq[warp];
      ok = drain_dq(gs - 1, l.x, l.y, l.z);
    }
    (void)ok;
    grid_dep_launch();  // the finishing grid may be scheduled
    if (C::DQ_TMA && lane == 0) bulk_wait_all();  // reductions complete before smem is released
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 17) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The same backward as a plain grid of one CTA per (key tile, head, document), used for long
// documents: each CTA walks many query tiles, so there is no set-up to hide, and the hardware
// hands out CTAs in key-tile order (the CTAs in flight share few heads) and balances them.
// TAIL: the launch that takes the split last wave (see BwdParams::tail_first): CTA t of its 1-D
// grid takes part t % tail_splits of key tile CTA tail_first + t / tail_splits; the main launch
// (TAIL = false) leaves those CTAs out.
template <int D, int NSTAGES, bool TAIL>
__global__ void __launch_bounds__(640, 1)
    fat_bwd_tiles_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D, NSTAGES>;
  constexpr int QW = C::QW;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (the 128-byte swizzle atoms need it), reached by indexing the
  // shared array itself so every derived pointer stays a shared-memory pointer
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.seq.total_tokens, H = p.seq.num_heads;
  int kb, h, doc, part = 0, nparts = 1;
  if constexpr (TAIL) {
    const long long cta = p.tail_first + blockIdx.x / p.tail_splits;
    part = (int)(blockIdx.x % p.tail_splits);
    nparts = p.tail_splits;
    kb = (int)(cta % p.nkb);
    h = (int)((cta / p.nkb) % H);
    doc = (int)(cta / ((long long)p.nkb * H));
  } else {
    kb = blockIdx.x;
    h = blockIdx.y;
    doc = blockIdx.z;
    // the split last wave is another launch's
    if (p.tail_splits > 0 &&
        kb + (long long)gridDim.x * (h + (long long)gridDim.y * doc) >= p.tail_first)
      return;
  }
  const DocSpan span = doc_span(p.seq, doc);
  if (!span.ok) {
    if (tid == 0 && kb == 0 && h == 0 && part == 0) atomicOr(p.err, FAT_DEVERR_SEQLENS);
    return;
  }
  const int seq_start = span.sq, L = span.lq;  // queries
  const int seq_start_k = span.sk, Lk = span.lk, shift = span.shift;  // keys
  const int hk = h / p.seq.group;
  if ((L > p.seq.max_seqlen || Lk > p.seq.max_seqlen_k) && kb == 0 && part == 0 && tid == 0)
    atomicOr(p.err, FAT_DEVERR_SEQLENS);
  const int ks = kb * 128;
  if (ks >= Lk) return;
  // causal: query p sees key r iff r <= p + shift, so the walk starts at query ks - shift
  const int i0 = p.causal ? max(0, ks - shift) / C::BQ : 0;
  const int nq_all = (L + C::BQ - 1) / C::BQ - i0;
  if (nq_all <= 0) return;  // no query of the document sees this key tile
  // this CTA's share of the walk: steps [it_lo, it_lo + nq)
  const int it_lo = (int)((long long)part * nq_all / nparts);
  const int nq = (int)((long long)(part + 1) * nq_all / nparts) - it_lo;
  if (nq <= 0) return;
  // Query tiles are walked starting at a per-CTA offset, so the key-tile CTAs of one head do not
  // all add into the same dQ rows at the same time (same-address reductions serialise in L2).
  const int rot = it_lo + kb % nq_all;  // < 2 nq_all
  auto qtile_start = [&](int it) {
    const int k = it + rot;
    return (i0 + (k >= nq_all ? k - nq_all : k)) * C::BQ;
  };
  const bool do_dbias = p.dbias != nullptr && p.bias.table != nullptr;
  // dK, dV of own key/value heads go back as whole rows through the Q/dO ring (a thread holds
  // D / 4 channels of one row, and rows of one head lie H d 2 bytes apart)
  const bool staged_out = !TAIL && p.dk_acc == nullptr;
  static_assert(2 * C::NS * C::QTILE >= 2 * 128 * D * 2, "staging fits the Q/dO ring");

  uint8_t *sK = sm + C::OFF_K, *sV = sm + C::OFF_V, *sQ = sm + C::OFF_Q, *sDO = sm + C::OFF_DO;
  uint8_t *sDS = sm + C::OFF_DS;
  uint8_t *sDQS = sm + C::OFF_DQS;
  float *s_lse2 = reinterpret_cast<float *>(sm + C::OFF_STAT);
  float *s_dvec = s_lse2 + C::NS * C::BQ;
  // far sides: the bias c + kq * j of column j (kq = -k of the side) minus lse2, per column
  float *s_colneg = s_dvec + C::NS * C::BQ;
  float *s_colpos = s_colneg + C::NS * C::BQ;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
  uint64_t *kv_full = bars;
  uint64_t *qd_full = kv_full + 1;       // [NS]
  uint64_t *qd_empty = qd_full + C::NS;  // [NS]
  // (one slot unused: the P/dS warpgroups wait for dP^T only, whose commit follows S^T's
  // products, so its completion covers both)
  uint64_t *dp_full = qd_empty + C::NS + 1;
  uint64_t *p_ready = dp_full + 1;
  uint64_t *ds_ready = p_ready + 1;
  uint64_t *ds_empty = ds_ready + 1;     // [2]
  uint64_t *dq_full = ds_empty + 2;
  uint64_t *dq_empty = dq_full + 1;
  uint64_t *dkdv_done = dq_empty + 1;
  uint64_t *mma_done = dkdv_done + 1;  // [3], one per issuer
  uint64_t *s_consumed = mma_done + 3;  // S^T and dP^T of the tile are in registers
  uint64_t *p_free = s_consumed + 1;    // the dV product has read P^T
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(p_free + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *lut = reinterpret_cast<float *>(sm + C::OFF_LUT);
  float *diag = lut + p.bias.lut_len;
  uint8_t *lbk = reinterpret_cast<uint8_t *>(diag + p.bias.lut_len);

  // The producer warp sets up the barriers and starts its first step (K, V, the first Q/dO tile
  // and the loads of its row statistics) before the rest of the block builds its tables, so the
  // load latency overlaps them. The statistics are stored and announced after the block sync.
  const bool early_q = !(p.debug_flags & 2);
  float lv0[C::BQ / 32];
  if (warp == 16) {
    if (lane == 0) {
      mbar_init(kv_full, 1);
      for (int s = 0; s < C::NS; ++s) {
        mbar_init(qd_full + s, 32);
        mbar_init(qd_empty + s, 2);  // both MMA issuers release a stage
      }
      mbar_init(dp_full, 1);
      mbar_init(p_ready, C::NCOMP);
      mbar_init(ds_ready, C::NCOMP);
      mbar_init(ds_empty, 2);  // the dQ and dK products both read dS
      mbar_init(ds_empty + 1, 2);
      mbar_init(dq_full, 1);
      mbar_init(dq_empty, C::NCOMP);
      mbar_init(dkdv_done, 2);
      for (int i = 0; i < 3; ++i) mbar_init(mma_done + i, 1);
      mbar_init(s_consumed, C::NCOMP);
      mbar_init(p_free, 1);
      *abort_flag = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
    }
    __syncwarp();
    if (early_q) {
      const int qs0 = qtile_start(0);
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, 2 * C::KTILE);
        for (int b = 0; b < C::DB; ++b) {
          tma_load_3d(&tm_k, kv_full, sK + b * C::KBLK, 64 * b, hk, seq_start_k + ks);
          tma_load_3d(&tm_v, kv_full, sV + b * C::KBLK, 64 * b, hk, seq_start_k + ks);
        }
      }
#pragma unroll
      for (int k = 0; k < C::BQ / 32; ++k) {
        const int q = qs0 + lane + 32 * k;
        const size_t idx = (size_t)h * T + seq_start + q;
        lv0[k] = q < L ? __ldg(p.lse + idx) : 0.f;
      }
      if (lane == 0) {
        mbar_expect_tx(qd_full, 2 * C::QTILE);  // the warp's 32 arrivals follow the block sync
        for (int b = 0; b < C::DB; ++b) {
          tma_load_3d(&tm_q, qd_full, sQ + b * C::QBLK, 64 * b, h, seq_start + qs0);
          tma_load_3d(&tm_do, qd_full, sDO + b * C::QBLK, 64 * b, h, seq_start + qs0);
        }
      }
    }
  }
  if (warp == 17) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  {  // bias table of head h; bucket ids and zeroed per-delta sums for the table gradient
    float *col_s = reinterpret_cast<float *>(sm + C::OFF_LUT + ((p.bias.lut_len * 9 + 15) & ~15));
    int *thr_s = reinterpret_cast<int *>(col_s + 256);
    bias_stage(p.bias, h, H, thr_s, col_s, tid, C::NTHREADS);
    const float slope = p.bias.slopes != nullptr ? __ldg(p.bias.slopes + h) : 0.f;
    __syncthreads();
    for (int i = tid; i < p.bias.lut_len; i += C::NTHREADS) {
      const int delta = p.bias.lut_lo + i;
      const int b = p.bias.table ? t5_bucket_staged(delta, p.bias, thr_s) : 0;
      lut[i] = bias_log2_staged(b, delta, slope, p.bias, col_s);
      if (do_dbias) {
        diag[i] = 0.f;
        lbk[i] = static_cast<uint8_t>(b);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Everything above reads only inputs of the backward. D, the zeroed dQ accumulator and the
  // zeroed table gradient come from the preprocessing grid, which this launch may overlap.
  grid_dep_wait();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{abort_flag, p.err, FAT_DEVERR_TIMEOUT_BWD, p.timeout_ns};
  float acc_pos = 0.f, acc_neg = 0.f;  // bias-gradient sums of far tiles (P/dS warps)

  if (warp == 16) {
    // ------------------------------------------------------------------ producer
    int last_q[C::NS];
#pragma unroll
    for (int x = 0; x < C::NS; ++x) last_q[x] = -1;
    const bool kv_issued = early_q && lane == 0;
    // the far-side constants and slope in log2 units (as the P/dS warpgroups' FarBias)
    const FarBias pfb = far_bias_staged(
        p.bias, reinterpret_cast<const int *>(sm + C::OFF_LUT + ((p.bias.lut_len * 9 + 15) & ~15) + 1024),
        reinterpret_cast<const float *>(sm + C::OFF_LUT + ((p.bias.lut_len * 9 + 15) & ~15)),
        p.bias.slopes != nullptr ? __ldg(p.bias.slopes + h) : 0.f);
    auto stage_stats = [&](int st, int k, float lv, float dv) {
      const int j = lane + 32 * k;
      s_lse2[st * C::BQ + j] = lv;
      s_dvec[st * C::BQ + j] = dv;
      s_colneg[st * C::BQ + j] = fmaf(-pfb.k_neg, (float)j, pfb.c_neg - lv);
      s_colpos[st * C::BQ + j] = fmaf(-pfb.k_pos, (float)j, pfb.c_pos - lv);
    };
    if (early_q) {
      // step 0: copies started with the block set-up; store its statistics and arrive
      const int qs0 = qtile_start(0);
#pragma unroll
      for (int k = 0; k < C::BQ / 32; ++k) {
        const int q = qs0 + lane + 32 * k;
        stage_stats(0, k, lse_to_log2_stat(lv0[k]),
                    q < L ? __ldg(p.dvec + (size_t)h * T + seq_start + q) : 0.f);
      }
      mbar_arrive(qd_full);
      if (lane == 0) last_q[0] = 0;
      for (int it = 1; it < nq; ++it) {
        const int st = it % C::NS, u = it / C::NS;
        const int qs = qtile_start(it);
        // fetch this tile's row statistics before waiting for the stage to be free
        float lv[C::BQ / 32], dv[C::BQ / 32];
#pragma unroll
        for (int k = 0; k < C::BQ / 32; ++k) {
          const int q = qs + lane + 32 * k;
          const size_t idx = (size_t)h * T + seq_start + q;
          lv[k] = q < L ? lse_to_log2_stat(__ldg(p.lse + idx)) : 0.f;
          dv[k] = q < L ? __ldg(p.dvec + idx) : 0.f;
        }
        if (u > 0 && !__all_sync(0xffffffffu, mbar_wait(qd_empty + st, (u - 1) & 1, wd))) break;
#pragma unroll
        for (int k = 0; k < C::BQ / 32; ++k) stage_stats(st, k, lv[k], dv[k]);
        if (lane == 0) {
          mbar_arrive_expect_tx(qd_full + st, 2 * C::QTILE);
          for (int b = 0; b < C::DB; ++b) {
            tma_load_3d(&tm_q, qd_full + st, sQ + st * C::QTILE + b * C::QBLK, 64 * b, h,
                        seq_start + qs);
            tma_load_3d(&tm_do, qd_full + st, sDO + st * C::QTILE + b * C::QBLK, 64 * b, h,
                        seq_start + qs);
          }
#pragma unroll
          for (int x = 0; x < C::NS; ++x)
            if (x == st) last_q[x] = u;
        } else {
          mbar_arrive(qd_full + st);
        }
      }
    }
    if (lane == 0) {
      if (kv_issued) mbar_wait_teardown(kv_full, 0, kTeardownNs);
#pragma unroll
      for (int x = 0; x < C::NS; ++x)
        if (last_q[x] >= 0) mbar_wait_teardown(qd_full + x, last_q[x] & 1, kTeardownNs);
    }
  } else if (warp == C::WARP_A || warp == C::WARP_B || warp == C::WARP_C) {
    // ------------------------------------------------------------------ MMA issuers
    // Three warps on three schedulers: A issues the products that feed and consume P (S^T,
    // dP^T, dV), B the dQ product and C the dK product, so that no chain of hand-offs waits
    // behind another and the issue cost is spread; each Q/dO stage is released by A and C, each
    // dS buffer by B and C.
    {  // the whole warp runs the loop; one elected lane issues each instruction
      // descriptors built once; moving the start address by b bytes adds b >> 4
      const uint64_t dKk = sw128_desc(smem_u32(sK), 16, 1024);         // K, K-major
      const uint64_t dVk = sw128_desc(smem_u32(sV), 16, 1024);         // V, K-major
      const uint64_t dQk = sw128_desc(smem_u32(sQ), 16, 1024);         // Q_i, K-major
      const uint64_t dDOk = sw128_desc(smem_u32(sDO), 16, 1024);       // dO_i, K-major
      const uint64_t dQm = sw128_desc(smem_u32(sQ), C::QBLK, 1024);    // Q_i, MN-major
      const uint64_t dDOm = sw128_desc(smem_u32(sDO), C::QBLK, 1024);  // dO_i, MN-major
      const uint64_t dDSk = sw128_desc(smem_u32(sDS), 16, 1024);       // dS^T, K-major
      const uint64_t dDSm = sw128_desc(smem_u32(sDS), C::DSBLK, 1024); // dS^T, MN-major
      const uint64_t dKm = sw128_desc(smem_u32(sK), C::KBLK, 1024);    // K, MN-major
      auto issue_qk = [&](uint64_t a0, uint64_t b0, uint32_t dcol) {
        // D[key][q] = sum_c A[key][c] * B[q][c]; A, B K-major
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss_e(tmem + dcol, a0 + (((kk >> 2) * C::KBLK + (kk & 3) * 32) >> 4),
                      b0 + (((kk >> 2) * C::QBLK + (kk & 3) * 32) >> 4), C::IDESC_S, kk > 0);
      };
      bool ok = true;
      if (warp == C::WARP_A) {
        auto issue_dv = [&](int st, bool acc) {
          // dV[key][c] += sum_q P^T[key][q] dO[q][c]; A = P^T in TMEM, B = dO MN-major
          const uint64_t b0 = dDOm + ((st * C::QTILE) >> 4);
#pragma unroll
          for (int k16 = 0; k16 < C::BQ / 16; ++k16)
            mma_bf16_ts_e(tmem + C::COL_DV, tmem + C::COL_P + 8 * k16, b0 + ((k16 * 2048) >> 4),
                        C::IDESC_DKV, (acc || k16 > 0) ? 1u : 0u);
        };
        ok = warp_wait(kv_full, 0, wd) && warp_wait(qd_full, 0, wd);
        if (ok) {
          tc_fence_after();
          issue_qk(dKk, dQk, C::COL_S);
          issue_qk(dVk, dDOk, C::COL_DP);
          mma_commit_e(dp_full);
        }
        // The next tile's S^T and dP^T as soon as this tile's have been read into registers
        // (they run while the P/dS pass computes); dV once P^T is in TMEM.
        for (int it = 0; ok && it < nq; ++it) {
          const int st = it % C::NS;
          const int stn = (it + 1) % C::NS, un = (it + 1) / C::NS;
          if (it + 1 < nq) {
            if (!warp_wait(s_consumed, it & 1, wd) || !warp_wait(qd_full + stn, un & 1, wd)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_qk(dKk, dQk + ((stn * C::QTILE) >> 4), C::COL_S);
            issue_qk(dVk, dDOk + ((stn * C::QTILE) >> 4), C::COL_DP);
            mma_commit_e(dp_full);
          }
          if (!warp_wait(p_ready, it & 1, wd)) { ok = false; break; }
          tc_fence_after();
          issue_dv(st, it > 0);
          mma_commit_e(p_free);
          mma_commit_e(qd_empty + st);  // this issuer is done with Q_i / dO_i
        }
      } else {
        auto issue_dk = [&](int buf, int st, bool acc) {
          // dK[key][c] += sum_q dS^T[key][q] Q[q][c]; A = dS^T K-major, B = Q MN-major
          const uint64_t a0 = dDSk + ((buf * C::DSTILE) >> 4);
          const uint64_t b0 = dQm + ((st * C::QTILE) >> 4);
#pragma unroll
          for (int k16 = 0; k16 < C::BQ / 16; ++k16)
            mma_bf16_ss_e(tmem + C::COL_DK,
                        a0 + ((((16 * k16) >> 6) * C::DSBLK + (((16 * k16) & 63) >> 4) * 32) >> 4),
                        b0 + ((k16 * 2048) >> 4), C::IDESC_DKV, (acc || k16 > 0) ? 1u : 0u);
        };
        auto issue_dq = [&](int buf) {
          const uint64_t ds0 = dDSm + ((buf * C::DSTILE) >> 4);
#pragma unroll
          for (int k16 = 0; k16 < 8; ++k16) {  // 128 keys
            if (D == 64)  // dQ[q][c] = sum_key dS[q][key] K[key][c]
              mma_bf16_ss_e(tmem + C::COL_DQ, ds0 + ((k16 * 2048) >> 4), dKm + ((k16 * 2048) >> 4),
                          C::IDESC_DQ, k16 > 0);
            else          // dQ^T[c][q] = sum_key K[key][c] dS^T[key][q]
              mma_bf16_ss_e(tmem + C::COL_DQ, dKm + ((k16 * 2048) >> 4), ds0 + ((k16 * 2048) >> 4),
                          C::IDESC_DQ, k16 > 0);
          }
        };
        if (warp == C::WARP_B) {
          for (int it = 0; ok && it < nq; ++it) {
            if (!warp_wait(ds_ready, it & 1, wd)) { ok = false; break; }
            if (it >= 1 && !warp_wait(dq_empty, (it - 1) & 1, wd)) { ok = false; break; }
            tc_fence_after();
            issue_dq(it & 1);
            mma_commit_e(dq_full);
            mma_commit_e(ds_empty + (it & 1));
          }
        } else {
          for (int it = 0; ok && it < nq; ++it) {
            const int st = it % C::NS;
            if (!warp_wait(ds_ready, it & 1, wd)) { ok = false; break; }
            tc_fence_after();
            issue_dk(it & 1, st, it > 0);
            mma_commit_e(ds_empty + (it & 1));
            mma_commit_e(qd_empty + st);  // this issuer is done with Q_i
          }
        }
      }
      if (ok && warp != C::WARP_B) mma_commit_e(dkdv_done);  // the dV and dK issuers
      const int who = warp == C::WARP_A ? 0 : (warp == C::WARP_B ? 1 : 2);
      mma_commit_e(mma_done + who);
      mbar_wait_teardown(mma_done + who, 0, kTeardownNs);
    }
  } else if (warp < 16) {
    // ------------------------------------------------------------------ P / dS warpgroups
    const int wg = warp >> 2;
    const int r = tid & 127;
    const int c0 = wg * QW;  // this warpgroup's first query column
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::COL_S + c0;
    const uint32_t tP = tmem + lane_off + C::COL_P + c0 / 2;
    const uint32_t tDP = tmem + lane_off + C::COL_DP + c0;
    // dS^T store addresses: row r of the 128-byte swizzled tile; the 16-byte group 2 sub + gg of
    // this warpgroup's columns sits at chunk ((c0 & 63) / 8 + 2 sub + gg) ^ (r & 7) (the two
    // terms of the sum have no bit in common)
    const uint32_t ds_row = smem_u32(sDS) + (c0 >> 6) * C::DSBLK + r * 128;
    const uint32_t ds_x = static_cast<uint32_t>((((c0 & 63) >> 3) ^ (r & 7)) << 4);
    const uint32_t tDQ = tmem + lane_off + C::COL_DQ + 16 * wg;  // this warpgroup's dQ quarter
    const int krow = ks + r;
    const bool row_valid = krow < Lk;
    const FarBias fb = far_bias_staged(
        p.bias, reinterpret_cast<const int *>(sm + C::OFF_LUT + ((p.bias.lut_len * 9 + 15) & ~15) + 1024),
        reinterpret_cast<const float *>(sm + C::OFF_LUT + ((p.bias.lut_len * 9 + 15) & ~15)),
        p.bias.slopes != nullptr ? __ldg(p.bias.slopes + h) : 0.f);
    const bool has_slopes = p.bias.slopes != nullptr;

    // dQ tile `it` (quarter of its 64 columns) into the fp32 accumulator (`known`: its product
    // was already seen complete, with the P^T wait of the following step)
    auto drain_dq = [&](int it, bool known) -> bool {
      if (!known && !__all_sync(0xffffffffu, mbar_wait(dq_full, it & 1, wd))) return false;
      tc_fence_after();
      uint32_t v[16];
      tmem_ld16(tDQ, v);
      tc_fence_before();
      mbar_arrive(dq_empty);
      const int qs = qtile_start(it);
      if (C::DQ_TMA) {
        // lane = query row, columns = channels 16*wg ..: each warp stages its 32 x 16 block and
        // lane 0 adds it with one bulk tensor reduction (no synchronisation beyond the warp).
        uint8_t *slice = sDQS + warp * C::DQS_SLICE;
        if (it >= 1) {  // the previous reduction of this slice has finished reading it
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
        }
        // 64-byte swizzle (the tensor map's): chunk c of row `lane` sits at c ^ ((lane / 2) % 4)
        uint4 *dst = reinterpret_cast<uint4 *>(slice + lane * 64);
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dst[c ^ sw] = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        // rows past the document end carry zeros (their dS is masked), rows past T are clipped
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, slice, 16 * wg, h, seq_start + qs + 32 * (warp & 3));
          bulk_commit_group();
        }
      } else {  // lane = channel, columns = query rows 16*wg ..
        float *dst = p.dq_acc + ((size_t)(seq_start + qs + 16 * wg) * H + h) * D + r;
        const size_t step = (size_t)H * D;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (qs + 16 * wg + j < L) red_add(dst + j * step, __uint_as_float(v[j]));
      }
      return true;
    };

    bool ok = true;
    for (int it = 0; it < nq; ++it) {
      const int st = it % C::NS;
      bool dq_known = false;  // the previous step's dQ product seen complete (with P^T's wait)
      const int qs = qtile_start(it);
      {  // the three phases tested at once (usually all complete), else waited for in turn
        const uint32_t pq = (it / C::NS) & 1, pd = it & 1, pe = ((it >> 1) - 1) & 1;
        const bool all = it >= 2 ? mbar_try_wait3(qd_full + st, pq, dp_full, pd, ds_empty + (it & 1), pe)
                                 : mbar_try_wait2(qd_full + st, pq, dp_full, pd);
        ok = __all_sync(0xffffffffu, all) ||
             (__all_sync(0xffffffffu, mbar_wait(qd_full + st, pq, wd)) &&
              __all_sync(0xffffffffu, mbar_wait(dp_full, pd, wd)) &&
              (it < 2 || __all_sync(0xffffffffu, mbar_wait(ds_empty + (it & 1), pe, wd))));
      }
      if (!ok) break;
      tc_fence_after();
      const int d0 = ks - qs - shift;  // delta of (key row 0, query column 0)
      const bool need_mask = (ks + 128 > Lk) || (qs + C::BQ > L) || (p.causal && d0 + 127 > 0);
      const int lo_j = p.causal ? krow - shift - qs : -1;  // first query column that sees it
      const int hi_j = row_valid ? L - qs : 0;
      // side: 0 = lookup table, 1 = positive far side, 2 = negative far side, 3 = no bias
      int side;
      float rowc = 0.f, kq = 0.f;  // bias = rowc + kq * j
      if (!p.bias.has_bias) {
        side = 3;
      } else if (d0 - (C::BQ - 1) >= p.bias.sat_pos) {
        side = 1;
        rowc = fb.k_pos * (float)(d0 + r);  // the row's part; c is in the column terms
        kq = -fb.k_pos;
      } else if (d0 + 127 <= -p.bias.sat_neg) {
        side = 2;
        rowc = fb.k_neg * (float)(d0 + r);
        kq = -fb.k_neg;
      } else {
        side = 0;
      }
      const bool linear = has_slopes && (side == 1 || side == 2);
      const int lut_base = d0 + r - p.bias.lut_lo;  // index of (r, j) is lut_base - j
      const float4 *lse4 = reinterpret_cast<const float4 *>(s_lse2 + st * C::BQ + c0);
      const float4 *dvs4 = reinterpret_cast<const float4 *>(s_dvec + st * C::BQ + c0);
      // far sides (and no bias at all): c + kq * j - lse2 per column, staged by the producer
      const float4 *col4 = reinterpret_cast<const float4 *>(
          (side == 1 ? s_colpos : s_colneg) + st * C::BQ + c0);
      // ---- one pass per 16 query columns: P^T = 2^(x - lse2) (bf16 to TMEM for the dV
      // product), dS^T = P^T (dP^T - D) in fp32 from the same registers (bf16, swizzled, to
      // shared memory for the dK / dQ products). Table gradient: far tiles add into one register
      // per side; near tiles sum each 32-row block along its diagonals with warp shuffles (lane
      // m collects deltas base + m and base + m - 32) and add two values per lane into the
      // per-delta array.
      {
        const float *lut_row = lut + lut_base;
        const float sl = p.scale_log2;
        const uint32_t dsb = ds_row + (it & 1) * C::DSTILE;
        const bool near_db = do_dbias && side == 0;
        float acc_a = 0.f, acc_b = 0.f, part = 0.f;
        // The whole pass is instantiated per (bias form, mask, diagonal reduction) and chosen
        // once per tile, so no chunk carries the other forms' instructions.
        auto pass = [&](auto bias_c, auto mask_c, auto near_c, auto sum_c) -> bool {
          constexpr int BIAS = decltype(bias_c)::value;
          constexpr bool MASK = decltype(mask_c)::value;
          constexpr bool NEAR = decltype(near_c)::value;
          constexpr bool SUM = decltype(sum_c)::value;  // far-side table-gradient sum wanted
          // bf16 P^T of every chunk, written to TMEM (the dV product's A operand) after the pass:
          // the previous tile's dV product, queued behind this tile's S^T and dP^T, has then had
          // time to finish reading the columns
          uint32_t pks[QW / 16][8];
#pragma unroll
          for (int sub = 0; sub < QW / 16; ++sub) {
            uint32_t raw[16], dp[16];
            uint32_t (&pk)[8] = pks[sub];
            tmem_ld16_issue(tS + 16 * sub, raw);
            tmem_ld16_issue(tDP + 16 * sub, dp);
            tmem_ld16_fence(raw);
            tmem_ld16_fence(dp);
            if (sub == QW / 16 - 1) {  // S^T, dP^T fully read: the next tile's may be computed
              tc_fence_before();
              mbar_arrive(s_consumed);
            }
            bwd_p_chunk<16, BIAS, MASK>(raw, pk, (BIAS >= 3 ? col4 : lse4) + 4 * sub, lut_row,
                                        c0 + 16 * sub, rowc, kq, sl, lo_j, hi_j);
            uint32_t dsk[8];
            const float4 *d4 = dvs4 + 4 * sub;
            if (sub == 0)
              part += bwd_ds_chunk<16, NEAR, 0, SUM>(raw, dp, d4, dsk, lane, acc_a, acc_b);
            else
              part += bwd_ds_chunk<16, NEAR, 16, SUM>(raw, dp, d4, dsk, lane, acc_a, acc_b);
#pragma unroll
            for (int gg = 0; gg < 2; ++gg)  // groups of 8 queries = 16 bytes each
              st_shared_v4(dsb + (ds_x ^ ((2 * sub + gg) << 4)), dsk[4 * gg], dsk[4 * gg + 1],
                           dsk[4 * gg + 2], dsk[4 * gg + 3]);
          }
          if (it >= 1) {  // the previous tile's dV product has read P^T; its dQ, tested with it
            dq_known = __all_sync(0xffffffffu, mbar_try_wait2(p_free, (it - 1) & 1, dq_full, (it - 1) & 1));
            if (!dq_known && !__all_sync(0xffffffffu, mbar_wait(p_free, (it - 1) & 1, wd)))
              return false;
            tc_fence_after();
          }
#pragma unroll
          for (int sub = 0; sub < QW / 16; ++sub) tmem_st8(tP + 8 * sub, pks[sub]);
          return true;
        };
        using B0 = std::integral_constant<int, 0>;
        using B3 = std::integral_constant<int, 3>;
        using B4 = std::integral_constant<int, 4>;
        using Y = std::true_type;
        using N = std::false_type;
        // the far sides' sums feed only the table gradient
        if (side == 0) {  // lookup table
          if (near_db)
            ok = need_mask ? pass(B0{}, Y{}, Y{}, N{}) : pass(B0{}, N{}, Y{}, N{});
          else
            ok = need_mask ? pass(B0{}, Y{}, N{}, N{}) : pass(B0{}, N{}, N{}, N{});
        } else if (!linear) {  // constant over the tile (or no bias): the column terms alone
          if (do_dbias)
            ok = need_mask ? pass(B4{}, Y{}, N{}, Y{}) : pass(B4{}, N{}, N{}, Y{});
          else
            ok = need_mask ? pass(B4{}, Y{}, N{}, N{}) : pass(B4{}, N{}, N{}, N{});
        } else {  // linear in the query index (column terms staged with the statistics)
          if (do_dbias)
            ok = need_mask ? pass(B3{}, Y{}, N{}, Y{}) : pass(B3{}, N{}, N{}, Y{});
          else
            ok = need_mask ? pass(B3{}, Y{}, N{}, N{}) : pass(B3{}, N{}, N{}, N{});
        }
        if (!ok) break;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_ready);
        if (near_db) {
          // delta of (row of lane m, column t) = base + m - t
          const int base = d0 + 32 * (warp & 3) - c0 - p.bias.lut_lo;
          red_add_shared(diag + base + lane, acc_a);
          if (lane > 0) red_add_shared(diag + base + lane - 32, acc_b);
        } else if (side == 1) {
          acc_pos += part;
        } else if (side == 2) {
          acc_neg += part;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(ds_ready);
      // ---- the previous tile's dQ (its product was issued after this tile's S^T and dP^T)
      if (it >= 1 && !drain_dq(it - 1, dq_known)) {
        ok = false;
        break;
      }
    }
    if (ok && nq >= 1) ok = drain_dq(nq - 1, false);
    if (C::DQ_TMA && lane == 0) bulk_wait_all();  // reductions complete before shared memory is released
    grid_dep_launch();  // the finishing grid may be scheduled
    // ---- dK, dV: this warpgroup's quarter of the channels
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(dkdv_done, 0, wd));
    if (ok) {
      tc_fence_after();
      const int cb = wg * (D / 4);
      const size_t kvrow = ((size_t)(seq_start_k + krow) * p.seq.num_heads_kv + hk) * D + cb;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t a[16], b[16];
        tmem_ld16_issue(tmem + lane_off + C::COL_DK + cb + 16 * c, a);
        tmem_ld16_issue(tmem + lane_off + C::COL_DV + cb + 16 * c, b);
        tmem_ld16_fence(a);
        tmem_ld16_fence(b);
        if (staged_out) {
          // bf16 rows into the Q/dO ring (its last readers, the dK and dV products, are done):
          // row r at r D 2, its 16-byte chunk j in 128-byte segment j / 8 at ((j % 8) ^ (r % 8))
          uint32_t pa[8], pb[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            pa[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * p.scale,
                                __uint_as_float(a[2 * i + 1]) * p.scale);
            pb[i] = pack_bf16x2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
          }
          const uint32_t row = smem_u32(sQ) + r * (D * 2);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int j = (cb + 16 * c) / 8 + h2;
            const uint32_t off =
                static_cast<uint32_t>((j >> 3) * 128 + (((j & 7) ^ (r & 7)) << 4));
            st_shared_v4(row + off, pa[4 * h2], pa[4 * h2 + 1], pa[4 * h2 + 2], pa[4 * h2 + 3]);
            st_shared_v4(row + 128 * D * 2 + off, pb[4 * h2], pb[4 * h2 + 1], pb[4 * h2 + 2],
                         pb[4 * h2 + 3]);
          }
          continue;
        }
        if (!row_valid) continue;
        if (TAIL && p.dk_acc == nullptr)
          add_dkdv_tail<D>(p, blockIdx.x / p.tail_splits, r, cb + 16 * c, a, b);
        else
          store_dkdv_row(p, kvrow + 16 * c, a, b);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (staged_out && !*abort_flag) {
    // the staged dK, dV rows written back whole: consecutive threads take consecutive 16-byte
    // chunks of a row (2 tensors x 128 rows x D / 8 chunks)
    const int nvalid = min(128, Lk - ks);
    constexpr int CPR = D / 8;  // chunks per row
    for (int idx = tid; idx < 2 * 128 * CPR; idx += C::NTHREADS) {
      const int t = idx / (128 * CPR), rem = idx - t * (128 * CPR);
      const int rr = rem / CPR, j = rem - rr * CPR;
      if (rr >= nvalid) continue;
      const uint4 val = ld_shared_v4(smem_u32(sQ) + t * (128 * D * 2) + rr * (D * 2) +
                                     (j >> 3) * 128 + (((j & 7) ^ (rr & 7)) << 4));
      *reinterpret_cast<uint4 *>((t == 0 ? p.dk : p.dv) +
                                 ((size_t)(seq_start_k + ks + rr) * p.seq.num_heads_kv + hk) * D +
                                 8 * j) = val;
    }
  }
  if (warp == 17) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (do_dbias && !*abort_flag) {
    // Per-delta sums to per-bucket sums: each warp takes 32 consecutive deltas, runs of equal
    // buckets are summed with a segmented scan, and each run adds once to the global gradient.
    for (int base = warp * 32; base < p.bias.lut_len; base += C::NTHREADS) {
      const int i = base + lane;
      const bool in = i < p.bias.lut_len;
      float v = in ? diag[i] : 0.f;
      const int b = in ? static_cast<int>(lbk[i]) : -1;
      const int b_prev = __shfl_up_sync(0xffffffffu, b, 1);
      const uint32_t heads = __ballot_sync(0xffffffffu, lane == 0 || b_prev != b);
      const int seg = __popc(heads & (0xffffffffu >> (31 - lane)));  // run index of this lane
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float vo = __shfl_up_sync(0xffffffffu, v, off);
        const int so = __shfl_up_sync(0xffffffffu, seg, off);
        if (lane >= off && so == seg) v += vo;
      }
      const int seg_next = __shfl_down_sync(0xffffffffu, seg, 1);
      if (in && (lane == 31 || seg_next != seg) && v != 0.f)
        red_add(p.dbias + (size_t)b * H + h, v);
    }
    if (warp < 16) {  // far tiles: one bucket per side
      float a = acc_pos, b = acc_neg;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
      }
      if (lane == 0) {
        if (a != 0.f) red_add(p.dbias + (size_t)t5_bucket_dev(p.bias.sat_pos, p.bias) * H + h, a);
        if (b != 0.f) red_add(p.dbias + (size_t)t5_bucket_dev(-p.bias.sat_neg, p.bias) * H + h, b);
      }
    }
  }
}

int launch_bwd(const BwdParams &p, int head_dim, const void *q, const void *k, const void *v,
               const void *dout, cudaStream_t stream, bool overlap_previous) {
  CUtensorMap mq, mk, mv, mdo, mdq;
  const int T = p.seq.total_tokens, H = p.seq.num_heads;
  const int Tk = p.seq.total_k, Hkv = p.seq.num_heads_kv;
  const int bq = head_dim == 64 ? BwdCfg<64, 2>::BQ : BwdCfg<128, 2>::BQ;
  if (make_tmap_thd(&mq, q, T, H, head_dim, bq) || make_tmap_thd(&mk, k, Tk, Hkv, head_dim, 128) ||
      make_tmap_thd(&mv, v, Tk, Hkv, head_dim, 128) ||
      make_tmap_thd(&mdo, dout, T, H, head_dim, bq) ||
      make_tmap_thd_f32(&mdq, p.dq_acc, T, H, head_dim, 16, 32))
    return (int)cudaErrorInvalidValue;
  const size_t smem = bwd_smem_bytes(head_dim, p.bias.lut_len);
  const int ns = bwd_stages(head_dim, p.bias.lut_len);
  // Short documents with d = 64: the persistent kernel (one CTA per SM walking the items, so
  // the set-up and tail of one item overlap the next). Otherwise one CTA per key tile.
  BwdParams pp = p;
  pp.nkb = (p.seq.max_seqlen_k + 127) / 128;
  const bool persistent = !bwd_uses_tiles(head_dim, p.seq.max_seqlen_k);
  const long long items = (long long)pp.nkb * H * p.seq.num_seqs;
  const int sms = sm_count();
  // one CTA per key tile; a split last wave (CTAs tail_first .. items - 1 in key-tile-fastest
  // order) runs as a second launch of tail_splits CTAs per key tile
  if (persistent || pp.tail_splits <= 1 || pp.tail_first < 0 || pp.tail_first >= items) {
    pp.tail_splits = 0;
    pp.tail_first = items;
  }
  const long long tail_ctas = (items - pp.tail_first) * pp.tail_splits;
  if (tail_ctas > 0x7fffffffLL) return (int)cudaErrorInvalidConfiguration;
  // The persistent grid runs as clusters of two CTAs, which puts CTAs 2c and 2c + 1 on the two
  // SMs of one TPC. Neighbouring CTAs walk neighbouring items (the same document and key tile,
  // adjacent heads), so the two SMs of a pair run the same code path in step. Placed apart (as a
  // launch that overlaps the preprocessing grid places them, SM by SM as it drains), the pairs
  // run unrelated paths and stall on instruction fetch: on the causal varlen workload 3.2 warps
  // per issue instead of 0.9, and 20% longer CTAs. The grid is then an even number of CTAs that
  // fit at once as pairs.
  long long pgrid = std::min<long long>(items, sms > 0 ? sms : 1);
  bool pairs = false;
  if (persistent && items >= 2) {
    const void *fn = ns == 3 ? (const void *)fat_bwd_kernel<64, 3>
                             : (const void *)fat_bwd_kernel<64, 2>;
    if (prepare_kernel(fn, smem, BwdCfg<64, 2>::NTHREADS, 0) == (int)cudaSuccess) {
      const int cap = max_pair_ctas(fn, smem, BwdCfg<64, 2>::NTHREADS) & ~1;
      if (cap >= 2) {
        pgrid = std::min<long long>((items + 1) & ~1LL, cap);
        pairs = true;
      }
    }
  }
  const dim3 grid = persistent ? dim3((unsigned)pgrid) : dim3((unsigned)pp.nkb, H, p.seq.num_seqs);
  // documents of different lengths: the persistent CTAs walk their items longest-first (with
  // equal documents the rank order already is)
  const bool unequal = (long long)p.seq.total_tokens != (long long)p.seq.num_seqs * p.seq.max_seqlen ||
                       (long long)p.seq.total_k != (long long)p.seq.num_seqs * p.seq.max_seqlen_k;
  pp.lpt = (persistent && head_dim == 64 && unequal &&
            (long long)pp.nkb * p.seq.num_seqs <= kLptGroups) ? 1 : 0;
  cudaError_t e;
  bool attr_failed = false;
  auto go = [&](auto kernel, dim3 g, bool overlap, bool cluster2 = false) {
    e = (cudaError_t)prepare_kernel((const void *)kernel, smem, BwdCfg<64, 2>::NTHREADS, 0);
    if (e != cudaSuccess) {
      attr_failed = true;
      return;
    }
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = g;
    cfg.blockDim = dim3(BwdCfg<64, 2>::NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (overlap) {  // programmatic dependent launch on the preprocessing grid
      attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
      ++cfg.numAttrs;
    }
    if (cluster2) {
      attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
      attr[cfg.numAttrs].val.clusterDim.x = 2;
      attr[cfg.numAttrs].val.clusterDim.y = 1;
      attr[cfg.numAttrs].val.clusterDim.z = 1;
      ++cfg.numAttrs;
    }
    e = cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, mdo, mdq, pp);
  };
  // the split last wave: ordered after the main grid by the stream
  const dim3 tail_grid((unsigned)tail_ctas);
  if (head_dim == 64) {
    if (persistent) {
      if (ns == 3) go(fat_bwd_kernel<64, 3>, grid, overlap_previous, pairs);
      else go(fat_bwd_kernel<64, 2>, grid, overlap_previous, pairs);
    } else if (ns == 3) {
      go(fat_bwd_tiles_kernel<64, 3, false>, grid, overlap_previous);
      if (e == cudaSuccess && tail_ctas) go(fat_bwd_tiles_kernel<64, 3, true>, tail_grid, false);
    } else {
      go(fat_bwd_tiles_kernel<64, 2, false>, grid, overlap_previous);
      if (e == cudaSuccess && tail_ctas) go(fat_bwd_tiles_kernel<64, 2, true>, tail_grid, false);
    }
  } else if (ns == 3) {
    go(fat_bwd_tiles_kernel<128, 3, false>, grid, overlap_previous);
    if (e == cudaSuccess && tail_ctas) go(fat_bwd_tiles_kernel<128, 3, true>, tail_grid, false);
  } else {
    go(fat_bwd_tiles_kernel<128, 2, false>, grid, overlap_previous);
    if (e == cudaSuccess && tail_ctas) go(fat_bwd_tiles_kernel<128, 2, true>, tail_grid, false);
  }
  if (attr_failed) return (int)e;  // reason recorded by prepare_kernel
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFuncAttributes fa{};
    if (head_dim == 64)
      cudaFuncGetAttributes(&fa, fat_bwd_kernel<64, 3>);
    else
      cudaFuncGetAttributes(&fa, fat_bwd_kernel<128, 3>);
    char msg[160];
    snprintf(msg, sizeof msg, "%s [regs %d, max threads %d, local %zu B, dyn smem %zu B]",
             cudaGetErrorString(e), fa.numRegs, fa.maxThreadsPerBlock, (size_t)fa.localSizeBytes,
             smem);
    set_last_error("kernel launch", (int)e, msg);
  }
  return (int)e;
}

}  // namespace fat
