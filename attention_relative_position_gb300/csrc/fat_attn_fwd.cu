// fat_attn_fwd.cu -- forward kernel: fused attention with an in-kernel relative-position bias.
//
// FAT5 report, "Noyau CUDA" section, second kernel version: Q, K, V are brought from HBM to
// on-chip memory, S = Q K^T, S' = S + (bias built on the fly from relative positions),
// P = softmax(S') computed cumulatively (online), O = P V, and O is written back once.
//
// GB300 design (one CTA = one document x head x 256 query rows = two 128-row Q tiles; three
// warpgroups, so that every SM sub-partition holds one warp of each; short documents at d = 64
// use CTAs of one Q tile, two per SM, with the roles below renumbered):
//   warp 8      TMA producer: Q tiles once, K/V tiles through an NS-stage shared-memory ring.
//   warps 9-10  MMA issuers: S_t = Q_t K_j^T and O_t += P_t V_j with tcgen05.mma, accumulators
//               in tensor memory (TMEM). d = 64: one issuing thread per Q tile, P_t in its own
//               TMEM columns; d = 128: warp 9 issues for both tiles, P_t written over S_t.
//   warp 11     idle (it completes the third warpgroup, which gives its registers to the
//               softmax warpgroups: 216 + 216 + 72 per sub-partition fits its 512 x 32 registers).
//   warps 0-7   two softmax warpgroups, one per Q tile; thread i owns row i of its tile (TMEM
//               lane i), so row max/sum need no shuffles. Bias: closed form on tiles that lie
//               beyond the T5 saturation distance, a per-CTA lookup table over delta on the rest.
//               The running max is only raised (and O rescaled in TMEM) when it grows by more
//               than 2^32, which keeps P <= 2^32 and leaves the final result exact.
// While one warpgroup computes its softmax, the tensor cores run the other tile's MMAs. With
// d = 64 the two warpgroups take their exponential phases in turns (tile 0 of key tile j, then
// tile 1 of key tile j, then tile 0 of key tile j + 1, ...): each finds the special-function
// units to itself, and the other's logits and waits overlap it.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "fat_attn_internal.cuh"

namespace fat {

// NT = Q tiles (128 rows each, one softmax warpgroup each) per CTA. NT = 2: one CTA per SM, both
// tiles share every K/V tile (long documents). NT = 1 (d = 64, short documents): half the
// threads, tensor memory and shared memory, so two CTAs share an SM and one's set-up, first
// loads and epilogue overlap the other's steps.
template <int D, int NT = 2>
struct FwdCfg {
  static_assert(NT == 2 || (NT == 1 && D == 64), "one-tile CTAs are built for d = 64");
  static constexpr int DB = D / 64;           // 64-channel blocks (one 128-byte swizzle row)
  static constexpr int BLK = 128 * 128;       // bytes: 128 rows x 64 bf16
  static constexpr int TILE = DB * BLK;       // bytes: 128 rows x D bf16
  static constexpr int NS = (D == 64 && NT == 2) ? 3 : 2;
  static constexpr int ROWS = 128 * NT;       // query rows per CTA
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NT * TILE;
  static constexpr int OFF_V = OFF_K + NS * TILE;
  static constexpr int OFF_BAR = OFF_V + NS * TILE;
  // the watchdog record and the far-side bias constants (read on slow paths / once per step)
  static constexpr int OFF_WD = OFF_BAR + 256;
  static constexpr int OFF_LUT = OFF_WD + 64;
  static_assert((1 + 4 * NS + 12) * 8 + 8 <= 256, "barrier block");
  // warps 0 .. 4 NT - 1: softmax warpgroups; then the TMA producer, the MMA issuer(s) (the
  // first also allocates tensor memory) and idle warps completing the last warpgroup
  static constexpr int NTHREADS = 128 * NT + 128;
  static constexpr int MIN_BLOCKS = NT == 1 ? 2 : 1;  // CTAs per SM
  static constexpr int WARP_PROD = 4 * NT, WARP_MMA = WARP_PROD + 1;
  // setmaxnreg moves registers within what the block was launched with (NTHREADS x the
  // per-thread count of the launch bound): the split (softmax warpgroups at REG_SM, the other at
  // REG_OTHER) must fit that pool, or the increase waits forever. The launcher also checks it
  // against the compiled count before the first launch.
  static constexpr int REG_SM = NT == 2 ? 216 : 200, REG_OTHER = NT == 2 ? 72 : 56;
  static constexpr int REGS_NEEDED = 128 * NT * REG_SM + 128 * REG_OTHER;
  static_assert(REGS_NEEDED <= NTHREADS * ((65536 / (NTHREADS * MIN_BLOCKS)) & ~7),
                "register split");
  // TMEM columns: S_t at 128 t, O_t at 128 NT + O_STRIDE t. With d = 64 the O_t take 64
  // columns each and P_t (bf16 pairs) gets its own 64 columns after them, so S_t of the next key
  // tile can be computed while P_t is still being produced and consumed; with d = 128 P_t is
  // written over S_t.
  static constexpr bool SEP_P = (D == 64);
  static constexpr uint32_t COL_S0 = 0, COL_O0 = 128 * NT, O_STRIDE = SEP_P ? 64 : 128;
  static constexpr uint32_t COL_P0 = COL_O0 + NT * O_STRIDE;
  static constexpr uint32_t TMEM_COLS = NT == 2 ? 512 : 256;
  static_assert(COL_P0 + (SEP_P ? 64 * NT : 0) <= TMEM_COLS, "TMEM column budget");
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0, 0);  // Q (K-major), K (K-major)
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, 0, 1);   // P (TMEM), V (MN-major)
};

// the bias table, then the staged thresholds (64 int) and table column (256 fp32)
size_t fwd_smem_bytes(int head_dim, int lut_len, int nt) {
  size_t base = head_dim == 64 ? (nt == 1 ? (size_t)FwdCfg<64, 1>::OFF_LUT
                                          : (size_t)FwdCfg<64>::OFF_LUT)
                               : (size_t)FwdCfg<128>::OFF_LUT;
  return 1024 + base + (((size_t)lut_len * 4 + 15) & ~(size_t)15) + kMaxThresholds * 4 + 256 * 4;
}

// Load the S row from TMEM (all four 32-column loads in flight), form
// x = S * scale_log2 + bias - m_ref (log2 units, m_ref the row's current reference max) two
// columns per packed fp32x2 instruction, apply the mask, and return the row maximum of x.
//   MODE 0: bias - m_ref = rowc (constant over the tile; the caller folds m_ref in)
//   MODE 1: bias - m_ref = rowc + kk * j (linear in the key index; likewise)
//   MODE 2: bias = lut_row[j], and nm2 holds -m_ref twice (FOLD; else m_ref is 0)
template <int MODE, bool MASK, bool FOLD>
__device__ __forceinline__ float fwd_logits(uint32_t tS, uint32_t (&x)[4][32], float scale_log2,
                                            float rowc, float kk, const float *lut_row, int lim,
                                            uint64_t nm2) {
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32_issue(tS + c * 32, x[c]);
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32_fence(x[c]);
  const uint64_t sl2 = f2_pack(scale_log2, scale_log2);
  const uint64_t rc2 = f2_pack(rowc, rowc);
  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four short dependency chains
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const int j = c * 32 + i;
      uint64_t b2;
      if (MODE == 0)
        b2 = rc2;
      else if (MODE == 1)
        b2 = f2_pack(fmaf(kk, (float)j, rowc), fmaf(kk, (float)(j + 1), rowc));
      else
        b2 = FOLD ? f2_add(f2_pack(lut_row[j], lut_row[j + 1]), nm2)
                  : f2_pack(lut_row[j], lut_row[j + 1]);
      float v0, v1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(x[c][i]), __uint_as_float(x[c][i + 1])), sl2, b2),
                v0, v1);
      if (MASK) {
        v0 = (j < lim) ? v0 : -INFINITY;
        v1 = (j + 1 < lim) ? v1 : -INFINITY;
      }
      x[c][i] = __float_as_uint(v0);
      x[c][i + 1] = __float_as_uint(v1);
      mx[(i >> 1) & 3] = fmax3(mx[(i >> 1) & 3], v0, v1);
    }
  }
  return fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]);
}

// P = 2^(x - sub) for one row of 128 columns (x already relative to the row's reference max;
// sub is nonzero only when that reference has just moved), packed to bf16 pairs into TMEM,
// with the fp32 sum of the row accumulated in four short dependency chains.
template <bool SUB>
__device__ __forceinline__ void fwd_exp_pass(const uint32_t (&x)[4][32], uint64_t sub2,
                                             uint32_t tP, uint64_t (&sum2)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a = __uint_as_float(x[c][2 * i]), b = __uint_as_float(x[c][2 * i + 1]);
      if (SUB) f2_unpack(f2_sub(f2_pack(a, b), sub2), a, b);
      a = ex2(a);
      b = ex2(b);
      pk[i] = pack_bf16x2(a, b);
      sum2[i & 3] = f2_add(sum2[i & 3], f2_pack(a, b));
    }
    tmem_st16(tP + c * 16, pk);  // P (bf16 pairs): own columns (d 64) or over S (d 128)
  }
}

// Rows that see no key (in this block's key range): out = 0 and lse = -inf, or, for a key range
// of a split forward, a zero partial output with partial lse -inf. Threads thr, thr + nthr, ...
// take rows row0 .. row0 + nrows - 1 (document-local) of query head h.
template <int D, bool TAIL>
__device__ __forceinline__ void fwd_write_empty_rows(const FwdParams &p, int seq_start, int row0,
                                                     int nrows, int h, int split, int q0,
                                                     int thr = threadIdx.x,
                                                     int nthr = blockDim.x) {
  const int T = p.seq.total_tokens, H = p.seq.num_heads;
  for (int i = thr; i < nrows; i += nthr) {
    const size_t row = (size_t)seq_start + row0 + i;
    if (TAIL) {  // partial rows of a split last-wave CTA
      const size_t t = (size_t)blockIdx.x * 256 + (row0 - q0 + i);
      float4 *dst = reinterpret_cast<float4 *>(p.tail_o + t * D);
#pragma unroll
      for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      p.tail_lse[t] = -INFINITY;
    } else if (p.kv_splits == 1) {
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + (row * H + h) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
      if (p.lse != nullptr) p.lse[(size_t)h * T + row] = -INFINITY;
    } else {
      float4 *dst = reinterpret_cast<float4 *>(p.o_part + (((size_t)split * T + row) * H + h) * D);
#pragma unroll
      for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      p.lse_part[((size_t)split * H + h) * T + row] = -INFINITY;
    }
  }
}

// TAIL: the launch that takes a split last wave (FwdParams::tail_first); the main launch
// (TAIL = false) leaves those CTAs out.
template <int D, bool TAIL, int NT = 2>
__global__ void __launch_bounds__(FwdCfg<D, NT>::NTHREADS, FwdCfg<D, NT>::MIN_BLOCKS)
    fat_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D, NT>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (the 128-byte swizzle atoms need it), reached by indexing the
  // shared array itself so every derived pointer stays a shared-memory pointer
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.seq.total_tokens, H = p.seq.num_heads;
  int doc, split, h, qb;
  if constexpr (TAIL) {  // split = this CTA's share of the key tiles
    const long long cta = p.tail_first + blockIdx.x / p.tail_splits;
    split = (int)(blockIdx.x % p.tail_splits);
    h = (int)((cta / p.tail_gx) % H);
    doc = (int)(cta / ((long long)p.tail_gx * H));
    qb = p.tail_gx - 1 - (int)(cta % p.tail_gx);
  } else if (NT == 1 && p.flat) {
    // the last document whose first block id is <= this one (ids rise with the document); the
    // block within it is reversed below (longest rows first when causal)
    const int b = blockIdx.x;
    int lo = 0, hi = p.seq.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((__ldg(p.seq.cu_seqlens + mid) >> 7) + mid <= b)
        lo = mid;
      else
        hi = mid - 1;
    }
    doc = lo;
    split = 0;
    h = blockIdx.y;
    qb = b - ((__ldg(p.seq.cu_seqlens + lo) >> 7) + lo);
    if (b == 0 && h == 0) {  // the whole cu_seqlens array, once (a corrupt one may hide rows)
      const int *cu = p.seq.cu_seqlens;
      for (int i = threadIdx.x; i < p.seq.num_seqs; i += blockDim.x)
        if (__ldg(cu + i) < 0 || __ldg(cu + i + 1) < __ldg(cu + i) ||
            __ldg(cu + i + 1) > p.seq.total_tokens)
          atomicOr(p.err, FAT_DEVERR_SEQLENS);
    }
  } else {
    doc = blockIdx.z / p.kv_splits;
    split = blockIdx.z % p.kv_splits;
    h = blockIdx.y;
    qb = gridDim.x - 1 - blockIdx.x;  // longest rows first when causal
    // the split last wave is another launch's
    if (p.tail_splits > 0 &&
        blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z) >=
            p.tail_first)
      return;
  }
  const int hk = h / p.seq.group;  // key/value head read by query head h

  const DocSpan span = doc_span(p.seq, doc);
  if (!span.ok) {
    if (tid == 0 && qb == 0 && h == 0 && split == 0) atomicOr(p.err, FAT_DEVERR_SEQLENS);
    return;
  }
  const int seq_start = span.sq, L = span.lq, seq_start_k = span.sk, Lk = span.lk;
  const int shift = span.shift;  // query p sits at key position p + shift
  // a document longer than the caller's bounds has rows or keys no block covers: reported
  if ((L > p.seq.max_seqlen || Lk > p.seq.max_seqlen_k) && qb == 0 && split == 0 && tid == 0)
    atomicOr(p.err, FAT_DEVERR_SEQLENS);
  if (NT == 1 && !TAIL && p.flat) {
    const int nblk = (L + 127) >> 7;
    if (qb >= nblk) return;
    qb = nblk - 1 - qb;
  }
  const int q0 = qb * C::ROWS;
  if (q0 >= L) return;  // whole CTA, before any barrier or TMEM allocation
  const int ntile = (NT == 2 && q0 + 128 < L) ? 2 : 1;
  const int nkv_all = (Lk + 127) >> 7;
  // Key tiles Q tile t sees: all of them, or (causal) those up to the key position of its last
  // valid row; intersected with this block's key range [klo, khi) when the keys are split.
  int klo, khi;
  if constexpr (TAIL) {
    klo = (int)((long long)split * nkv_all / p.tail_splits);
    khi = (int)((long long)(split + 1) * nkv_all / p.tail_splits);
  } else {
    klo = split * p.split_tiles;
    khi = min(nkv_all, klo + p.split_tiles);
  }
  auto visible = [&](int t) -> int {
    if (!p.causal) return nkv_all;
    const int last = min(L, q0 + 128 * t + 128) - 1 + shift;
    return last < 0 ? 0 : min((last >> 7) + 1, nkv_all);
  };
  const int nkv0 = max(0, min(khi, visible(0)) - klo);
  const int nkv1 = ntile == 2 ? max(0, min(khi, visible(1)) - klo) : 0;
  const int nkv_max = max(nkv0, nkv1);
  if (nkv_max == 0) {  // no key for any row of the block (in this key range): empty rows
    fwd_write_empty_rows<D, TAIL>(p, seq_start, q0, min(L - q0, C::ROWS), h, split, q0);
    return;
  }
  // Causal rows take their key tiles from the diagonal backwards: the first tile holds each
  // row's largest ALiBi bias, so the running max rarely grows afterwards. Stream position j
  // (the order of the K/V ring) holds key tile kt0 + kdir * j; Q tile t uses positions
  // [jbeg_t, jbeg_t + nkv_t).
  const int kt0 = p.causal ? klo + nkv_max - 1 : klo, kdir = p.causal ? -1 : 1;
  const int jbeg0 = p.causal ? nkv_max - nkv0 : 0, jbeg1 = p.causal ? nkv_max - nkv1 : 0;
  const int nissuers = (nkv0 > 0 ? 1 : 0) + (nkv1 > 0 ? 1 : 0);

  uint8_t *sQ = sm + C::OFF_Q, *sK = sm + C::OFF_K, *sV = sm + C::OFF_V;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *k_full = q_full + 1;
  uint64_t *v_full = k_full + C::NS;
  uint64_t *k_empty = v_full + C::NS;
  uint64_t *v_empty = k_empty + C::NS;
  uint64_t *s_full = v_empty + C::NS;
  uint64_t *p_ready = s_full + 2;
  uint64_t *o_ready = p_ready + 2;
  uint64_t *s_free = o_ready + 2;  // S_t has been read into registers (separate-P layout)
  uint64_t *mma_done = s_free + 2;  // [2], one per issuer
  uint64_t *turn = mma_done + 2;  // [2]: the exponential phase of warpgroup t may start
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(turn + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *lut = reinterpret_cast<float *>(sm + C::OFF_LUT);

  // The producer thread sets up the barriers and starts the first copies (Q, K_0, V_0) before
  // the block builds its bias table, so the load latency overlaps it.
  const bool early = !(p.debug_flags & 1);
  if (warp == C::WARP_PROD && lane == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(k_empty + s, C::SEP_P ? nissuers : 1);  // one release per MMA issuer
      mbar_init(v_empty + s, C::SEP_P ? nissuers : 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full + t, 1);
      mbar_init(p_ready + t, 128);
      mbar_init(o_ready + t, 1);
      mbar_init(s_free + t, 128);
    }
    mbar_init(mma_done, 1);
    mbar_init(mma_done + 1, 1);
    mbar_init(turn, 4);  // one arrival per warp of the other warpgroup
    mbar_init(turn + 1, 4);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (early) {
      mbar_arrive_expect_tx(q_full, ntile * C::TILE);
      for (int t = 0; t < ntile; ++t)
        for (int b = 0; b < C::DB; ++b)
          tma_load_3d(&tm_q, q_full, sQ + t * C::TILE + b * C::BLK, 64 * b, h,
                      seq_start + q0 + 128 * t);
      mbar_arrive_expect_tx(k_full, C::TILE);
      for (int b = 0; b < C::DB; ++b)
        tma_load_3d(&tm_k, k_full, sK + b * C::BLK, 64 * b, hk, seq_start_k + 128 * kt0);
      mbar_arrive_expect_tx(v_full, C::TILE);
      for (int b = 0; b < C::DB; ++b)
        tma_load_3d(&tm_v, v_full, sV + b * C::BLK, 64 * b, hk, seq_start_k + 128 * kt0);
    }
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  {  // bias table of head h over the block's deltas
    int *thr_s = reinterpret_cast<int *>(sm + C::OFF_LUT + ((p.bias.lut_len * 4 + 15) & ~15));
    float *col_s = reinterpret_cast<float *>(thr_s + kMaxThresholds);
    bias_stage(p.bias, h, H, thr_s, col_s, tid, C::NTHREADS);
    const float slope = p.bias.slopes != nullptr ? __ldg(p.bias.slopes + h) : 0.f;
    __syncthreads();
    for (int i = tid; i < p.bias.lut_len; i += C::NTHREADS) {
      const int delta = p.bias.lut_lo + i;
      const int bk = p.bias.table ? t5_bucket_staged(delta, p.bias, thr_s) : 0;
      lut[i] = bias_log2_staged(bk, delta, slope, p.bias, col_s);
    }
    if (tid == 0) {
      *reinterpret_cast<Watchdog *>(sm + C::OFF_WD) =
          Watchdog{abort_flag, p.err, FAT_DEVERR_TIMEOUT_FWD, p.timeout_ns};
      *reinterpret_cast<FarBias *>(sm + C::OFF_WD + 32) =
          far_bias_staged(p.bias, thr_s, col_s, slope);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The watchdog record lives in shared memory: it is read only when a wait is slow, so the
  // roles do not keep it in registers.
  const Watchdog &wd = *reinterpret_cast<const Watchdog *>(sm + C::OFF_WD);

  if (warp >= C::WARP_PROD) regs_dec<C::REG_OTHER>();

  if (warp == C::WARP_PROD) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_k[C::NS], last_v[C::NS];
#pragma unroll
      for (int s = 0; s < C::NS; ++s) last_k[s] = last_v[s] = -1;
      const bool q_issued = early;
      if (early) {
        last_k[0] = last_v[0] = 0;  // Q, K_0 and V_0 were started with the block set-up
        for (int j = 1; j < nkv_max; ++j) {
          const int s = j % C::NS, u = j / C::NS;
          if (u > 0 && !mbar_wait(k_empty + s, (u - 1) & 1, wd)) break;
          mbar_arrive_expect_tx(k_full + s, C::TILE);
          for (int b = 0; b < C::DB; ++b)
            tma_load_3d(&tm_k, k_full + s, sK + s * C::TILE + b * C::BLK, 64 * b, hk,
                        seq_start_k + 128 * (kt0 + kdir * j));
#pragma unroll
          for (int x = 0; x < C::NS; ++x)
            if (x == s) last_k[x] = u;
          if (u > 0 && !mbar_wait(v_empty + s, (u - 1) & 1, wd)) break;
          mbar_arrive_expect_tx(v_full + s, C::TILE);
          for (int b = 0; b < C::DB; ++b)
            tma_load_3d(&tm_v, v_full + s, sV + s * C::TILE + b * C::BLK, 64 * b, hk,
                        seq_start_k + 128 * (kt0 + kdir * j));
#pragma unroll
          for (int x = 0; x < C::NS; ++x)
            if (x == s) last_v[x] = u;
        }
      }
      // teardown: every copy this thread issued has landed before the CTA exits
      if (q_issued) mbar_wait_teardown(q_full, 0, kTeardownNs);
#pragma unroll
      for (int s = 0; s < C::NS; ++s) {
        if (last_k[s] >= 0) mbar_wait_teardown(k_full + s, last_k[s] & 1, kTeardownNs);
        if (last_v[s] >= 0) mbar_wait_teardown(v_full + s, last_v[s] & 1, kTeardownNs);
      }
    }
  } else if (warp == C::WARP_MMA && !C::SEP_P) {
    // ------------------------------------------------------------------ MMA issuer (d = 128)
    // One thread issues for both Q tiles (S_t is overwritten only after P_t V is issued).
    if (lane == 0) {
      const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
      auto issue_S = [&](int t, int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::BLK + (kk & 3) * 32;
          const uint64_t a = sw128_desc(sQa + t * C::TILE + off, 16, 1024);
          const uint64_t b = sw128_desc(sKa + s * C::TILE + off, 16, 1024);
          mma_bf16_ss(tmem + 128 * t, a, b, C::IDESC_S, kk > 0);
        }
      };
      auto issue_PV = [&](int t, int s, bool acc) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t b = sw128_desc(sVa + s * C::TILE + kk * 2048, C::BLK, 1024);
          mma_bf16_ts(tmem + C::COL_O0 + C::O_STRIDE * t, tmem + 128 * t + kk * 8, b, C::IDESC_PV,
                      (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(q_full, 0, wd) && mbar_wait(k_full, 0, wd);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < ntile; ++t) {
          if ((t == 0 ? jbeg0 : jbeg1) > 0) continue;  // this tile starts further down the stream
          issue_S(t, 0);
          mma_commit(s_full + t);
        }
        mma_commit(k_empty);
      }
      for (int j = 0; ok && j < nkv_max; ++j) {
        const int s = j % C::NS, u = j / C::NS;
        const int jn = j + 1, sn = jn % C::NS, un = jn / C::NS;
        if (!mbar_wait(v_full + s, u & 1, wd)) {
          ok = false;
          break;
        }
        bool k_next = false;
        for (int t = 0; t < ntile && ok; ++t) {
          const int jb = t == 0 ? jbeg0 : jbeg1, je = jb + (t == 0 ? nkv0 : nkv1);
          if (j >= jb && j < je) {
            const int jl = j - jb;  // this tile's own step count
            if (!mbar_wait(p_ready + t, jl & 1, wd)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_PV(t, s, jl > 0);
            mma_commit(o_ready + t);
          }
          if (jn >= jb && jn < je) {
            if (!k_next) {
              if (!mbar_wait(k_full + sn, un & 1, wd)) {
                ok = false;
                break;
              }
              tc_fence_after();
              k_next = true;
            }
            issue_S(t, sn);
            mma_commit(s_full + t);
          }
        }
        if (!ok) break;
        mma_commit(v_empty + s);
        if (k_next) mma_commit(k_empty + sn);
      }
      mma_commit(mma_done);
      mbar_wait_teardown(mma_done, 0, kTeardownNs);
    }
  } else if (C::SEP_P && warp >= C::WARP_MMA && warp < C::WARP_MMA + NT) {
    // ------------------------------------------------------------------ MMA issuers (d = 64)
    // One issuing thread per Q tile, so neither tile's hand-offs wait behind the other's.
    // Each K/V stage is released once per active issuer (the barriers count ntile arrivals).
    const int t = warp - C::WARP_MMA;
    const int nk = t == 0 ? nkv0 : nkv1;
    if (lane == 0 && t < ntile && nk > 0) {
      const uint32_t dS_t = tmem + C::COL_S0 + 128 * t;
      const uint32_t dO_t = tmem + C::COL_O0 + C::O_STRIDE * t;
      const uint32_t aP_t = C::SEP_P ? tmem + C::COL_P0 + 64 * t : dS_t;
      // descriptors built once; moving the start address by b bytes adds b >> 4
      const uint64_t dQd = sw128_desc(smem_u32(sQ) + t * C::TILE, 16, 1024);
      const uint64_t dKd = sw128_desc(smem_u32(sK), 16, 1024);
      const uint64_t dVd = sw128_desc(smem_u32(sV), C::BLK, 1024);
      auto issue_S = [&](int st) {
        const uint64_t kd = dKd + ((st * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::BLK + (kk & 3) * 32) >> 4;
          mma_bf16_ss(dS_t, dQd + off, kd + off, C::IDESC_S, kk > 0);
        }
      };
      auto issue_PV = [&](int st, bool acc) {
        const uint64_t vd = dVd + ((st * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(dO_t, aP_t + kk * 8, vd + ((kk * 2048) >> 4), C::IDESC_PV,
                      (acc || kk > 0) ? 1u : 0u);
      };
      const int jb = t == 0 ? jbeg0 : jbeg1, je = jb + nk;
      bool ok = true;
      // stream positions before this tile's first one: release them once loaded, in order
      for (int j = 0; ok && j < jb; ++j) {
        const int s = j % C::NS, u = j / C::NS;
        if (!mbar_wait(k_full + s, u & 1, wd)) { ok = false; break; }
        mbar_arrive(k_empty + s);
        if (!mbar_wait(v_full + s, u & 1, wd)) { ok = false; break; }
        mbar_arrive(v_empty + s);
      }
      ok = ok && mbar_wait(q_full, 0, wd) &&
           mbar_wait(k_full + jb % C::NS, static_cast<uint32_t>((jb / C::NS) & 1), wd);
      if (ok) {
        tc_fence_after();
        issue_S(jb % C::NS);
        mma_commit(s_full + t);
        mma_commit(k_empty + jb % C::NS);
      }
      for (int j = jb; ok && j < je; ++j) {
        const int jl = j - jb;  // this tile's own step count
        const int s = j % C::NS, u = j / C::NS;
        const int jn = j + 1, sn = jn % C::NS, un = jn / C::NS;
        if (C::SEP_P) {  // next key tile's S_t as soon as the softmax has read S_t
          if (!mbar_wait(s_free + t, jl & 1, wd)) { ok = false; break; }
          if (jn < je) {
            if (!mbar_wait(k_full + sn, un & 1, wd)) { ok = false; break; }
            tc_fence_after();
            issue_S(sn);
            mma_commit(s_full + t);
            mma_commit(k_empty + sn);
          }
        }
        if (!mbar_wait(v_full + s, u & 1, wd) || !mbar_wait(p_ready + t, jl & 1, wd)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_PV(s, jl > 0);
        mma_commit(o_ready + t);
        mma_commit(v_empty + s);
        if (!C::SEP_P && jn < je) {  // S_t is overwritten only after P_t V is issued
          if (!mbar_wait(k_full + sn, un & 1, wd)) { ok = false; break; }
          tc_fence_after();
          issue_S(sn);
          mma_commit(s_full + t);
          mma_commit(k_empty + sn);
        }
      }
      // key tiles this Q tile does not need (causal): release them once they have been loaded,
      // in order, so each release lands in the phase of its stage
      for (int j = je; ok && j < nkv_max; ++j) {
        const int s = j % C::NS, u = j / C::NS;
        if (!mbar_wait(k_full + s, u & 1, wd)) { ok = false; break; }
        mbar_arrive(k_empty + s);
        if (!mbar_wait(v_full + s, u & 1, wd)) { ok = false; break; }
        mbar_arrive(v_empty + s);
      }
      mma_commit(mma_done + t);
      mbar_wait_teardown(mma_done + t, 0, kTeardownNs);
    }
  } else if (warp < 4 * NT) {
    // ------------------------------------------------------------------ softmax warpgroups
    regs_inc<C::REG_SM>();
    const int t = warp >> 2;
    if (t < ntile) {
      const int nk = t == 0 ? nkv0 : nkv1;
      const int nk_other = t == 0 ? nkv1 : nkv0;
      const int r = tid & 127;
      const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t tS = tmem + lane_off + C::COL_S0 + 128 * t;
      const uint32_t tO = tmem + lane_off + C::COL_O0 + C::O_STRIDE * t;
      const uint32_t tP = C::SEP_P ? tmem + lane_off + C::COL_P0 + 64 * t : tS;
      const int qs = q0 + 128 * t;  // document-local first row of this tile
      const int qrow = qs + r;
      const FarBias &fb = *reinterpret_cast<const FarBias *>(sm + C::OFF_WD + 32);
      const bool has_slopes = p.bias.slopes != nullptr;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nk; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(s_full + t, j & 1, wd));
        if (!ok) break;
        tc_fence_after();
        const int ks = 128 * (kt0 + kdir * ((t == 0 ? jbeg0 : jbeg1) + j));
        const int d0 = ks - qs - shift;  // delta of (row 0, key 0) of the tile
        const bool need_mask = (ks + 128 > Lk) || (p.causal && d0 + 127 > 0);
        const int lim = min(Lk - ks, p.causal ? (qrow + shift - ks + 1) : 128);
        int mode;
        float rowc = 0.f, kk = 0.f;
        if (!p.bias.has_bias) {
          mode = 0;
        } else if (d0 - 127 >= p.bias.sat_pos) {
          kk = fb.k_pos;
          rowc = fmaf(fb.k_pos, (float)(d0 - r), fb.c_pos);
          mode = has_slopes ? 1 : 0;
        } else if (d0 + 127 <= -p.bias.sat_neg) {
          kk = fb.k_neg;
          rowc = fmaf(fb.k_neg, (float)(d0 - r), fb.c_neg);
          mode = has_slopes ? 1 : 0;
        } else {
          mode = 2;
        }
        const float *lut_row = lut + (d0 - r - p.bias.lut_lo);
        // d = 128: logits relative to the row's current max, so that the exponentials need no
        // subtraction unless the max moves (with d = 64 the extra registers cost more than the
        // subtraction saves)
        constexpr bool FOLD = !C::SEP_P;
        const float m_ref = (FOLD && m != -INFINITY) ? m : 0.f;
        rowc -= m_ref;
        const uint64_t nm2 = f2_pack(-m_ref, -m_ref);
        uint32_t x[4][32];
        float mx;  // row max of x (relative to m_ref)
#define FAT_LOGITS(MODE, MASK) \
  fwd_logits<MODE, MASK, FOLD>(tS, x, p.scale_log2, rowc, kk, lut_row, lim, nm2)
        if (mode == 0)
          mx = need_mask ? FAT_LOGITS(0, true) : FAT_LOGITS(0, false);
        else if (mode == 1)
          mx = need_mask ? FAT_LOGITS(1, true) : FAT_LOGITS(1, false);
        else
          mx = need_mask ? FAT_LOGITS(2, true) : FAT_LOGITS(2, false);
#undef FAT_LOGITS

        if (C::SEP_P) {  // S_t is in registers: the next S_t may be computed
          tc_fence_before();
          mbar_arrive(s_free + t);
        }
        float sub = 0.f;  // what the exponentials still subtract from x (FOLD)
        if (j == 0) {      // m_ref was 0
          m = mx;
          sub = (mx == -INFINITY) ? 0.f : mx;
        } else {
          const bool fresh = m == -INFINITY;  // no key of this row so far
          const bool need = fresh ? (mx != -INFINITY) : (mx > (FOLD ? 0.f : m) + 32.0f);
          if (C::SEP_P) {  // P_t and O_t are still read by PV_{j-1}
            ok = __all_sync(0xffffffffu, mbar_wait(o_ready + t, (j - 1) & 1, wd));
            if (!ok) break;
            tc_fence_after();
          }
          if (__any_sync(0xffffffffu, need)) {
            // O holds sum_{i<j} P_i V_i relative to the old max: rescale it once PV_{j-1} is done
            if (!C::SEP_P) {
              ok = __all_sync(0xffffffffu, mbar_wait(o_ready + t, (j - 1) & 1, wd));
              if (!ok) break;
              tc_fence_after();
            }
            const float f = need ? (fresh ? 0.f : ex2(FOLD ? -mx : m - mx)) : 1.0f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
              tmem_st32(tO + c * 32, o);
            }
            if (need) {
              l *= f;
              m = (fresh || !FOLD) ? mx : m + mx;
              sub = mx;
            }
          }
        }
        // turn order (d = 64, two tiles): tile 0 waits for tile 1's exponentials of the previous
        // key tile, tile 1 for tile 0's of this one. Only the order of work depends on it, so the
        // wait gives up quietly after a bounded time.
        const bool turns = C::SEP_P && ntile == 2;
        if (turns && (t == 0 ? (j >= 1 && j - 1 < nk_other) : (j < nk_other))) {
          (void)mbar_wait_hint(turn + t, static_cast<uint32_t>((t == 0 ? j - 1 : j) & 1), kTurnNs);
          __syncwarp();
        }
        uint64_t sum2[4];  // four short dependency chains
#pragma unroll
        for (int k = 0; k < 4; ++k) sum2[k] = f2_pack(0.f, 0.f);
        if (!FOLD) {  // x is absolute: subtract the row max
          const float m_use = (m == -INFINITY) ? 0.f : m;
          fwd_exp_pass<true>(x, f2_pack(m_use, m_use), tP, sum2);
        } else if (__any_sync(0xffffffffu, sub != 0.f)) {
          fwd_exp_pass<true>(x, f2_pack(sub, sub), tP, sum2);
        } else {
          fwd_exp_pass<false>(x, 0, tP, sum2);
        }
        if (turns && lane == 0) mbar_arrive(turn + (1 - t));
        {
          float s0, s1, s2, s3;
          f2_unpack(f2_add(sum2[0], sum2[2]), s0, s1);
          f2_unpack(f2_add(sum2[1], sum2[3]), s2, s3);
          l += (s0 + s1) + (s2 + s3);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_ready + t);
      }
      grid_dep_launch();  // a dependent grid (the backward preprocessing) may be scheduled
      if (nk == 0) {  // this tile sees no key (in this key range): empty rows, TMEM untouched
        fwd_write_empty_rows<D, TAIL>(p, seq_start, qs, min(L - qs, 128), h, split, q0, r, 128);
      } else {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_ready + t, (nk - 1) & 1, wd));
        if (ok) {
          tc_fence_after();
          const float inv_l = l > 0.f ? 1.0f / l : 0.f;
          const bool valid = qrow < L;
          const float m_use = (m == -INFINITY) ? 0.f : m;
          const float lse_row = l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
          if (!TAIL && p.kv_splits == 1) {
            __nv_bfloat16 *orow = p.out + ((size_t)(seq_start + qrow) * H + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l,
                                    __uint_as_float(o[2 * i + 1]) * inv_l);
              if (valid) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                  dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
              }
            }
            if (valid && p.lse != nullptr) p.lse[(size_t)h * T + seq_start + qrow] = lse_row;
          } else {  // partial result of this key range, normalised, in fp32
            const size_t trow = (size_t)blockIdx.x * 256 + (qrow - q0);
            float *orow = TAIL ? p.tail_o + trow * D
                               : p.o_part + (((size_t)split * T + seq_start + qrow) * H + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              if (valid) {
                float4 *dst = reinterpret_cast<float4 *>(orow + c * 32);
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4)
                  dst[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv_l,
                                        __uint_as_float(o[4 * v4 + 1]) * inv_l,
                                        __uint_as_float(o[4 * v4 + 2]) * inv_l,
                                        __uint_as_float(o[4 * v4 + 3]) * inv_l);
              }
            }
            if (valid) {
              if (TAIL)
                p.tail_lse[trow] = lse_row;
              else
                p.lse_part[((size_t)split * H + h) * T + seq_start + qrow] = lse_row;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// Persistent one-tile forward (d = 64, documents of at most kFwdOneTileMaxRows rows, whole key
// ranges). Short documents give each CTA of the one-tile grid only a few key-tile steps, so its
// fixed costs (barriers, TMEM allocation, bias table, the first loads, the epilogue and the
// block's own launch) weigh as much as its steps. Here two CTAs per SM walk all items (document,
// head, 128-row block) in turn with the roles of the one-tile CTA: the producer loads the next
// item's Q and K/V tiles while the softmax warpgroup writes the current item's rows, the MMA
// issuer computes the next item's first S as soon as the current one's last S has been read,
// and the bias table is rebuilt only when the head changes. Item ranks r = a (n H) + doc H + h
// with block qb = blocks(doc) - 1 - a (longest rows first when causal); documents of different
// lengths walk them longest-first (lpt_order), else in alternating rounds over the ranks.

// One item of the persistent forward.
struct FwdItem {
  int h, seq_start, L, seq_start_k, Lk, shift, q0;
  int nkv;       // key tiles its rows see (0: rows without keys)
  int kt0, kdir;  // stream position j holds key tile kt0 + kdir j
};

// Bucket of block group g = a * nseq + doc for lpt_order: 64 - the key tiles its rows see
// (1..64; more first), 63 for rows without keys, 64 when the document has no block a.
struct FwdLptBucket {
  const FwdParams &p;
  __device__ int operator()(int g) const {
    const int nseq = p.seq.num_seqs;
    const int a = g / nseq, doc = g - a * nseq;
    const DocSpan sp = doc_span(p.seq, doc);
    if (!sp.ok) return 64;
    const int nblk = (sp.lq + 127) >> 7;
    if (a >= nblk) return 64;
    const int q0 = (nblk - 1 - a) * 128;
    const int nkv_all = (sp.lk + 127) >> 7;
    int nkv = nkv_all;
    if (p.causal) {
      const int last = min(sp.lq, q0 + 128) - 1 + sp.shift;
      nkv = last < 0 ? 0 : min((last >> 7) + 1, nkv_all);
    }
    return nkv > 0 ? 64 - min(nkv, 64) : 63;
  }
};

// Every head's slope and table column fit the staging area (H + nb H floats).
constexpr int kFwdHeadStage = 2304;
__host__ __device__ inline bool fwd_pers_stages_heads(const BiasParams &b, int H) {
  return b.has_bias && H + (b.table ? b.nb * H : 0) <= kFwdHeadStage;
}
size_t fwd_pers_smem_bytes(const BiasParams &b, int H) {
  return fwd_smem_bytes(64, b.lut_len, 1) + (((size_t)b.lut_len + 15) & ~(size_t)15) +
         kLptRounds * 4 + (fwd_pers_stages_heads(b, H) ? (size_t)kFwdHeadStage * 4 : 0);
}

template <int D>
__global__ void __launch_bounds__(FwdCfg<D, 1>::NTHREADS, FwdCfg<D, 1>::MIN_BLOCKS)
    fat_fwd_pers_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D, 1>;
  static_assert(C::SEP_P, "one-tile CTAs keep P in its own TMEM columns");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.seq.total_tokens, H = p.seq.num_heads, nseq = p.seq.num_seqs;
  const int nqb = (p.seq.max_seqlen + 127) >> 7;
  const long long n_dh = (long long)H * nseq;
  const long long n_virtual = (long long)nqb * n_dh;

  uint8_t *sQ = sm + C::OFF_Q, *sK = sm + C::OFF_K, *sV = sm + C::OFF_V;
  float *lut = reinterpret_cast<float *>(sm + C::OFF_LUT);
  int *thr_s = reinterpret_cast<int *>(sm + C::OFF_LUT + ((p.bias.lut_len * 4 + 15) & ~15));
  float *col_s = reinterpret_cast<float *>(thr_s + kMaxThresholds);
  uint8_t *lbk = reinterpret_cast<uint8_t *>(col_s + 256);  // bucket of each delta
  int *lpt_list = reinterpret_cast<int *>(lbk + ((p.bias.lut_len + 15) & ~15));
  // every head's slope and table column, staged once when they fit (fwd_pers_stages_heads), so
  // that a change of head between items reads shared memory only
  float *heads_s = reinterpret_cast<float *>(lpt_list + kLptRounds);
  const bool staged_heads = fwd_pers_stages_heads(p.bias, H);

  // corrupt or out-of-bound cu_seqlens entries, reported once (their items are skipped)
  if (blockIdx.x == 0) {
    for (int i = tid; i < nseq; i += blockDim.x) {
      const DocSpan sp = doc_span(p.seq, i);
      if (!sp.ok || sp.lq > p.seq.max_seqlen || sp.lk > p.seq.max_seqlen_k)
        atomicOr(p.err, FAT_DEVERR_SEQLENS);
    }
  }
  // this CTA's ranks, longest first (the K/V ring is the scratch: nothing is loaded yet)
  static_assert(2 * C::NS * C::TILE >= lpt_scratch_bytes(C::NTHREADS), "ordering scratch");
  const int lpt_n = p.lpt ? lpt_order(nqb * nseq, nseq, H, kLptRounds, FwdLptBucket{p}, sK,
                                      lpt_list)
                          : -1;
  // the item of round v (advanced past items without rows); false when the walk is done
  auto next_item = [&](long long &v, FwdItem &it) -> bool {
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
      const int a = (int)(rank / n_dh);
      const long long rest = rank - (long long)a * n_dh;
      const int doc = (int)(rest / H);
      const DocSpan sp = doc_span(p.seq, doc);
      if (!sp.ok) continue;
      const int nblk = (sp.lq + 127) >> 7;
      if (a >= nblk) continue;
      it.h = (int)(rest - (long long)doc * H);
      it.seq_start = sp.sq;
      it.L = sp.lq;
      it.seq_start_k = sp.sk;
      it.Lk = sp.lk;
      it.shift = sp.shift;
      it.q0 = (nblk - 1 - a) * 128;
      const int nkv_all = (sp.lk + 127) >> 7;
      int nkv = nkv_all;
      if (p.causal) {
        const int last = min(sp.lq, it.q0 + 128) - 1 + sp.shift;
        nkv = last < 0 ? 0 : min((last >> 7) + 1, nkv_all);
      }
      it.nkv = nkv;
      // causal rows take their key tiles from the diagonal backwards (the largest ALiBi bias
      // first, so the running max rarely grows afterwards)
      it.kt0 = p.causal ? nkv - 1 : 0;
      it.kdir = p.causal ? -1 : 1;
      return true;
    }
  };
  long long v_first = 0;
  FwdItem first;
  if (!next_item(v_first, first)) return;  // nothing to do: before any barrier or allocation

  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *q_empty = q_full + 1;   // the item's S products have read Q
  uint64_t *k_full = q_empty + 1;   // [NS]
  uint64_t *v_full = k_full + C::NS;
  uint64_t *k_empty = v_full + C::NS;
  uint64_t *v_empty = k_empty + C::NS;
  uint64_t *s_full = v_empty + C::NS;
  uint64_t *p_ready = s_full + 1;
  uint64_t *o_ready = p_ready + 1;
  uint64_t *s_free = o_ready + 1;   // S has been read into registers
  uint64_t *o_free = s_free + 1;    // the item's O has been read out of TMEM
  uint64_t *mma_done = o_free + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  static_assert((2 + 4 * C::NS + 6) * 8 + 8 <= 256, "barrier block");

  if (warp == C::WARP_PROD && lane == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(k_empty + s, 1);
      mbar_init(v_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_ready, 128);
    mbar_init(o_ready, 1);
    mbar_init(s_free, 128);
    mbar_init(o_free, 128);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  // bias: thresholds and the first head's table column staged, the bucket of every delta kept
  // (head-independent), the first head's table built
  const bool has_table = p.bias.table != nullptr, has_slopes = p.bias.slopes != nullptr;
  FarBias *fbs = reinterpret_cast<FarBias *>(sm + C::OFF_WD + 32);
  bias_stage(p.bias, first.h, H, thr_s, col_s, tid, C::NTHREADS);
  if (staged_heads) {  // slopes [H], then the columns [H][nb] (table rows are [nb][H])
    if (has_slopes)
      for (int i = tid; i < H; i += C::NTHREADS) heads_s[i] = __ldg(p.bias.slopes + i);
    if (has_table)
      for (int i = tid; i < p.bias.nb * H; i += C::NTHREADS)
        heads_s[H + (i % H) * p.bias.nb + i / H] = __ldg(p.bias.table + i);
  }
  __syncthreads();
  {
    const float slope = has_slopes ? __ldg(p.bias.slopes + first.h) : 0.f;
    for (int i = tid; i < p.bias.lut_len; i += C::NTHREADS) {
      const int delta = p.bias.lut_lo + i;
      const int bk = has_table ? t5_bucket_staged(delta, p.bias, thr_s) : 0;
      lbk[i] = static_cast<uint8_t>(bk);
      lut[i] = bias_log2_staged(bk, delta, slope, p.bias, col_s);
    }
    if (tid == 0) {
      *reinterpret_cast<Watchdog *>(sm + C::OFF_WD) =
          Watchdog{abort_flag, p.err, FAT_DEVERR_TIMEOUT_FWD, p.timeout_ns};
      *fbs = far_bias_staged(p.bias, thr_s, col_s, slope);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watchdog &wd = *reinterpret_cast<const Watchdog *>(sm + C::OFF_WD);

  if (warp >= C::WARP_PROD) regs_dec<C::REG_OTHER>();

  if (warp == C::WARP_PROD) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int last_k[C::NS], last_v[C::NS];
#pragma unroll
      for (int s = 0; s < C::NS; ++s) last_k[s] = last_v[s] = -1;
      int ni = 0;       // items with keys so far (the phases of q_full / q_empty)
      int last_q = -1;  // phase of the last Q copy issued
      long long J = 0;  // K/V stream position
      bool ok = !(p.debug_flags & 1);  // test hook: no copies, the consumers' waits run out
      long long v = v_first;
      FwdItem it = first;
      if (ok) do {
        if (it.nkv == 0) continue;
        if (ni > 0 && !mbar_wait(q_empty, (ni - 1) & 1, wd)) { ok = false; break; }
        mbar_arrive_expect_tx(q_full, C::TILE);
        tma_load_3d(&tm_q, q_full, sQ, 0, it.h, it.seq_start + it.q0);
        last_q = ni;
        const int hk = it.h / p.seq.group;
        for (int j = 0; ok && j < it.nkv; ++j) {
          const long long g = J + j;
          const int s = (int)(g % C::NS), u = (int)(g / C::NS);
          const int krow = it.seq_start_k + 128 * (it.kt0 + it.kdir * j);
          if (u > 0 && !mbar_wait(k_empty + s, (u - 1) & 1, wd)) { ok = false; break; }
          mbar_arrive_expect_tx(k_full + s, C::TILE);
          tma_load_3d(&tm_k, k_full + s, sK + s * C::TILE, 0, hk, krow);
#pragma unroll
          for (int x = 0; x < C::NS; ++x)
            if (x == s) last_k[x] = u;
          if (u > 0 && !mbar_wait(v_empty + s, (u - 1) & 1, wd)) { ok = false; break; }
          mbar_arrive_expect_tx(v_full + s, C::TILE);
          tma_load_3d(&tm_v, v_full + s, sV + s * C::TILE, 0, hk, krow);
#pragma unroll
          for (int x = 0; x < C::NS; ++x)
            if (x == s) last_v[x] = u;
        }
        if (!ok) break;
        J += it.nkv;
        ++ni;
      } while (++v, next_item(v, it));
      // teardown: every copy this thread issued has landed before the CTA exits
      if (last_q >= 0) mbar_wait_teardown(q_full, last_q & 1, kTeardownNs);
#pragma unroll
      for (int s = 0; s < C::NS; ++s) {
        if (last_k[s] >= 0) mbar_wait_teardown(k_full + s, last_k[s] & 1, kTeardownNs);
        if (last_v[s] >= 0) mbar_wait_teardown(v_full + s, last_v[s] & 1, kTeardownNs);
      }
      (void)ok;
    }
  } else if (warp == C::WARP_MMA) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t dS = tmem + C::COL_S0, dO = tmem + C::COL_O0, aP = tmem + C::COL_P0;
      const uint64_t dQd = sw128_desc(smem_u32(sQ), 16, 1024);
      const uint64_t dKd = sw128_desc(smem_u32(sK), 16, 1024);
      const uint64_t dVd = sw128_desc(smem_u32(sV), C::BLK, 1024);
      auto issue_S = [&](int st) {
        const uint64_t kd = dKd + ((st * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::BLK + (kk & 3) * 32) >> 4;
          mma_bf16_ss(dS, dQd + off, kd + off, C::IDESC_S, kk > 0);
        }
      };
      auto issue_PV = [&](int st, bool acc) {
        const uint64_t vd = dVd + ((st * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(dO, aP + kk * 8, vd + ((kk * 2048) >> 4), C::IDESC_PV,
                      (acc || kk > 0) ? 1u : 0u);
      };
      int ni = 0;
      long long J = 0, GS = 0;  // K/V stream position, steps so far
      bool ok = true;
      long long v = v_first;
      FwdItem it = first;
      do {
        if (it.nkv == 0) continue;
        const int s0 = (int)(J % C::NS), u0 = (int)(J / C::NS);
        // S is free: the softmax has read the previous step's S (waited for below, in order)
        if (!mbar_wait(q_full, ni & 1, wd) || !mbar_wait(k_full + s0, u0 & 1, wd)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_S(s0);
        mma_commit(s_full);
        mma_commit(k_empty + s0);
        if (it.nkv == 1) mma_commit(q_empty);
        for (int jl = 0; jl < it.nkv; ++jl) {
          const long long g = GS + jl, j = J + jl;
          const int s = (int)(j % C::NS), u = (int)(j / C::NS);
          // the next S once the softmax has read this one
          if (!mbar_wait(s_free, g & 1, wd)) { ok = false; break; }
          if (jl + 1 < it.nkv) {
            const int sn = (int)((j + 1) % C::NS), un = (int)((j + 1) / C::NS);
            if (!mbar_wait(k_full + sn, un & 1, wd)) { ok = false; break; }
            tc_fence_after();
            issue_S(sn);
            mma_commit(s_full);
            mma_commit(k_empty + sn);
            if (jl + 2 == it.nkv) mma_commit(q_empty);  // the item's last S reads Q
          }
          if (!mbar_wait(v_full + s, u & 1, wd) || !mbar_wait(p_ready, g & 1, wd)) {
            ok = false;
            break;
          }
          // the first P V overwrites O: the previous item's rows have been read out
          if (jl == 0 && ni > 0 && !mbar_wait(o_free, (ni - 1) & 1, wd)) { ok = false; break; }
          tc_fence_after();
          issue_PV(s, jl > 0);
          mma_commit(o_ready);
          mma_commit(v_empty + s);
        }
        if (!ok) break;
        GS += it.nkv;
        J += it.nkv;
        ++ni;
      } while (++v, next_item(v, it));
      (void)ok;
      mma_commit(mma_done);
      mbar_wait_teardown(mma_done, 0, kTeardownNs);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------------ softmax warpgroup
    regs_inc<C::REG_SM>();
    const int r = tid & 127;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::COL_S0;
    const uint32_t tO = tmem + lane_off + C::COL_O0;
    const uint32_t tP = tmem + lane_off + C::COL_P0;
    int cur_h = first.h;
    long long GS = 0;  // steps so far (the phases of s_full, s_free, p_ready, o_ready)
    int ni = 0;        // items with keys so far (the phases of o_free)
    bool ok = true;
    long long v = v_first;
    FwdItem it = first;
    do {
      if (it.h != cur_h && p.bias.has_bias) {
        // the next head's table column and bias table (only these 128 threads read them)
        named_bar_sync(1, 128);
        float slope;
        const float *col;
        if (staged_heads) {
          slope = has_slopes ? heads_s[it.h] : 0.f;
          col = heads_s + H + it.h * p.bias.nb;
        } else {
          slope = has_slopes ? __ldg(p.bias.slopes + it.h) : 0.f;
          if (has_table)
            for (int i = r; i < p.bias.nb; i += 128)
              col_s[i] = __ldg(p.bias.table + (size_t)i * H + it.h);
          named_bar_sync(1, 128);
          col = col_s;
        }
        for (int i = r; i < p.bias.lut_len; i += 128) {
          const int delta = p.bias.lut_lo + i;
          lut[i] = bias_log2_staged(lbk[i], delta, slope, p.bias, col);
        }
        if (r == 0) *fbs = far_bias_staged(p.bias, thr_s, col, slope);
        named_bar_sync(1, 128);
      }
      cur_h = it.h;
      const int qrow = it.q0 + r;
      if (it.nkv == 0) {  // no key for any row of the block: empty rows, TMEM untouched
        fwd_write_empty_rows<D, false>(p, it.seq_start, it.q0, min(it.L - it.q0, 128), it.h, 0,
                                       it.q0, r, 128);
        continue;
      }
      const FarBias fb = *fbs;
      float m = -INFINITY, l = 0.f;
      for (int jl = 0; jl < it.nkv; ++jl) {
        const long long g = GS + jl;
        ok = __all_sync(0xffffffffu, mbar_wait(s_full, g & 1, wd));
        if (!ok) break;
        tc_fence_after();
        const int ks = 128 * (it.kt0 + it.kdir * jl);
        const int d0 = ks - it.q0 - it.shift;  // delta of (row 0, key 0) of the tile
        const bool need_mask = (ks + 128 > it.Lk) || (p.causal && d0 + 127 > 0);
        const int lim = min(it.Lk - ks, p.causal ? (qrow + it.shift - ks + 1) : 128);
        int mode;
        float rowc = 0.f, kk = 0.f;
        if (!p.bias.has_bias) {
          mode = 0;
        } else if (d0 - 127 >= p.bias.sat_pos) {
          kk = fb.k_pos;
          rowc = fmaf(fb.k_pos, (float)(d0 - r), fb.c_pos);
          mode = has_slopes ? 1 : 0;
        } else if (d0 + 127 <= -p.bias.sat_neg) {
          kk = fb.k_neg;
          rowc = fmaf(fb.k_neg, (float)(d0 - r), fb.c_neg);
          mode = has_slopes ? 1 : 0;
        } else {
          mode = 2;
        }
        const float *lut_row = lut + (d0 - r - p.bias.lut_lo);
        uint32_t x[4][32];
        float mx;  // row max of x
#define FAT_LOGITS(MODE, MASK) \
  fwd_logits<MODE, MASK, false>(tS, x, p.scale_log2, rowc, kk, lut_row, lim, 0)
        if (mode == 0)
          mx = need_mask ? FAT_LOGITS(0, true) : FAT_LOGITS(0, false);
        else if (mode == 1)
          mx = need_mask ? FAT_LOGITS(1, true) : FAT_LOGITS(1, false);
        else
          mx = need_mask ? FAT_LOGITS(2, true) : FAT_LOGITS(2, false);
#undef FAT_LOGITS
        tc_fence_before();
        mbar_arrive(s_free);  // S is in registers: the next S may be computed
        if (jl == 0) {
          m = mx;
        } else {
          // P and O are still read by the previous step's P V
          ok = __all_sync(0xffffffffu, mbar_wait(o_ready, (g - 1) & 1, wd));
          if (!ok) break;
          tc_fence_after();
          const bool fresh = m == -INFINITY;  // no key of this row so far
          const bool need = fresh ? (mx != -INFINITY) : (mx > m + 32.0f);
          if (__any_sync(0xffffffffu, need)) {
            // O holds sum_{i<j} P_i V_i relative to the old max: rescaled once
            const float f = need ? (fresh ? 0.f : ex2(m - mx)) : 1.0f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
              tmem_st32(tO + c * 32, o);
            }
            if (need) {
              l *= f;
              m = mx;
            }
          }
        }
        uint64_t sum2[4];  // four short dependency chains
#pragma unroll
        for (int k = 0; k < 4; ++k) sum2[k] = f2_pack(0.f, 0.f);
        {
          const float m_use = (m == -INFINITY) ? 0.f : m;
          fwd_exp_pass<true>(x, f2_pack(m_use, m_use), tP, sum2);
        }
        {
          float s0, s1, s2, s3;
          f2_unpack(f2_add(sum2[0], sum2[2]), s0, s1);
          f2_unpack(f2_add(sum2[1], sum2[3]), s2, s3);
          l += (s0 + s1) + (s2 + s3);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_ready);
      }
      if (!ok) break;
      // the item's rows: O / l and lse once its last P V is done; then O is free for the next
      const long long g_last = GS + it.nkv - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(o_ready, g_last & 1, wd));
      if (!ok) break;
      tc_fence_after();
      {
        const float inv_l = l > 0.f ? 1.0f / l : 0.f;
        const bool valid = qrow < it.L;
        const float m_use = (m == -INFINITY) ? 0.f : m;
        const float lse_row = l > 0.f ? (m_use + __log2f(l)) * kLn2 : -INFINITY;
        __nv_bfloat16 *orow = p.out + ((size_t)(it.seq_start + qrow) * H + it.h) * D;
        uint32_t o[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32_issue(tO + c * 32, o[c]);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32_fence(o[c]);
        tc_fence_before();
        mbar_arrive(o_free);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[c][2 * i]) * inv_l,
                                __uint_as_float(o[c][2 * i + 1]) * inv_l);
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        if (valid && p.lse != nullptr) p.lse[(size_t)it.h * T + it.seq_start + qrow] = lse_row;
      }
      GS += it.nkv;
      ++ni;
    } while (++v, next_item(v, it));
    (void)ni;
    grid_dep_launch();  // a dependent grid (the backward preprocessing) may be scheduled
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// One output row merged from S <= 64 normalised partial rows o_s with their (natural) lse l_s
// by one warp: lse = log sum_s exp(l_s), out = sum_s exp(l_s - lse) o_s; a row with no key in
// any range gets out 0, lse -inf. Lane s loads l_s and l_{s+32} (all S loads in flight at once),
// the maximum and the weights' sum are warp reductions, and the partial rows are read four
// splits at a time with each weight broadcast from its lane. Writes out (bf16, this lane's
// D / 32 channels) and, from lane 0, lse when lse_out is not null.
template <int D>
__device__ __forceinline__ void merge_partial_rows(const float *lse_p, size_t lse_stride,
                                                   const float *o_p, size_t o_stride, int S,
                                                   int lane, __nv_bfloat16 *orow, float *lse_out) {
  constexpr int CPL = D / 32;
  const float l0 = lane < S ? lse_p[(size_t)lane * lse_stride] : -INFINITY;
  const float l1 = lane + 32 < S ? lse_p[(size_t)(lane + 32) * lse_stride] : -INFINITY;
  float m = fmaxf(l0, l1);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const float w0 = (m == -INFINITY || l0 == -INFINITY) ? 0.f : __expf(l0 - m);
  const float w1 = (m == -INFINITY || l1 == -INFINITY) ? 0.f : __expf(l1 - m);
  float wsum = w0 + w1;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  float acc[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) acc[i] = 0.f;
  const float *o = o_p + lane * CPL;
#pragma unroll 4
  for (int sp = 0; sp < S; ++sp) {
    const float wgt = __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31);
    if (wgt == 0.f) continue;  // the same for every lane
    const float *os = o + (size_t)sp * o_stride;
    if constexpr (CPL == 2) {
      const float2 v = *reinterpret_cast<const float2 *>(os);
      acc[0] += wgt * v.x;
      acc[1] += wgt * v.y;
    } else {
      const float4 v = *reinterpret_cast<const float4 *>(os);
      acc[0] += wgt * v.x;
      acc[1] += wgt * v.y;
      acc[2] += wgt * v.z;
      acc[3] += wgt * v.w;
    }
  }
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  __nv_bfloat16 *dst = orow + lane * CPL;
  if constexpr (CPL == 2) {
    *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  } else {
    uint2 v;
    v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2 *>(dst) = v;
  }
  if (lane == 0 && lse_out != nullptr) *lse_out = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
}

// Merge of a split last wave: one warp per (split CTA row), the tail_splits partial rows (each
// normalised, with its lse) combined as in the split-key merge below, written to out and lse.
// Documents have equal length (the condition of the split), so row q of document doc is token
// doc * max_seqlen + q.
template <int D>
__global__ void __launch_bounds__(256) fat_fwd_tail_combine_kernel(const FwdParams p) {
  const int T = p.seq.total_tokens, H = p.seq.num_heads, S = p.tail_splits;
  const int L = p.seq.max_seqlen;
  const int lane = threadIdx.x & 31;
  const long long nrows = (long long)p.tail_ntail * 256;
  const long long w0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long rw = w0; rw < nrows; rw += nw) {
    const long long c = rw / 256;
    const int row = (int)(rw % 256);
    const long long cta = p.tail_first + c;
    const int h = (int)((cta / p.tail_gx) % H);
    const long long doc = cta / ((long long)p.tail_gx * H);
    const int q = (p.tail_gx - 1 - (int)(cta % p.tail_gx)) * 256 + row;
    if (q >= L) continue;
    const long long tok = doc * L + q;
    merge_partial_rows<D>(p.tail_lse + (size_t)c * S * 256 + row, 256,
                          p.tail_o + ((size_t)c * S * 256 + row) * D, (size_t)256 * D, S, lane,
                          p.out + ((size_t)tok * H + h) * D,
                          p.lse != nullptr ? p.lse + (size_t)h * T + tok : nullptr);
  }
}

template <int D, int NT>
int launch_fwd_t(const FwdParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                 const CUtensorMap &mv, cudaStream_t stream) {
  using C = FwdCfg<D, NT>;
  const size_t smem = fwd_smem_bytes(D, p.bias.lut_len, NT);
  const dim3 grid = (NT == 1 && p.flat)
                        ? dim3((unsigned)(p.seq.total_tokens / 128 + p.seq.num_seqs),
                               p.seq.num_heads, 1)
                        : dim3((p.seq.max_seqlen + C::ROWS - 1) / C::ROWS, p.seq.num_heads,
                               p.seq.num_seqs * p.kv_splits);
  // the register re-balancing needs the launch pool the split was designed for
  cudaError_t e = (cudaError_t)prepare_kernel((const void *)fat_fwd_kernel<D, false, NT>, smem,
                                              C::NTHREADS, C::REGS_NEEDED);
  if (e != cudaSuccess) return (int)e;  // reason recorded by prepare_kernel
  fat_fwd_kernel<D, false, NT><<<grid, C::NTHREADS, smem, stream>>>(mq, mk, mv, p);
  e = cudaGetLastError();
  const long long tail_ctas = (long long)p.tail_ntail * p.tail_splits;
  if constexpr (NT == 2) {
  if (e == cudaSuccess && p.tail_splits > 0 && tail_ctas > 0) {
    // the split last wave, then its merge (ordered by the stream)
    e = (cudaError_t)prepare_kernel((const void *)fat_fwd_kernel<D, true, NT>, smem,
                                    C::NTHREADS, C::REGS_NEEDED);
    if (e != cudaSuccess) return (int)e;
    fat_fwd_kernel<D, true, NT><<<(unsigned)tail_ctas, C::NTHREADS, smem, stream>>>(
        mq, mk, mv, p);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
      const int blocks = (int)std::min<long long>(((long long)p.tail_ntail * 256 + 7) / 8,
                                                  152LL * 8);
      fat_fwd_tail_combine_kernel<D><<<blocks, 256, 0, stream>>>(p);
      e = cudaGetLastError();
    }
  }
  }
  if (e != cudaSuccess) {
    cudaFuncAttributes fa{};
    cudaFuncGetAttributes(&fa, fat_fwd_kernel<D, false, NT>);
    char msg[160];
    snprintf(msg, sizeof msg, "%s [regs %d, max threads %d, local %zu B, dyn smem %zu B]",
             cudaGetErrorString(e), fa.numRegs, fa.maxThreadsPerBlock, (size_t)fa.localSizeBytes,
             smem);
    set_last_error("kernel launch", (int)e, msg);
  }
  return (int)e;
}

// Persistent one-tile forward: as many CTAs as fit at once (two per SM unless the bias table
// makes them too large), at most one per item. Shared memory beyond the one-tile CTA's: the
// bucket of each delta, the CTA's item list and, when they fit, every head's bias constants.
int launch_fwd_pers(const FwdParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                    const CUtensorMap &mv, cudaStream_t stream) {
  using C = FwdCfg<64, 1>;
  const size_t smem = fwd_pers_smem_bytes(p.bias, p.seq.num_heads);
  if (smem > (size_t)kSmemLimit) return (int)cudaErrorInvalidValue;
  const void *fn = (const void *)fat_fwd_pers_kernel<64>;
  cudaError_t e = (cudaError_t)prepare_kernel(fn, smem, C::NTHREADS, C::REGS_NEEDED);
  if (e != cudaSuccess) return (int)e;  // reason recorded by prepare_kernel
  // CTAs per SM: the launch bound's two unless shared memory holds fewer (1 KB per block is
  // reserved by the system)
  static std::mutex mu;
  static int smem_sm[64] = {0};
  int dev = 0, per_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lk(mu);
    if (smem_sm[dev] == 0) {
      // the largest shared-memory share of the SM, so that the CTAs counted here fit at once
      if (cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
          cudaDeviceGetAttribute(&smem_sm[dev], cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                 dev) != cudaSuccess) {
        (void)cudaGetLastError();
        smem_sm[dev] = 0;
      }
    }
    per_sm = smem_sm[dev];
  }
  const int bps = std::max(1, std::min<int>(C::MIN_BLOCKS, (int)(per_sm / (smem + 1024))));
  const int sms = sm_count();
  const long long nqb = (p.seq.max_seqlen + 127) / 128;
  const long long items = nqb * p.seq.num_heads * p.seq.num_seqs;
  if (items == 0) return 0;
  const long long grid = std::min<long long>(items, (long long)(sms > 0 ? sms : 1) * bps);
  FwdParams pp = p;
  // documents of different lengths: longest-first (with equal documents the rank order is)
  const bool unequal =
      (long long)p.seq.total_tokens != (long long)p.seq.num_seqs * p.seq.max_seqlen ||
      (long long)p.seq.total_k != (long long)p.seq.num_seqs * p.seq.max_seqlen_k;
  pp.lpt = (unequal && nqb * p.seq.num_seqs <= kLptGroups) ? 1 : 0;
  fat_fwd_pers_kernel<64><<<(unsigned)grid, C::NTHREADS, smem, stream>>>(mq, mk, mv, pp);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFuncAttributes fa{};
    cudaFuncGetAttributes(&fa, fat_fwd_pers_kernel<64>);
    char msg[160];
    snprintf(msg, sizeof msg, "%s [regs %d, max threads %d, local %zu B, dyn smem %zu B]",
             cudaGetErrorString(e), fa.numRegs, fa.maxThreadsPerBlock, (size_t)fa.localSizeBytes,
             smem);
    set_last_error("kernel launch", (int)e, msg);
  }
  return (int)e;
}

int fwd_tiles_per_cta(int head_dim, int max_seqlen) {
  return head_dim == 64 && max_seqlen <= kFwdOneTileMaxRows ? 1 : 2;
}

int launch_fwd(const FwdParams &p, int head_dim, const void *q, const void *k, const void *v,
               cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const int T = p.seq.total_tokens, H = p.seq.num_heads;
  const int Tk = p.seq.total_k, Hkv = p.seq.num_heads_kv;
  if (make_tmap_thd(&mq, q, T, H, head_dim, 128) || make_tmap_thd(&mk, k, Tk, Hkv, head_dim, 128) ||
      make_tmap_thd(&mv, v, Tk, Hkv, head_dim, 128))
    return (int)cudaErrorInvalidValue;
  if (head_dim == 128) return launch_fwd_t<128, 2>(p, mq, mk, mv, stream);
  // a split last wave is planned for two-tile CTAs
  if (p.tail_splits == 0 && fwd_tiles_per_cta(head_dim, p.seq.max_seqlen) == 1 &&
      p.kv_splits == 1 && !(p.debug_flags & 4)) {
    // Persistent CTAs once each resident CTA gets three items or more (at most T / 128 + n
    // blocks per head): with fewer, the grid of one-tile CTAs, two per SM, overlaps the fixed
    // costs as well and runs its steps with fewer registers spilled.
    const long long blocks = ((long long)p.seq.total_tokens / 128 + p.seq.num_seqs) *
                             p.seq.num_heads;
    if ((p.debug_flags & 8) || blocks >= 3LL * 2 * std::max(1, sm_count()))
      return launch_fwd_pers(p, mq, mk, mv, stream);
  }
  if (p.tail_splits == 0 && fwd_tiles_per_cta(head_dim, p.seq.max_seqlen) == 1) {
    FwdParams pf = p;
    // documents of different lengths: the flat grid, when it has fewer blocks
    const long long blocks_3d = (long long)((p.seq.max_seqlen + 127) / 128) * p.seq.num_seqs;
    const long long blocks_flat = (long long)p.seq.total_tokens / 128 + p.seq.num_seqs;
    pf.flat = p.kv_splits == 1 && p.seq.num_seqs > 1 && blocks_flat < blocks_3d;
    return launch_fwd_t<64, 1>(pf, mq, mk, mv, stream);
  }
  return launch_fwd_t<64, 2>(p, mq, mk, mv, stream);
}

// Merge of a split forward's partial results, one warp per (query row, head): with partial lse
// l_s and normalised partial outputs O_s, lse = log sum_s exp(l_s) and
// out = sum_s exp(l_s - lse) O_s (a row with no key in any range: out 0, lse -inf).
// Memory bound: each lane reads D/32 channels of every split's row.
template <int D>
__global__ void __launch_bounds__(256) fat_fwd_combine_kernel(const FwdParams p) {
  const int T = p.seq.total_tokens, H = p.seq.num_heads, S = p.kv_splits;
  const int lane = threadIdx.x & 31;
  const long long nrows = (long long)T * H;
  const long long w0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long rh = w0; rh < nrows; rh += nw) {
    const int t = (int)(rh / H), h = (int)(rh % H);
    merge_partial_rows<D>(p.lse_part + (size_t)h * T + t, (size_t)H * T,
                          p.o_part + ((size_t)t * H + h) * D, (size_t)T * H * D, S, lane,
                          p.out + ((size_t)t * H + h) * D,
                          p.lse != nullptr ? p.lse + (size_t)h * T + t : nullptr);
  }
}

int launch_fwd_combine(const FwdParams &p, int head_dim, cudaStream_t stream) {
  const long long nrows = (long long)p.seq.total_tokens * p.seq.num_heads;
  if (nrows == 0) return 0;
  const int blocks = (int)std::min<long long>((nrows + 7) / 8, 152LL * 8);
  if (head_dim == 64)
    fat_fwd_combine_kernel<64><<<blocks, 256, 0, stream>>>(p);
  else
    fat_fwd_combine_kernel<128><<<blocks, 256, 0, stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) set_last_error("split forward combine launch", (int)e, cudaGetErrorString(e));
  return (int)e;
}

}  // namespace fat
