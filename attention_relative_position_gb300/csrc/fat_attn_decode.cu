// fat_attn_decode.cu -- forward of documents with few query rows per key/value head: a decode
// step (one new query per document over its key cache, FAT5 report, "Motivation" and "La suite"
// sections: T5 decoder at inference), a short chunk of queries, or very short documents, with
// the query heads of a group sharing their key/value head. Same result as the tiled forward:
// per row, softmax(scale * q K^T + bias) V over the row's visible keys, with the bias (T5
// bucket table, ALiBi) and the bottom-right causal mask built in the kernel.
//
// The work is a read of the key/value cache with a handful of rows to apply it to, so the
// kernel is built around the HBM read, not the tensor cores (a 128-row MMA tile would be
// 94-99% padding):
//   one CTA = (key split, key/value head, document); its rows are every query of the document
//   times every query head of the group (R <= 8 rows).
//   warp 4      TMA producer: 32-key tiles of K and V (128-byte swizzle) through a 96 KB ring.
//   warps 0-3   consumers; warp w takes ring stages w, w + 4, ... and keeps its own running
//               max, sum and output rows. Scores: lane i owns key i of the stage and forms its
//               dot product with every row (query rows in shared memory, read as broadcasts,
//               packed fp32x2 FMAs), adds the bias (bucket lookup table over the near deltas,
//               the saturated bucket beyond them, ALiBi slope * |delta|), masks, and the row's
//               max over the warp is one shuffle reduction. P V: lane i owns D/32 channels and
//               walks the stage's keys with the probabilities broadcast from shared memory.
//   merge       the four warps' states are combined in shared memory (over the drained ring);
//               the CTA writes out (bf16) and lse, or, with key splits, the normalised partial
//               output and partial lse the split combine pass merges.
// Two CTAs fit on an SM (100-111 KB of shared memory each), so up to 12 (d 128) or 24 (d 64)
// tiles per SM are in flight.
#include <algorithm>
#include <cstdio>

#include "fat_attn_internal.cuh"

namespace fat {
namespace {

constexpr int kDecKT = 32;                 // keys per ring stage (one per lane)
constexpr int kDecWarps = 4;               // consumer warps
constexpr int kDecThreads = (kDecWarps + 1) * 32;
constexpr int kDecRingBytes = 96 * 1024;
constexpr int kDecMaxLut = 16384;          // near deltas with a bucket lookup entry

template <int D, int R>
struct DecCfg {
  static constexpr int BOXES = D / 64;                  // 64-channel TMA boxes per tile
  static constexpr int BOX = kDecKT * 128;              // bytes: 32 rows x 64 bf16
  static constexpr int TILE = BOXES * BOX;              // one K or V tile
  static constexpr int STAGE = 2 * TILE;
  static constexpr int NS = kDecRingBytes / STAGE;      // 6 (d 128) or 12 (d 64)
  static constexpr int OFF_Q = NS * STAGE;              // rows * scale * log2(e), fp32 [R][D]
  static constexpr int OFF_P = OFF_Q + R * D * 4;       // per warp: (p, p) pairs [32][R]
  static constexpr int OFF_BAR = OFF_P + kDecWarps * 32 * R * 8;  // full[NS], empty[NS]
  static constexpr int OFF_TAG = OFF_BAR + 2 * NS * 8;   // stage held by each slot, int [NS]
  static constexpr int OFF_MISC = OFF_TAG + ((NS * 4 + 15) & ~15);  // abort flag, watchdog
  static constexpr int OFF_TAB = OFF_MISC + 64;          // bias table rows, then bucket lut
  static constexpr int MERGE = kDecWarps * R * (D + 2) * 4;
  static_assert(MERGE <= NS * STAGE, "the merge area lives in the drained ring");
  static_assert(NS >= 2, "ring");
};

// Shared-memory tail of the layout: the T5 table entries of the group's heads (fp32, log2
// units, [G][nb]) and the bucket of every near delta (uint8, deltas -sat_neg + 1 ..
// sat_pos - 1).
struct DecTail {
  int tab, lut, total;
};
__host__ __device__ inline DecTail dec_tail(int base, int G, int nb, int lutn) {
  DecTail t;
  t.tab = base;
  t.lut = base + ((G * nb * 4 + 15) & ~15);
  t.total = t.lut + ((lutn + 15) & ~15);
  return t;
}

__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t x) {
  return f2_pack(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}
__device__ __forceinline__ float dec_warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float dec_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Wait until ring slot `tag` has been handed to stage `want` (bounded like mbar_wait). A slot is
// used by different consumer warps in turn, so a warp may ask for stage i + NS while the slot's
// barrier is still in the phase of stage i; a parity wait alone would then succeed on the older
// phase. Once the tag shows stage `want`, the slot's previous phase has completed and the parity
// names `want`'s phase unambiguously.
__device__ __forceinline__ bool wait_slot_tag(const volatile int *tag, int want,
                                              const Watchdog &wd) {
  if (*tag == want) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t spins = 1;; ++spins) {
    __nanosleep(64);
    if (*tag == want) return true;
    if ((spins & 63u) == 0) {
      if (*wd.abort_flag) return false;
      if ((long long)(global_timer_ns() - t0) > wd.timeout_ns) {
        *wd.abort_flag = 1;
        atomicOr(wd.err_word, wd.err_bit);
        return false;
      }
    }
  }
}

template <int D, int R>
__global__ void __launch_bounds__(kDecThreads, 2)
    fat_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __nv_bfloat16 *__restrict__ qg,
                      const FwdParams p) {
  using C = DecCfg<D, R>;
  constexpr int CPL = D / 32;  // output channels per lane
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, hk = blockIdx.y, doc = blockIdx.z;
  const int T = p.seq.total_tokens, H = p.seq.num_heads, G = p.seq.group;

  const DocSpan span = doc_span(p.seq, doc);
  if (!span.ok) {
    if (tid == 0 && split == 0 && hk == 0) atomicOr(p.err, FAT_DEVERR_SEQLENS);
    return;
  }
  if ((span.lq > p.seq.max_seqlen || span.lk > p.seq.max_seqlen_k) && tid == 0 && split == 0 &&
      hk == 0)
    atomicOr(p.err, FAT_DEVERR_SEQLENS);
  if (span.lq == 0) return;
  const int nrows = min(span.lq * G, R);  // row r = query (r / G) of head hk * G + r % G
  // this split's keys [kbeg, kend) (document-local); none: the rows get empty partials
  const long long ksplit = (long long)split * p.split_tiles * 128;
  const int kbeg = (int)min(ksplit, (long long)span.lk);
  const int kend = (int)min(ksplit + (long long)p.split_tiles * 128, (long long)span.lk);
  const int nst = (kend - kbeg + kDecKT - 1) / kDecKT;

  float *q_s = reinterpret_cast<float *>(sm + C::OFF_Q);
  uint64_t *p_s = reinterpret_cast<uint64_t *>(sm + C::OFF_P);
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
  uint64_t *empty = full + C::NS;
  volatile int *slot_tag = reinterpret_cast<volatile int *>(sm + C::OFF_TAG);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC);
  Watchdog *wdp = reinterpret_cast<Watchdog *>(sm + C::OFF_MISC + 16);
  const bool t5 = p.bias.table != nullptr;
  const int nb = t5 ? p.bias.nb : 0;
  const int lutn = t5 ? p.bias.sat_pos + p.bias.sat_neg - 1 : 0;
  const DecTail tail = dec_tail(C::OFF_TAB, G, nb, lutn);
  float *tab_s = reinterpret_cast<float *>(sm + tail.tab);
  uint8_t *lut_s = sm + tail.lut;

  if (warp == kDecWarps) {
    if (lane == 0) {
      for (int s = 0; s < C::NS; ++s) {
        mbar_init(full + s, 1);
        mbar_init(empty + s, 1);
        slot_tag[s] = -1;
      }
      *abort_flag = 0;
      *wdp = Watchdog{abort_flag, p.err, FAT_DEVERR_TIMEOUT_FWD, p.timeout_ns};
      fence_mbar_init();
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
  } else {
    const float sc = p.scale_log2;
    for (int i = tid; i < R * (D / 8); i += kDecWarps * 32) {
      const int r = i / (D / 8), c8 = i % (D / 8);
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (r < nrows) {
        const int qi = r / G, g = r - qi * G;
        const uint4 w = *reinterpret_cast<const uint4 *>(
            qg + ((size_t)(span.sq + qi) * H + (size_t)hk * G + g) * D + c8 * 8);
        a = make_float4(__uint_as_float(w.x << 16) * sc, __uint_as_float(w.x & 0xffff0000u) * sc,
                        __uint_as_float(w.y << 16) * sc, __uint_as_float(w.y & 0xffff0000u) * sc);
        b = make_float4(__uint_as_float(w.z << 16) * sc, __uint_as_float(w.z & 0xffff0000u) * sc,
                        __uint_as_float(w.w << 16) * sc, __uint_as_float(w.w & 0xffff0000u) * sc);
      }
      float4 *dst = reinterpret_cast<float4 *>(q_s + r * D + c8 * 8);
      dst[0] = a;
      dst[1] = b;
    }
    if (t5) {
      for (int i = tid; i < G * nb; i += kDecWarps * 32) {
        const int g = i / nb, bk = i - g * nb;
        tab_s[i] = __ldg(p.bias.table + (size_t)bk * H + (size_t)hk * G + g) * kLog2e;
      }
      for (int i = tid; i < lutn; i += kDecWarps * 32)
        lut_s[i] = (uint8_t)t5_bucket_dev(i - (p.bias.sat_neg - 1), p.bias);
    }
  }
  __syncthreads();
  const Watchdog &wd = *wdp;

  if (warp == kDecWarps) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int i = 0;
      for (; i < nst; ++i) {
        const int s = i % C::NS;
        if (i >= C::NS && !mbar_wait(empty + s, ((i / C::NS) - 1) & 1, wd)) break;
        slot_tag[s] = i;  // the slot's previous stage has been consumed
        mbar_arrive_expect_tx(full + s, C::STAGE);
        uint8_t *dst = sm + s * C::STAGE;
        const int row = span.sk + kbeg + i * kDecKT;
#pragma unroll
        for (int b = 0; b < C::BOXES; ++b) {
          tma_load_3d(&tm_k, full + s, dst + b * C::BOX, 64 * b, hk, row);
          tma_load_3d(&tm_v, full + s, dst + C::TILE + b * C::BOX, 64 * b, hk, row);
        }
      }
      // copies still in flight (after an abort) land before this thread, and so the block,
      // exits
      for (int j = max(0, i - C::NS); j < i; ++j)
        mbar_wait_teardown(full + (j % C::NS), (j / C::NS) & 1, kTeardownNs);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  // per row: last visible key (document-local; -1: padding row), query position in key
  // coordinates, head within the group, ALiBi slope in log2 units
  int lim[R], qpos[R], grow[R];
  float slope[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int qi = r / G, g = r - qi * G;
    qpos[r] = qi + span.shift;
    grow[r] = g;
    lim[r] = r >= nrows ? -1 : (p.causal ? min(qpos[r], kend - 1) : kend - 1);
    slope[r] = (p.bias.slopes != nullptr && r < nrows)
                   ? __ldg(p.bias.slopes + (size_t)hk * G + g) * kLog2e
                   : 0.f;
  }
  // the saturated buckets: every delta >= sat_pos, every delta <= -sat_neg
  const int sat_pos = p.bias.sat_pos, sat_neg = p.bias.sat_neg;
  const int bucket_pos = t5 ? t5_bucket_dev(sat_pos, p.bias) : 0;
  const int bucket_neg = t5 ? t5_bucket_dev(-sat_neg, p.bias) : 0;

  float m[R], l[R];
  uint64_t o2[R][CPL / 2];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL / 2; ++c) o2[r][c] = 0ull;
  }
  uint64_t *pw = p_s + warp * 32 * R;

  for (int i = warp; i < nst; i += kDecWarps) {
    const int s = i % C::NS;
    if (!__all_sync(0xffffffffu, wait_slot_tag(slot_tag + s, i, wd))) break;
    if (!warp_wait(full + s, (i / C::NS) & 1, wd)) break;
    const uint8_t *kt = sm + s * C::STAGE, *vt = kt + C::TILE;
    const int k0 = kbeg + i * kDecKT;  // document-local index of the stage's first key
    const int key = k0 + lane;
    // scores of this lane's key against every row
    uint64_t acc[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r][0] = acc[r][1] = 0ull;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 kw = *reinterpret_cast<const uint4 *>(kt + (c >> 3) * C::BOX + lane * 128 +
                                                        (((c & 7) ^ (lane & 7)) << 4));
      const uint64_t k01 = bf16x2_to_f2(kw.x), k23 = bf16x2_to_f2(kw.y);
      const uint64_t k45 = bf16x2_to_f2(kw.z), k67 = bf16x2_to_f2(kw.w);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const ulonglong2 qa = *reinterpret_cast<const ulonglong2 *>(q_s + r * D + c * 8);
        const ulonglong2 qb = *reinterpret_cast<const ulonglong2 *>(q_s + r * D + c * 8 + 4);
        acc[r][c & 1] = f2_fma(qa.x, k01, acc[r][c & 1]);
        acc[r][c & 1] = f2_fma(qa.y, k23, acc[r][c & 1]);
        acc[r][c & 1] = f2_fma(qb.x, k45, acc[r][c & 1]);
        acc[r][c & 1] = f2_fma(qb.y, k67, acc[r][c & 1]);
      }
    }
    float pr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float a0, a1, b0, b1;
      f2_unpack(acc[r][0], a0, a1);
      f2_unpack(acc[r][1], b0, b1);
      float x = -INFINITY;
      if (key <= lim[r]) {
        const int delta = key - qpos[r];
        x = (a0 + a1) + (b0 + b1);
        if (t5) {
          const int bk = delta >= sat_pos ? bucket_pos
                         : delta <= -sat_neg ? bucket_neg
                                             : (int)lut_s[delta + sat_neg - 1];
          x += tab_s[grow[r] * nb + bk];
        }
        x -= slope[r] * (float)(delta < 0 ? -delta : delta);
      }
      // running max of the row over this warp's keys; the output is rescaled only when it grows
      const float mt = dec_warp_max(x);
      if (mt > m[r]) {
        const float corr = ex2(m[r] - mt);  // 0 while the row had no key
        l[r] *= corr;
        const uint64_t c2 = f2_pack(corr, corr);
#pragma unroll
        for (int c = 0; c < CPL / 2; ++c) o2[r][c] = f2_mul(o2[r][c], c2);
        m[r] = mt;
      }
      pr[r] = x == -INFINITY ? 0.f : ex2(x - m[r]);
      l[r] += pr[r];
    }
    // the probabilities, as (p, p) pairs, for the P V walk
#pragma unroll
    for (int r = 0; r < R; r += 2)
      *reinterpret_cast<ulonglong2 *>(pw + lane * R + r) =
          make_ulonglong2(f2_pack(pr[r], pr[r]), f2_pack(pr[r + 1], pr[r + 1]));
    __syncwarp();
    // P V over the stage's keys inside the split (later rows of the tile belong to another
    // range or document and are not read)
    const int nk = min(kDecKT, kend - k0);
    const int ch = lane * CPL;                 // first channel of this lane
    const int box = ch >> 6, cin = (ch & 63) >> 3, within = (ch & 7) * 2;
    const uint8_t *vbase = vt + box * C::BOX + within;
    for (int j = 0; j < nk; ++j) {
      const uint8_t *vrow = vbase + j * 128 + ((cin ^ (j & 7)) << 4);
      uint64_t v2[CPL / 2];
      if constexpr (CPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(vrow);
        v2[0] = bf16x2_to_f2(w.x);
        v2[1] = bf16x2_to_f2(w.y);
      } else {
        v2[0] = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(vrow));
      }
#pragma unroll
      for (int r = 0; r < R; r += 2) {
        const ulonglong2 pp = *reinterpret_cast<const ulonglong2 *>(pw + j * R + r);
#pragma unroll
        for (int c = 0; c < CPL / 2; ++c) {
          o2[r][c] = f2_fma(pp.x, v2[c], o2[r][c]);
          o2[r + 1][c] = f2_fma(pp.y, v2[c], o2[r + 1][c]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + s);
  }

  // ------------------------------------------------------------- merge and store
  named_bar_sync(1, kDecWarps * 32);
  const bool ok = *abort_flag == 0;
  float *mo = reinterpret_cast<float *>(sm);  // [warps][R][D] over the drained ring
  float *ml = mo + kDecWarps * R * D;         // [warps][R] x (max, sum)
  if (ok) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float ls = dec_warp_sum(l[r]);
      if (lane == 0) {
        ml[(warp * R + r) * 2] = m[r];
        ml[(warp * R + r) * 2 + 1] = ls;
      }
      float *dst = mo + (warp * R + r) * D + lane * CPL;
      if constexpr (CPL == 4) {
        float a, b, c, d;
        f2_unpack(o2[r][0], a, b);
        f2_unpack(o2[r][1], c, d);
        *reinterpret_cast<float4 *>(dst) = make_float4(a, b, c, d);
      } else {
        float a, b;
        f2_unpack(o2[r][0], a, b);
        *reinterpret_cast<float2 *>(dst) = make_float2(a, b);
      }
    }
  }
  named_bar_sync(1, kDecWarps * 32);
  if (!ok) return;
  for (int i = tid; i < nrows * (D / 4); i += kDecWarps * 32) {
    const int r = i / (D / 4), c4 = (i - r * (D / 4)) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, ml[(w * R + r) * 2]);
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = ml[(w * R + r) * 2];
        if (mw == -INFINITY) continue;
        const float f = ex2(mw - M);
        wsum += f * ml[(w * R + r) * 2 + 1];
        const float4 o = *reinterpret_cast<const float4 *>(mo + (w * R + r) * D + c4);
        acc.x += f * o.x;
        acc.y += f * o.y;
        acc.z += f * o.z;
        acc.w += f * o.w;
      }
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    const float lse = wsum > 0.f ? (M + __log2f(wsum)) * kLn2 : -INFINITY;
    const int qi = r / G, h = hk * G + (r - qi * G), row = span.sq + qi;
    if (p.kv_splits == 1) {
      uint2 v;
      v.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      v.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2 *>(p.out + ((size_t)row * H + h) * D + c4) = v;
      if (c4 == 0 && p.lse != nullptr) p.lse[(size_t)h * T + row] = lse;
    } else {
      *reinterpret_cast<float4 *>(p.o_part + (((size_t)split * T + row) * H + h) * D + c4) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      if (c4 == 0) p.lse_part[((size_t)split * H + h) * T + row] = lse;
    }
  }
}

template <int D, int R>
int launch_decode_t(const FwdParams &p, const void *qp, const void *k, const void *v,
                    cudaStream_t stream) {
  using C = DecCfg<D, R>;
  CUtensorMap mk, mv;
  if (make_tmap_thd(&mk, k, p.seq.total_k, p.seq.num_heads_kv, D, kDecKT) ||
      make_tmap_thd(&mv, v, p.seq.total_k, p.seq.num_heads_kv, D, kDecKT))
    return (int)cudaErrorInvalidValue;
  const size_t smem = decode_smem_bytes(D, R, p.seq.group, p.bias);
  cudaError_t e = (cudaError_t)prepare_kernel((const void *)fat_decode_kernel<D, R>, smem,
                                              kDecThreads, 0);
  if (e != cudaSuccess) return (int)e;
  const dim3 grid(p.kv_splits, p.seq.num_heads_kv, p.seq.num_seqs);
  fat_decode_kernel<D, R><<<grid, kDecThreads, smem, stream>>>(
      mk, mv, static_cast<const __nv_bfloat16 *>(qp), p);
  e = cudaGetLastError();
  if (e != cudaSuccess) set_last_error("decode kernel launch", (int)e, cudaGetErrorString(e));
  return (int)e;
}

}  // namespace

int decode_rows(int head_dim, int rows) {
  (void)head_dim;
  return rows <= 2 ? 2 : rows <= 4 ? 4 : rows <= 8 ? 8 : 0;
}

size_t decode_smem_bytes(int head_dim, int R, int group, const BiasParams &b) {
  const int nb = b.table ? b.nb : 0;
  const int lutn = b.table ? b.sat_pos + b.sat_neg - 1 : 0;
  int base = 0;
#define FAT_DEC_BASE(DD, RR) \
  if (head_dim == DD && R == RR) base = DecCfg<DD, RR>::OFF_TAB;
  FAT_DEC_BASE(64, 2) FAT_DEC_BASE(64, 4) FAT_DEC_BASE(64, 8)
  FAT_DEC_BASE(128, 2) FAT_DEC_BASE(128, 4) FAT_DEC_BASE(128, 8)
#undef FAT_DEC_BASE
  if (base == 0) return 0;
  return 1024 + (size_t)dec_tail(base, group, nb, lutn).total;
}

bool decode_eligible(int head_dim, int max_rows, int group, const BiasParams &b) {
  if (decode_rows(head_dim, max_rows) == 0) return false;
  if (b.table && b.sat_pos + b.sat_neg - 1 > kDecMaxLut) return false;
  const size_t smem = decode_smem_bytes(head_dim, decode_rows(head_dim, max_rows), group, b);
  return smem != 0 && smem <= (size_t)kSmemLimit;
}

int decode_blocks_per_sm() { return 2; }

int launch_decode(const FwdParams &p, int head_dim, const void *q, const void *k, const void *v,
                  cudaStream_t stream) {
  const int R = decode_rows(head_dim, p.seq.max_seqlen * p.seq.group);
  if (head_dim == 64) {
    if (R == 2) return launch_decode_t<64, 2>(p, q, k, v, stream);
    if (R == 4) return launch_decode_t<64, 4>(p, q, k, v, stream);
    if (R == 8) return launch_decode_t<64, 8>(p, q, k, v, stream);
  } else if (head_dim == 128) {
    if (R == 2) return launch_decode_t<128, 2>(p, q, k, v, stream);
    if (R == 4) return launch_decode_t<128, 4>(p, q, k, v, stream);
    if (R == 8) return launch_decode_t<128, 8>(p, q, k, v, stream);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace fat
