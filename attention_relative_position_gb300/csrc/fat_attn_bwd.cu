// fat_attn_bwd.cu -- backward kernel of the fused relative-position attention.
//
// The FAT5 report benchmarks the backward of its bias kernel ("Benchmark / TFLOPS" section)
// without describing it; this is the standard softmax-attention backward of loss = sum(O * dO):
//   P = exp(S' - lse), dV = P^T dO, dP = dO V^T, dS = P * (dP - D) with D = rowsum(dO * O),
//   dK = scale * dS^T Q, dQ = scale * dS K, dTable[b, h] = sum of dS over pairs in bucket b.
//
// GB300 design: one CTA per (document, head, 128-key tile); it walks the query tiles of the
// document (only those at or after the key tile when causal). Everything is computed in the
// key-major frame (TMEM lane = key row):
//   warp 12      TMA producer: K, V once; Q_i, dO_i (and lse_i, D_i) through a 2-stage ring.
//   warp 13      MMA issuer: S^T = K Q_i^T, dP^T = V dO_i^T, dV += P^T dO_i (P^T from TMEM),
//                dK += dS^T Q_i, and dQ_i = dS K (d = 64) or dQ_i^T = K^T dS^T (d = 128), all
//                tcgen05 with fp32 accumulators in TMEM; dK and dV stay in TMEM for the whole
//                walk.
//   warps 0-7    two warpgroups, each owning half of the query columns: P^T = 2^(x - lse),
//                written to TMEM as bf16; dS^T = P^T (dP^T - D), written to shared memory in the
//                128-byte-swizzled layout the MMAs read; bias-gradient partial sums.
//   warps 8-11   drain dQ_i from TMEM into the fp32 dQ accumulator with vector reductions, then
//                write dK, dV.
//   warps 14-15  idle; with warps 12-13 they form the fourth warpgroup, whose registers go to
//                the P/dS warpgroups (168 + 168 + 112 + 64 = 512 per SM sub-partition).
// Bias gradient: tiles beyond the T5 saturation distance add dS into one register per side;
// the other tiles add into a shared-memory array indexed by delta (one conflict-free shared
// reduction per element, consecutive lanes hit consecutive deltas); at the end the CTA maps
// deltas to buckets and issues one global atomic per (bucket, head).
// Query tiles are 128 wide for d = 64 and 64 wide for d = 128 so that S, dP, dQ, dK and dV fit
// the 512 TMEM columns together.
#include <cstdio>

#include "fat_attn_internal.cuh"

namespace fat {

template <int D>
struct BwdCfg {
  static constexpr int BQ = (D == 64) ? 128 : 64;
  static constexpr int HALF = BQ / 2;           // query columns per softmax warpgroup
  static constexpr int DB = D / 64;
  static constexpr int KBLK = 128 * 128;        // 128 rows x 64 bf16
  static constexpr int KTILE = DB * KBLK;       // K or V tile: 128 keys x D
  static constexpr int QBLK = BQ * 128;         // BQ rows x 64 bf16
  static constexpr int QTILE = DB * QBLK;       // Q_i or dO_i tile
  static constexpr int NS = 2;
  static constexpr int DSBLK = 128 * 128;       // 128 keys x 64 queries bf16
  static constexpr int DSTILE = (BQ / 64) * DSBLK;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KTILE;
  static constexpr int OFF_Q = OFF_V + KTILE;
  static constexpr int OFF_DO = OFF_Q + NS * QTILE;
  static constexpr int OFF_DS = OFF_DO + NS * QTILE;
  static constexpr int OFF_STAT = OFF_DS + 2 * DSTILE;  // lse2[NS][BQ] then dvec[NS][BQ]
  static constexpr int OFF_BAR = OFF_STAT + NS * 2 * BQ * 4;
  static constexpr int OFF_BACC = OFF_BAR + 256;        // per-bucket sums, 256 floats
  static constexpr int OFF_LUT = OFF_BACC + 256 * 4;    // lut[lut_len], then diag[lut_len]
  static constexpr int NTHREADS = 512;
  static constexpr int COL_S = 0, COL_DP = BQ, COL_DQ = 2 * BQ;
  static constexpr int COL_DK = 512 - 2 * D, COL_DV = 512 - D;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, BQ, 0, 0);
  static constexpr uint32_t IDESC_DKV = idesc_bf16_f32(128, D, 0, 1);
  static constexpr uint32_t IDESC_DQ = idesc_bf16_f32(128, 64, 1, 1);
};

size_t bwd_smem_bytes(int head_dim, int lut_len) {
  size_t base = head_dim == 64 ? (size_t)BwdCfg<64>::OFF_LUT : (size_t)BwdCfg<128>::OFF_LUT;
  return 1024 + base + (size_t)lut_len * 8;
}

template <int D>
__global__ void __launch_bounds__(512, 1)
    fat_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kb = blockIdx.x, h = blockIdx.y, doc = blockIdx.z;
  const int T = p.seq.total_tokens, H = p.seq.num_heads;
  const int seq_start = __ldg(p.seq.cu_seqlens + doc);
  const int seq_end = __ldg(p.seq.cu_seqlens + doc + 1);
  if (seq_start < 0 || seq_end > T || seq_end < seq_start) {
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.err, FAT_DEVERR_SEQLENS);
    return;
  }
  const int L = seq_end - seq_start;
  const int ks = kb * 128;
  if (ks >= L) return;
  const int i0 = p.causal ? ks / C::BQ : 0;
  const int nq = (L + C::BQ - 1) / C::BQ - i0;
  const bool do_dbias = p.dbias != nullptr && p.bias.table != nullptr;

  uint8_t *sK = sm + C::OFF_K, *sV = sm + C::OFF_V, *sQ = sm + C::OFF_Q, *sDO = sm + C::OFF_DO;
  uint8_t *sDS = sm + C::OFF_DS;
  float *s_lse2 = reinterpret_cast<float *>(sm + C::OFF_STAT);
  float *s_dvec = s_lse2 + C::NS * C::BQ;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
  uint64_t *kv_full = bars;
  uint64_t *qd_full = kv_full + 1;       // [NS]
  uint64_t *qd_empty = qd_full + C::NS;  // [NS]
  uint64_t *s_full = qd_empty + C::NS;
  uint64_t *dp_full = s_full + 1;
  uint64_t *p_ready = dp_full + 1;
  uint64_t *ds_ready = p_ready + 1;
  uint64_t *ds_empty = ds_ready + 1;     // [2]
  uint64_t *dq_full = ds_empty + 2;
  uint64_t *dq_empty = dq_full + 1;
  uint64_t *dkdv_done = dq_empty + 1;
  uint64_t *mma_done = dkdv_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *bacc = reinterpret_cast<float *>(sm + C::OFF_BACC);
  float *lut = reinterpret_cast<float *>(sm + C::OFF_LUT);
  float *diag = lut + p.bias.lut_len;

  if (tid == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(qd_full + s, 32);
      mbar_init(qd_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(ds_empty, 1);
    mbar_init(ds_empty + 1, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(dkdv_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 12 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  for (int i = tid; i < p.bias.lut_len; i += C::NTHREADS) {
    lut[i] = bias_log2_dev(p.bias.lut_lo + i, h, H, p.bias);
    if (do_dbias) diag[i] = 0.f;
  }
  if (do_dbias)
    for (int i = tid; i < 256; i += C::NTHREADS) bacc[i] = 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Watchdog wd{abort_flag, p.err, FAT_DEVERR_TIMEOUT_BWD, p.timeout_ns};
  float acc_pos = 0.f, acc_neg = 0.f;  // bias-gradient sums of far tiles (softmax warps)
  if (warp >= 12) regs_dec<64>();
  else if (warp >= 8) regs_dec<112>();

  if (warp == 12) {
    // ------------------------------------------------------------------ producer
    int last_q[C::NS] = {-1, -1};
    bool kv_issued = false;
    if (!(p.debug_flags & 2)) {
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, 2 * C::KTILE);
        for (int b = 0; b < C::DB; ++b) {
          tma_load_3d(&tm_k, kv_full, sK + b * C::KBLK, 64 * b, h, seq_start + ks);
          tma_load_3d(&tm_v, kv_full, sV + b * C::KBLK, 64 * b, h, seq_start + ks);
        }
        kv_issued = true;
      }
      for (int it = 0; it < nq; ++it) {
        const int st = it % C::NS, u = it / C::NS;
        if (u > 0 && !__all_sync(0xffffffffu, mbar_wait(qd_empty + st, (u - 1) & 1, wd))) break;
        const int qs = (i0 + it) * C::BQ;
        for (int c = lane; c < C::BQ; c += 32) {
          const int q = qs + c;
          const bool valid = q < L;
          const size_t idx = (size_t)h * T + seq_start + q;
          s_lse2[st * C::BQ + c] = valid ? __ldg(p.lse + idx) * kLog2e : 0.f;
          s_dvec[st * C::BQ + c] = valid ? __ldg(p.dvec + idx) : 0.f;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(qd_full + st, 2 * C::QTILE);
          for (int b = 0; b < C::DB; ++b) {
            tma_load_3d(&tm_q, qd_full + st, sQ + st * C::QTILE + b * C::QBLK, 64 * b, h,
                        seq_start + qs);
            tma_load_3d(&tm_do, qd_full + st, sDO + st * C::QTILE + b * C::QBLK, 64 * b, h,
                        seq_start + qs);
          }
          if (st == 0) last_q[0] = u; else last_q[1] = u;
        } else {
          mbar_arrive(qd_full + st);
        }
      }
    }
    if (lane == 0) {
      if (kv_issued) mbar_wait_teardown(kv_full, 0, kTeardownNs);
      if (last_q[0] >= 0) mbar_wait_teardown(qd_full, last_q[0] & 1, kTeardownNs);
      if (last_q[1] >= 0) mbar_wait_teardown(qd_full + 1, last_q[1] & 1, kTeardownNs);
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), aDO = smem_u32(sDO);
      const uint32_t aDS = smem_u32(sDS);
      auto issue_qk = [&](uint32_t a_base, uint32_t b_base, uint32_t dcol) {
        // D[key][q] = sum_c A[key][c] * B[q][c]; A, B K-major
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = sw128_desc(a_base + (kk >> 2) * C::KBLK + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sw128_desc(b_base + (kk >> 2) * C::QBLK + (kk & 3) * 32, 16, 1024);
          mma_bf16_ss(tmem + dcol, a, b, C::IDESC_S, kk > 0);
        }
      };
      auto issue_dv = [&](int st, bool acc) {
        // dV[key][c] += sum_q P^T[key][q] dO[q][c]; A = P^T in TMEM, B = dO MN-major
#pragma unroll
        for (int k16 = 0; k16 < C::BQ / 16; ++k16) {
          const int q0 = 16 * k16;
          const uint32_t a_t = tmem + C::COL_S + (q0 / C::HALF) * C::HALF + (q0 % C::HALF) / 2;
          const uint64_t b = sw128_desc(aDO + st * C::QTILE + k16 * 2048, C::QBLK, 1024);
          mma_bf16_ts(tmem + C::COL_DV, a_t, b, C::IDESC_DKV, (acc || k16 > 0) ? 1u : 0u);
        }
      };
      auto issue_dk = [&](int buf, int st, bool acc) {
        // dK[key][c] += sum_q dS^T[key][q] Q[q][c]; A = dS^T K-major, B = Q MN-major
#pragma unroll
        for (int k16 = 0; k16 < C::BQ / 16; ++k16) {
          const int q0 = 16 * k16;
          const uint64_t a = sw128_desc(
              aDS + buf * C::DSTILE + (q0 >> 6) * C::DSBLK + ((q0 & 63) >> 4) * 32, 16, 1024);
          const uint64_t b = sw128_desc(aQ + st * C::QTILE + k16 * 2048, C::QBLK, 1024);
          mma_bf16_ss(tmem + C::COL_DK, a, b, C::IDESC_DKV, (acc || k16 > 0) ? 1u : 0u);
        }
      };
      auto issue_dq = [&](int buf) {
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16) {  // 128 keys
          const uint64_t ds = sw128_desc(aDS + buf * C::DSTILE + k16 * 2048, C::DSBLK, 1024);
          const uint64_t kk = sw128_desc(aK + k16 * 2048, C::KBLK, 1024);
          if (D == 64)  // dQ[q][c] = sum_key dS[q][key] K[key][c]
            mma_bf16_ss(tmem + C::COL_DQ, ds, kk, C::IDESC_DQ, k16 > 0);
          else          // dQ^T[c][q] = sum_key K[key][c] dS^T[key][q]
            mma_bf16_ss(tmem + C::COL_DQ, kk, ds, C::IDESC_DQ, k16 > 0);
        }
      };
      bool ok = mbar_wait(kv_full, 0, wd) && mbar_wait(qd_full, 0, wd);
      if (ok) {
        tc_fence_after();
        issue_qk(aK, aQ, C::COL_S);
        mma_commit(s_full);
        issue_qk(aV, aDO, C::COL_DP);
        mma_commit(dp_full);
      }
      for (int it = 0; ok && it < nq; ++it) {
        const int st = it % C::NS;
        const int stn = (it + 1) % C::NS, un = (it + 1) / C::NS;
        if (!mbar_wait(p_ready, it & 1, wd)) { ok = false; break; }
        tc_fence_after();
        issue_dv(st, it > 0);
        if (it + 1 < nq) {
          if (!mbar_wait(qd_full + stn, un & 1, wd)) { ok = false; break; }
          tc_fence_after();
          issue_qk(aK, aQ + stn * C::QTILE, C::COL_S);
          mma_commit(s_full);
        }
        if (!mbar_wait(ds_ready, it & 1, wd)) { ok = false; break; }
        tc_fence_after();
        issue_dk(it & 1, st, it > 0);
        if (it >= 1) {
          if (!mbar_wait(dq_empty, (it - 1) & 1, wd)) { ok = false; break; }
          tc_fence_after();
        }
        issue_dq(it & 1);
        mma_commit(dq_full);
        mma_commit(ds_empty + (it & 1));
        mma_commit(qd_empty + st);
        if (it + 1 < nq) {
          issue_qk(aV, aDO + stn * C::QTILE, C::COL_DP);
          mma_commit(dp_full);
        }
      }
      if (ok) mma_commit(dkdv_done);
      mma_commit(mma_done);
      mbar_wait_teardown(mma_done, 0, kTeardownNs);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------------ P / dS warpgroups
    regs_inc<168>();
    const int wg = warp >> 2;
    const int r = tid & 127;
    const int c0 = wg * C::HALF;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::COL_S + c0;
    const uint32_t tDP = tmem + lane_off + C::COL_DP + c0;
    const int krow = ks + r;
    const bool row_valid = krow < L;
    const FarBias fb = far_bias_dev(h, H, p.bias);
    const bool has_slopes = p.bias.slopes != nullptr;
    float pv[C::HALF];
    for (int it = 0; it < nq; ++it) {
      const int st = it % C::NS;
      const int qs = (i0 + it) * C::BQ;
      if (!__all_sync(0xffffffffu, mbar_wait(qd_full + st, (it / C::NS) & 1, wd))) break;
      if (!__all_sync(0xffffffffu, mbar_wait(s_full, it & 1, wd))) break;
      tc_fence_after();
      const int d0 = ks - qs;  // delta of (key row 0, query column 0)
      const bool need_mask = (ks + 128 > L) || (qs + C::BQ > L) || (p.causal && d0 + 127 > 0);
      const int lo_j = p.causal ? krow - qs : -1;
      const int hi_j = row_valid ? L - qs : 0;
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
      const float *lse2 = s_lse2 + st * C::BQ;
      const float *dvs = s_dvec + st * C::BQ;
      // ---- P^T = 2^(x - lse2) for this warpgroup's query columns
#pragma unroll
      for (int c = 0; c < C::HALF / 32; ++c) {
        uint32_t raw[32];
        tmem_ld32(tS + 32 * c, raw);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int j = c0 + 32 * c + i;
          float b;
          if (side == 0)
            b = lut[lut_base - j];
          else
            b = linear ? fmaf(kq, (float)j, rowc) : rowc;
          float x = fmaf(__uint_as_float(raw[i]), p.scale_log2, b);
          if (need_mask) x = (j >= lo_j && j < hi_j) ? x : -INFINITY;
          const float pr = ex2(x - lse2[j]);
          pv[32 * c + i] = pr;
          if (i & 1) pk[i >> 1] = pack_bf16x2(pv[32 * c + i - 1], pr);
        }
        tmem_st16(tS + 16 * c, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_ready);
      // ---- dS^T = P^T (dP^T - D), to shared memory (bf16, swizzled) for the dK / dQ MMAs
      if (!__all_sync(0xffffffffu, mbar_wait(dp_full, it & 1, wd))) break;
      if (it >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(ds_empty + (it & 1), ((it >> 1) - 1) & 1, wd)))
        break;
      tc_fence_after();
      uint8_t *dsb = sDS + (it & 1) * C::DSTILE;
#pragma unroll
      for (int c = 0; c < C::HALF / 32; ++c) {
        uint32_t raw[32];
        tmem_ld32(tDP + 32 * c, raw);
        float dsv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int j = c0 + 32 * c + i;
          dsv[i] = pv[32 * c + i] * (__uint_as_float(raw[i]) - dvs[j]);
          if (do_dbias) {
            if (side == 0)
              red_add_shared(diag + (lut_base - j), dsv[i]);
            else if (side == 1)
              acc_pos += dsv[i];
            else
              acc_neg += dsv[i];
          }
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(dsv[2 * i], dsv[2 * i + 1]);
#pragma unroll
        for (int g = 0; g < 4; ++g) {  // 4 groups of 8 queries = 16 bytes each
          const int j0 = c0 + 32 * c + 8 * g;
          const int chunk = (j0 & 63) >> 3;
          uint8_t *dst = dsb + (j0 >> 6) * C::DSBLK + r * 128 + ((chunk ^ (r & 7)) << 4);
          *reinterpret_cast<uint4 *>(dst) =
              make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(ds_ready);
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------------ dQ drain, dK/dV out
    const int dr = tid - 256;  // TMEM lane 0..127
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    for (int it = 0; it < nq; ++it) {
      const int qs = (i0 + it) * C::BQ;
      ok = __all_sync(0xffffffffu, mbar_wait(dq_full, it & 1, wd));
      if (!ok) break;
      tc_fence_after();
      uint32_t va[32], vb[32];
      tmem_ld32(tmem + lane_off + C::COL_DQ, va);
      tmem_ld32(tmem + lane_off + C::COL_DQ + 32, vb);
      tc_fence_before();
      mbar_arrive(dq_empty);
      if (D == 64) {  // lane = query row, columns = channels
        const int q = qs + dr;
        if (q < L) {
          float *dst = p.dq_acc + ((size_t)(seq_start + q) * H + h) * D;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            red_add_v4(dst + 4 * c, __uint_as_float(va[4 * c]), __uint_as_float(va[4 * c + 1]),
                       __uint_as_float(va[4 * c + 2]), __uint_as_float(va[4 * c + 3]));
#pragma unroll
          for (int c = 0; c < 8; ++c)
            red_add_v4(dst + 32 + 4 * c, __uint_as_float(vb[4 * c]),
                       __uint_as_float(vb[4 * c + 1]), __uint_as_float(vb[4 * c + 2]),
                       __uint_as_float(vb[4 * c + 3]));
        }
      } else {  // lane = channel, columns = query rows
        float *dst = p.dq_acc + ((size_t)(seq_start + qs) * H + h) * D + dr;
        const size_t step = (size_t)H * D;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (qs + j < L) red_add(dst + j * step, __uint_as_float(va[j]));
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (qs + 32 + j < L) red_add(dst + (32 + j) * step, __uint_as_float(vb[j]));
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(dkdv_done, 0, wd));
    if (ok) {
      tc_fence_after();
      const int krow = ks + dr;
      const bool valid = krow < L;
      __nv_bfloat16 *dkrow = p.dk + ((size_t)(seq_start + krow) * H + h) * D;
      __nv_bfloat16 *dvrow = p.dv + ((size_t)(seq_start + krow) * H + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 16; ++c) {
        uint32_t a[16];
        tmem_ld16(tmem + lane_off + C::COL_DK + 16 * c, a);
        uint32_t pa[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pa[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * p.scale,
                              __uint_as_float(a[2 * i + 1]) * p.scale);
        if (valid) {
          uint4 *dk4 = reinterpret_cast<uint4 *>(dkrow + 16 * c);
          dk4[0] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
          dk4[1] = make_uint4(pa[4], pa[5], pa[6], pa[7]);
        }
        tmem_ld16(tmem + lane_off + C::COL_DV + 16 * c, a);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pa[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
        if (valid) {
          uint4 *dv4 = reinterpret_cast<uint4 *>(dvrow + 16 * c);
          dv4[0] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
          dv4[1] = make_uint4(pa[4], pa[5], pa[6], pa[7]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (do_dbias && !*abort_flag) {
    // fold the per-delta and per-side partial sums into per-bucket sums, then one global
    // atomic per (bucket, head)
    for (int i = tid; i < p.bias.lut_len; i += C::NTHREADS) {
      const float v = diag[i];
      if (v != 0.f) atomicAdd(bacc + t5_bucket_dev(p.bias.lut_lo + i, p.bias), v);
    }
    if (warp < 8) {
      float a = acc_pos, b = acc_neg;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
      }
      if (lane == 0) {
        if (a != 0.f) atomicAdd(bacc + t5_bucket_dev(p.bias.sat_pos, p.bias), a);
        if (b != 0.f) atomicAdd(bacc + t5_bucket_dev(-p.bias.sat_neg, p.bias), b);
      }
    }
    __syncthreads();
    for (int b = tid; b < p.bias.nb; b += C::NTHREADS)
      if (bacc[b] != 0.f) atomicAdd(p.dbias + (size_t)b * H + h, bacc[b]);
  }
}

int launch_bwd(const BwdParams &p, int head_dim, int max_seqlen, const void *q, const void *k,
               const void *v, const void *out, const void *dout, cudaStream_t stream) {
  (void)out;
  CUtensorMap mq, mk, mv, mdo;
  const int T = p.seq.total_tokens, H = p.seq.num_heads;
  const int bq = head_dim == 64 ? BwdCfg<64>::BQ : BwdCfg<128>::BQ;
  if (make_tmap_thd(&mq, q, T, H, head_dim, bq) || make_tmap_thd(&mk, k, T, H, head_dim, 128) ||
      make_tmap_thd(&mv, v, T, H, head_dim, 128) || make_tmap_thd(&mdo, dout, T, H, head_dim, bq))
    return (int)cudaErrorInvalidValue;
  const size_t smem = bwd_smem_bytes(head_dim, p.bias.lut_len);
  dim3 grid((max_seqlen + 127) / 128, H, p.seq.num_seqs);
  cudaError_t e;
  if (head_dim == 64) {
    e = cudaFuncSetAttribute(fat_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess)
      fat_bwd_kernel<64><<<grid, BwdCfg<64>::NTHREADS, smem, stream>>>(mq, mk, mv, mdo, p);
  } else {
    e = cudaFuncSetAttribute(fat_bwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess)
      fat_bwd_kernel<128><<<grid, BwdCfg<128>::NTHREADS, smem, stream>>>(mq, mk, mv, mdo, p);
  }
  if (e != cudaSuccess) {
    set_last_error("cudaFuncSetAttribute(max dynamic shared memory)", (int)e, cudaGetErrorString(e));
    return (int)e;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFuncAttributes fa{};
    if (head_dim == 64)
      cudaFuncGetAttributes(&fa, fat_bwd_kernel<64>);
    else
      cudaFuncGetAttributes(&fa, fat_bwd_kernel<128>);
    char msg[160];
    snprintf(msg, sizeof msg, "%s [regs %d, max threads %d, local %zu B, dyn smem %zu B]",
             cudaGetErrorString(e), fa.numRegs, fa.maxThreadsPerBlock, (size_t)fa.localSizeBytes,
             smem);
    set_last_error("kernel launch", (int)e, msg);
  }
  return (int)e;
}

}  // namespace fat
