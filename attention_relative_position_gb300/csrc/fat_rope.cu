// fat_rope.cu -- rotary position embedding (RoFormer's RoPE) of packed varlen rows, the
// rotation the FAT5 report lists among the positional encodings its attention kernels take
// ("Noyau CUDA" section, positional-encoding classes): channel pair (2i, 2i + 1) of a row at
// position m turns by m * theta_i, theta_i = base^(-2i/d), positions local to each document.
// Applied to Q and K before the attention kernels (inverse = transposed rotation for dQ, dK).
//
// Memory bound: a thread takes one (token, 16-byte chunk) position, computes its four angles
// once and turns that chunk of every head (16-byte loads and stores). The angle is
// taken exactly modulo one turn: each pair's rate theta_i / (2 pi) is a 64-bit fixed-point
// fraction of a turn (from double precision on the host), so m * rate mod 1 is one integer
// multiply that wraps, whatever the position; its top bits give the turn fraction in [0, 1), and
// sincospif turns it into the cosine and sine (fp32 accuracy at any position).
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "fat_attn_internal.cuh"

namespace fat {
namespace {

constexpr int kMaxPairs = 64;  // head_dim <= 128
constexpr int kHeadBatch = 8;  // heads whose loads one thread issues together

struct RopeParams {
  const int32_t *cu_seqlens;
  const uint4 *x;
  uint4 *y;
  int T, H, d, num_seqs, max_seqlen;
  int inverse;
  int *err;
  unsigned long long rate[kMaxPairs];  // turns per position of pair i, 2^-64 units
};

__global__ void __launch_bounds__(256) fat_rope_kernel(const RopeParams p) {
  const int doc = blockIdx.y;
  const int s = __ldg(p.cu_seqlens + doc), e = __ldg(p.cu_seqlens + doc + 1);
  if (s < 0 || e > p.T || e < s) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.err, FAT_DEVERR_SEQLENS);
    return;
  }
  if (e - s > p.max_seqlen && threadIdx.x == 0 && blockIdx.x == 0)
    atomicOr(p.err, FAT_DEVERR_SEQLENS);
  // one thread per (token, 16-byte chunk of a head): its four angles are computed once and
  // applied to that chunk of every head (the heads share the positions)
  const int cph = p.d / 8;  // chunks per head
  const long long n = (long long)(e - s) * cph;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int tok = (int)(i / cph);
    const int c = (int)(i % cph);  // pairs 4c .. 4c + 3
    const unsigned long long pos = (unsigned long long)tok;
    float cs[4], sn[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // fraction of a turn in [0, 1): the top 24 bits of pos * rate mod 2^64
      const unsigned long long turns = pos * p.rate[4 * c + k];
      const float frac = (float)(uint32_t)(turns >> 40) * (1.0f / 16777216.0f);
      sincospif(2.0f * frac, &sn[k], &cs[k]);
      if (p.inverse) sn[k] = -sn[k];
    }
    const long long base = (long long)(s + tok) * p.H * cph + c;
    // heads in groups of kHeadBatch: all loads of a group are issued before its stores, so a
    // thread keeps several 16-byte reads in flight (x and y may be the same buffer: each
    // thread reads and writes only its own chunks, reads first)
    for (int h0 = 0; h0 < p.H; h0 += kHeadBatch) {
      uint4 v[kHeadBatch];
#pragma unroll
      for (int j = 0; j < kHeadBatch; ++j)
        if (h0 + j < p.H) v[j] = p.x[base + (long long)(h0 + j) * cph];
#pragma unroll
      for (int j = 0; j < kHeadBatch; ++j) {
        if (h0 + j >= p.H) break;
        uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          __nv_bfloat162 pr = *reinterpret_cast<__nv_bfloat162 *>(&w[k]);
          const float2 a = __bfloat1622float2(pr);
          w[k] = pack_bf16x2(a.x * cs[k] - a.y * sn[k], a.x * sn[k] + a.y * cs[k]);
        }
        p.y[base + (long long)(h0 + j) * cph] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

}  // namespace
}  // namespace fat

using namespace fat;

extern "C" int fat_rope_apply(const fat_shape_t *sh, const void *x, void *y,
                              const int32_t *cu_seqlens, double base, int inverse) {
  if (!sh || !x || !y || !cu_seqlens) return FAT_EINVAL_NULL;
  if (sh->total_tokens < 0 || sh->num_seqs < 0 || sh->max_seqlen < 0 || sh->num_heads <= 0)
    return FAT_EINVAL_SHAPE;
  if (sh->head_dim != 64 && sh->head_dim != 128) return FAT_EINVAL_SHAPE;
  if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
        reinterpret_cast<uintptr_t>(cu_seqlens)) & 15u) != 0)
    return FAT_EINVAL_SHAPE;
  if (!(base > 1.0) || !std::isfinite(base)) return FAT_EINVAL_SHAPE;
  if (sh->num_seqs > 65535) return FAT_EUNSUPPORTED;
  if (sh->total_tokens == 0 || sh->num_seqs == 0 || sh->max_seqlen == 0) return FAT_OK;
  RopeParams p{};
  p.cu_seqlens = cu_seqlens;
  p.x = static_cast<const uint4 *>(x);
  p.y = static_cast<uint4 *>(y);
  p.T = sh->total_tokens;
  p.H = sh->num_heads;
  p.d = sh->head_dim;
  p.num_seqs = sh->num_seqs;
  p.max_seqlen = sh->max_seqlen;
  p.inverse = inverse ? 1 : 0;
  // rate_i = theta_i / (2 pi) turns per position, as a 64-bit fraction (theta_i < 2 pi for
  // base > 1, so the integer part is 0)
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < p.d / 2; ++i) {
    const double turns = std::pow(base, -2.0 * i / p.d) / two_pi;
    const double scaled = std::ldexp(turns - std::floor(turns), 64);
    p.rate[i] = scaled >= 18446744073709551615.0 ? ~0ull : (unsigned long long)scaled;
  }
  int rc = device_error_address(&p.err);
  if (rc) return rc;
  // enough blocks for every (token, chunk) of the longest document, at most ~8 per SM in all
  const long long per_doc = (long long)sh->max_seqlen * sh->head_dim / 8;
  const int sms = sm_count() > 0 ? sm_count() : 152;
  const long long cap = std::max<long long>(1, (long long)sms * 8 / sh->num_seqs);
  const int bx = (int)std::min<long long>((per_doc + 255) / 256, cap);
  const dim3 grid(bx > 0 ? bx : 1, sh->num_seqs);
  fat_rope_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(sh->stream)>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_error("rotary embedding launch", (int)e, cudaGetErrorString(e));
    rc = FAT_ECUDA;
  }
  return rc;
}
