// fat_norm_ce.cu -- the FAT5 report's two other fused kernels ("Noyau Triton" section; speed and
// memory in "Torch vs Triton"): RMSNorm (forward, backward) and the cross-entropy loss with a
// z-loss term, whose gradient is produced in the same pass over the logits.
//
//   RMSNorm: r = 1 / sqrt(mean_j x_j^2 + eps), y = w * x * r; backward of sum(y * dy), with
//            xh = x * r: dx = r (w dy - xh mean_j(w_j dy_j xh_j)), dw = sum over rows dy * xh.
//   Cross-entropy: lse = log sum_v exp(z_v), loss = lse - z_target + zc lse^2 (a negative target
//            is ignored: loss 0, gradient 0); gradient of scale * loss:
//            dz_v = scale (softmax_v (1 + 2 zc lse) - [v == target]).
//
// Both are bound by HBM: every element is read once (and, for the gradients, written once).
//   RMSNorm: one warp per row (grid-stride), each lane 8 consecutive channels per 16-byte chunk,
//            C chunks (D = 256 C); fp32 sums reduced with shuffles. The backward keeps its dw
//            partial sums in registers for all the rows a warp visits and reduces them per block
//            through shared memory, then once per block into dw.
//   Cross-entropy: one block (256 threads) per row; the row's logits stay in registers as
//            packed bf16 (CPT 16-byte chunks per thread), so max, sum of exponentials, loss and
//            gradient come from one read (the exponentials are taken twice, which the
//            special-function units afford); block reductions through shared memory.
#include <algorithm>
#include <cstdint>

#include "fat_attn_internal.cuh"

namespace fat {
namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}
// An opaque copy: the compiler must assume the value changed, so it converts the packed logits
// again in each pass instead of keeping every converted value live across the passes.
__device__ __forceinline__ uint4 opaque(uint4 v) {
  asm volatile("" : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int C>
__global__ void __launch_bounds__(256) fat_rmsnorm_fwd_kernel(const uint4 *__restrict__ x,
                                                              const float *__restrict__ w,
                                                              float eps, uint4 *__restrict__ y,
                                                              float *__restrict__ rstd,
                                                              long long rows) {
  constexpr int D = 256 * C;
  const int lane = threadIdx.x & 31;
  const long long w0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long row = w0; row < rows; row += nw) {
    float v[C][8];
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      bf16x8_to_f32(x[row * (D / 8) + c * 32 + lane], v[c]);
#pragma unroll
      for (int k = 0; k < 8; ++k) ss = fmaf(v[c][k], v[c][k], ss);
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(ss * (1.0f / D) + eps);
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int ch = (c * 32 + lane) * 8;
      const float4 wa = __ldg(reinterpret_cast<const float4 *>(w + ch));
      const float4 wb = __ldg(reinterpret_cast<const float4 *>(w + ch + 4));
      const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      float o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = wv[k] * (v[c][k] * r);
      y[row * (D / 8) + c * 32 + lane] = f32_to_bf16x8(o);
    }
    if (lane == 0 && rstd != nullptr) rstd[row] = r;
  }
}

template <int C>
__global__ void __launch_bounds__(256) fat_rmsnorm_bwd_kernel(
    const uint4 *__restrict__ x, const float *__restrict__ w, const float *__restrict__ rstd,
    const uint4 *__restrict__ dy, uint4 *__restrict__ dx, float *__restrict__ dw,
    long long rows) {
  constexpr int D = 256 * C;
  extern __shared__ float red[];  // [warps of the block][D] partial dw
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const long long w0 = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  float acc[C][8];
#pragma unroll
  for (int c = 0; c < C; ++c)
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[c][k] = 0.f;
  for (long long row = w0; row < rows; row += nw) {
    const float r = __ldg(rstd + row);
    float xh[C][8], g[C][8];
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int ch = (c * 32 + lane) * 8;
      float dyv[8];
      bf16x8_to_f32(x[row * (D / 8) + c * 32 + lane], xh[c]);
      bf16x8_to_f32(dy[row * (D / 8) + c * 32 + lane], dyv);
      const float4 wa = __ldg(reinterpret_cast<const float4 *>(w + ch));
      const float4 wb = __ldg(reinterpret_cast<const float4 *>(w + ch + 4));
      const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        xh[c][k] *= r;
        g[c][k] = wv[k] * dyv[k];
        s = fmaf(g[c][k], xh[c][k], s);
        acc[c][k] = fmaf(dyv[k], xh[c][k], acc[c][k]);
      }
    }
    const float mean = warp_sum(s) * (1.0f / D);
#pragma unroll
    for (int c = 0; c < C; ++c) {
      float o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = r * (g[c][k] - xh[c][k] * mean);
      dx[row * (D / 8) + c * 32 + lane] = f32_to_bf16x8(o);
    }
  }
  // dw: the block's warps add their partials in shared memory, then one global add per channel
#pragma unroll
  for (int c = 0; c < C; ++c)
#pragma unroll
    for (int k = 0; k < 8; ++k) red[wib * D + (c * 32 + lane) * 8 + k] = acc[c][k];
  __syncthreads();
  const int nwb = blockDim.x >> 5;
  for (int ch = threadIdx.x; ch < D; ch += blockDim.x) {
    float t = 0.f;
    for (int i = 0; i < nwb; ++i) t += red[i * D + ch];
    red_add(dw + ch, t);
  }
}

template <int CPT>
__global__ void __launch_bounds__(256, 2) fat_ce_kernel(const uint4 *__restrict__ z,
                                                     const int32_t *__restrict__ target, int V,
                                                     float zc, float scale,
                                                     float *__restrict__ loss,
                                                     float *__restrict__ lse_out,
                                                     uint4 *__restrict__ dz, long long rows,
                                                     int *err) {
  __shared__ float red[8];
  __shared__ float bc[2];
  const int tid = threadIdx.x, lane = tid & 31, wib = tid >> 5;
  const int n16 = V / 8;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint4 *zr = z + row * n16;
    uint4 raw[CPT];  // the row's logits, packed bf16 (the exponentials are taken twice)
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int i = c * 256 + tid;
      if (i < n16) {
        raw[c] = zr[i];
        float v[8];
        bf16x8_to_f32(raw[c], v);
#pragma unroll
        for (int k = 0; k < 8; ++k) m = fmaxf(m, v[k]);
      }
    }
    m = warp_max(m);
    if (lane == 0) red[wib] = m;
    __syncthreads();
    if (tid < 32) {
      float t = tid < 8 ? red[tid] : -INFINITY;
      t = warp_max(t);
      if (tid == 0) bc[0] = t;
    }
    __syncthreads();
    m = bc[0];
    const float ml = m * kLog2e;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      if (c * 256 + tid < n16) {
        float v[8];
        bf16x8_to_f32(opaque(raw[c]), v);
#pragma unroll
        for (int k = 0; k < 8; ++k) s += ex2(fmaf(v[k], kLog2e, -ml));  // exp(z - max)
      }
    }
    s = warp_sum(s);
    __syncthreads();  // every thread has read bc[0], and warp 0 red[], before they are reused
    if (lane == 0) red[wib] = s;
    __syncthreads();
    if (tid < 32) {
      float t = tid < 8 ? red[tid] : 0.f;
      t = warp_sum(t);
      if (tid == 0) bc[1] = t;
    }
    __syncthreads();
    const float sum = bc[1];
    const float lse = m + __logf(sum);
    const int t = __ldg(target + row);
    const bool valid = t >= 0 && t < V;
    if (tid == 0) {
      if (t >= V) atomicOr(err, FAT_DEVERR_INDEX);
      const float zt =
          valid ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(zr)[t]) : 0.f;
      if (loss != nullptr) loss[row] = valid ? (lse - zt + zc * lse * lse) : 0.f;
      if (lse_out != nullptr) lse_out[row] = lse;
    }
    if (dz != nullptr) {
      // softmax_v = exp(z_v - max) / sum; gradient as above
      const float coef = valid ? scale * (1.0f + 2.0f * zc * lse) / sum : 0.f;
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        const int i = c * 256 + tid;
        if (i < n16) {
          float v[8], o[8];
          bf16x8_to_f32(opaque(raw[c]), v);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            o[k] = coef * ex2(fmaf(v[k], kLog2e, -ml)) - ((valid && 8 * i + k == t) ? scale : 0.f);
          dz[row * n16 + i] = f32_to_bf16x8(o);
        }
      }
    }
    __syncthreads();  // red[] and bc[] are reused by the next row
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int launch_rc(const char *what) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return FAT_OK;
  set_last_error(what, (int)e, cudaGetErrorString(e));
  return FAT_ECUDA;
}

int grid_for(long long units, int per_sm) {
  const int sms = sm_count() > 0 ? sm_count() : 152;
  return (int)std::max<long long>(1, std::min<long long>(units, (long long)sms * per_sm));
}

}  // namespace
}  // namespace fat

using namespace fat;

extern "C" {

int fat_rmsnorm_fwd(long long rows, int dim, const void *x, const float *weight, float eps,
                    void *y, float *rstd, void *stream) {
  if (!x || !weight || !y) return FAT_EINVAL_NULL;
  if (rows < 0 || dim <= 0 || dim % 256 || dim / 256 > 8 || !(eps >= 0.f)) return FAT_EINVAL_SHAPE;
  if (!aligned16(x) || !aligned16(weight) || !aligned16(y)) return FAT_EINVAL_SHAPE;
  if (rows == 0) return FAT_OK;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int blocks = grid_for((rows + 7) / 8, 8);
  const auto *xp = static_cast<const uint4 *>(x);
  auto *yp = static_cast<uint4 *>(y);
  switch (dim / 256) {
#define FAT_CASE(C) \
  case C: fat_rmsnorm_fwd_kernel<C><<<blocks, 256, 0, s>>>(xp, weight, eps, yp, rstd, rows); break;
    FAT_CASE(1) FAT_CASE(2) FAT_CASE(3) FAT_CASE(4) FAT_CASE(5) FAT_CASE(6) FAT_CASE(7) FAT_CASE(8)
#undef FAT_CASE
  }
  return launch_rc("rmsnorm forward launch");
}

int fat_rmsnorm_bwd(long long rows, int dim, const void *x, const float *weight, const float *rstd,
                    const void *dy, void *dx, float *dweight, void *stream) {
  if (!x || !weight || !rstd || !dy || !dx || !dweight) return FAT_EINVAL_NULL;
  if (rows < 0 || dim <= 0 || dim % 256 || dim / 256 > 8) return FAT_EINVAL_SHAPE;
  if (!aligned16(x) || !aligned16(weight) || !aligned16(dy) || !aligned16(dx) ||
      !aligned16(dweight))
    return FAT_EINVAL_SHAPE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(dweight, 0, sizeof(float) * (size_t)dim, s);
  if (e != cudaSuccess) {
    set_last_error("cudaMemsetAsync(dweight)", (int)e, cudaGetErrorString(e));
    return FAT_ECUDA;
  }
  if (rows == 0) return FAT_OK;
  const int blocks = grid_for((rows + 7) / 8, 4);
  const size_t smem = (size_t)8 * dim * sizeof(float);
  const auto *xp = static_cast<const uint4 *>(x);
  const auto *gp = static_cast<const uint4 *>(dy);
  auto *dxp = static_cast<uint4 *>(dx);
  switch (dim / 256) {
#define FAT_CASE(C)                                                                          \
  case C:                                                                                    \
    e = cudaFuncSetAttribute(fat_rmsnorm_bwd_kernel<C>,                                      \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);        \
    if (e == cudaSuccess)                                                                    \
      fat_rmsnorm_bwd_kernel<C><<<blocks, 256, smem, s>>>(xp, weight, rstd, gp, dxp, dweight, \
                                                          rows);                             \
    break;
    FAT_CASE(1) FAT_CASE(2) FAT_CASE(3) FAT_CASE(4) FAT_CASE(5) FAT_CASE(6) FAT_CASE(7) FAT_CASE(8)
#undef FAT_CASE
  }
  if (e != cudaSuccess) {
    set_last_error("cudaFuncSetAttribute(rmsnorm backward)", (int)e, cudaGetErrorString(e));
    return FAT_ECUDA;
  }
  return launch_rc("rmsnorm backward launch");
}

int fat_cross_entropy(long long rows, int vocab, const void *logits, const int32_t *target,
                      float z_loss, float grad_scale, float *loss, float *lse, void *dlogits,
                      void *stream) {
  if (!logits || !target) return FAT_EINVAL_NULL;
  if (rows < 0 || vocab <= 0 || vocab % 8 || vocab > 8 * 256 * 32) return FAT_EINVAL_SHAPE;
  if (!aligned16(logits) || !aligned16(dlogits) || !(z_loss >= 0.f)) return FAT_EINVAL_SHAPE;
  if (rows == 0) return FAT_OK;
  int *err = nullptr;
  int rc = device_error_address(&err);
  if (rc) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n16 = vocab / 8;
  const int cpt = (n16 + 255) / 256;  // 16-byte chunks per thread
  const int blocks = grid_for(rows, 4);
  const auto *zp = static_cast<const uint4 *>(logits);
  auto *dzp = static_cast<uint4 *>(dlogits);
#define FAT_LAUNCH(C) \
  fat_ce_kernel<C><<<blocks, 256, 0, s>>>(zp, target, vocab, z_loss, grad_scale, loss, lse, dzp, rows, err)
  if (cpt <= 1) FAT_LAUNCH(1);
  else if (cpt <= 2) FAT_LAUNCH(2);
  else if (cpt <= 4) FAT_LAUNCH(4);
  else if (cpt <= 8) FAT_LAUNCH(8);
  else if (cpt <= 16) FAT_LAUNCH(16);
  else FAT_LAUNCH(32);
#undef FAT_LAUNCH
  return launch_rc("cross-entropy launch");
}

}  // extern "C"
