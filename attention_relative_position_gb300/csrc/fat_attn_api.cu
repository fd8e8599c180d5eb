// fat_attn_api.cu -- host side of the C ABI declared in include/fat_attn.h: argument checks,
// exact T5 bucket thresholds, tensor-map encoding, the device error word, and kernel launches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <mutex>
#include <vector>

#include "../../include/fat_attn_debug.h"
#include "fat_attn_internal.cuh"

// One error word per GPU that loads the library (file-scope device variable; never allocated).
__device__ int g_fat_device_error;

namespace fat {
namespace {

std::mutex g_mu;
thread_local char g_last_error[256] = "";
long long g_timeout_ns = kDefaultTimeoutNs;
int g_debug_flags = 0;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Address of the current device's error word, looked up on every call (a host-side query that
// allocates nothing), so that no address outlives a context that was torn down.
int device_error_ptr(int **out) {
  void *ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_fat_device_error);
  if (e != cudaSuccess) {
    set_last_error("cudaGetSymbolAddress(error word)", (int)e, cudaGetErrorString(e));
    return FAT_ECUDA;
  }
  *out = static_cast<int *>(ptr);
  return FAT_OK;
}

// ---- exact thresholds: unsigned big integers, base 2^32 ------------------------------------
struct Big {
  std::vector<uint32_t> w;  // little-endian limbs
  explicit Big(uint32_t v) { w.push_back(v); }
  void mul(uint32_t m) {
    uint64_t carry = 0;
    for (auto &x : w) {
      const uint64_t cur = (uint64_t)x * m + carry;
      x = (uint32_t)cur;
      carry = cur >> 32;
    }
    if (carry) w.push_back((uint32_t)carry);
  }
  void trim() {
    while (w.size() > 1 && w.back() == 0) w.pop_back();
  }
};
int big_cmp(Big a, Big b) {
  a.trim();
  b.trim();
  if (a.w.size() != b.w.size()) return a.w.size() < b.w.size() ? -1 : 1;
  for (size_t i = a.w.size(); i-- > 0;)
    if (a.w[i] != b.w[i]) return a.w[i] < b.w[i] ? -1 : 1;
  return 0;
}
// bucket offset of distance n is at least me + t  <=>  n^E * me^t >= md^t * me^E
bool reaches(long long n, int me, int E, int md, int t) {
  Big lhs(1), rhs(1);
  for (int i = 0; i < E; ++i) lhs.mul((uint32_t)n);
  for (int i = 0; i < t; ++i) lhs.mul((uint32_t)me);
  for (int i = 0; i < t; ++i) rhs.mul((uint32_t)md);
  for (int i = 0; i < E; ++i) rhs.mul((uint32_t)me);
  return big_cmp(lhs, rhs) >= 0;
}

int check_buckets(int nb, int md, int bidir, int *nbh_out) {
  if (bidir && (nb % 2)) return FAT_EINVAL_BUCKETS;
  const int nbh = bidir ? nb / 2 : nb;
  if (nbh < 2 || nbh > 128) return FAT_EINVAL_BUCKETS;
  if (md <= nbh / 2) return FAT_EINVAL_BUCKETS;
  *nbh_out = nbh;
  return FAT_OK;
}

int thresholds(int nbh, int md, int32_t *thr, int *count, int *sat) {
  const int me = nbh / 2, E = nbh - me;
  for (int t = 1; t < E; ++t) {
    long long lo = me, hi = md;  // predicate false below the answer, true at md
    while (lo < hi) {
      const long long mid = lo + (hi - lo) / 2;
      if (reaches(mid, me, E, md, t))
        hi = mid;
      else
        lo = mid + 1;
    }
    thr[t - 1] = (int32_t)lo;
  }
  *count = E - 1;
  *sat = E >= 2 ? thr[E - 2] : me;
  return FAT_OK;
}

int fill_bias(BiasParams *b, const float *table, int nb, int md, int bidir, const float *slopes) {
  *b = BiasParams{};
  b->table = table;
  b->slopes = slopes;
  b->has_bias = (table != nullptr) || (slopes != nullptr);
  if (table) {
    int nbh = 0;
    int rc = check_buckets(nb, md, bidir, &nbh);
    if (rc) return rc;
    b->nb = nb;
    b->bidir = bidir ? 1 : 0;
    b->nbh = nbh;
    b->me = nbh / 2;
    int sat = 0;
    thresholds(nbh, md, b->thr, &b->n_thr, &sat);
    b->sat_neg = sat;
    b->sat_pos = bidir ? sat : 0;
  }
  if (b->has_bias) {
    // a tile spans at most 127 + 127 distinct deltas beyond its corner
    b->lut_lo = -b->sat_neg - 253;
    b->lut_len = b->sat_pos + b->sat_neg + 507;
  }
  return FAT_OK;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

int check_shape(const fat_shape_t *sh) {
  if (!sh) return FAT_EINVAL_NULL;
  if (sh->total_tokens < 0 || sh->num_seqs < 0 || sh->max_seqlen < 0 || sh->num_heads <= 0)
    return FAT_EINVAL_SHAPE;
  if (sh->head_dim != 64 && sh->head_dim != 128) return FAT_EINVAL_SHAPE;
  if ((long long)sh->total_tokens * sh->num_heads * sh->head_dim > (1LL << 40)) return FAT_EINVAL_SHAPE;
  if (sh->num_heads > 65535 || sh->num_seqs > 65535) return FAT_EUNSUPPORTED;
  return FAT_OK;
}

int cuda_rc(int e) { return e == 0 ? FAT_OK : FAT_ECUDA; }

}  // namespace

int sm_count() {
  static std::mutex mu;
  static int cached[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      cached[dev] = n;
  }
  return cached[dev];
}

void set_last_error(const char *what, int code, const char *text) {
  snprintf(g_last_error, sizeof g_last_error, "%s: error %d (%s)", what, code, text ? text : "");
}

namespace {
// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda).
bool resolve_encode() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
      set_last_error("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)",
                     e != cudaSuccess ? (int)e : (int)q, cudaGetErrorString(e));
      return false;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return true;
}
}  // namespace

int make_tmap_thd(CUtensorMap *map, const void *ptr, int T, int H, int d, int box_rows) {
  if (!resolve_encode()) return -1;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled", (int)r, "");
    return -1;
  }
  return 0;
}

int make_tmap_thd_f32(CUtensorMap *map, const void *ptr, int T, int H, int d, int box_c,
                      int box_rows) {
  if (!resolve_encode()) return -1;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4};
  const cuuint32_t box[3] = {(cuuint32_t)box_c, 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled(fp32)", (int)r, "");
    return -1;
  }
  return 0;
}

}  // namespace fat

using namespace fat;

// ---- preprocessing and finishing kernels of the backward -----------------------------------
// D[h, t] = sum_c dout[t, h, c] * out[t, h, c] (fp32), the dQ accumulator zeroed, and the
// table gradient zeroed. Memory bound: each lane loads 16 bytes of out and of dout (D/8 lanes per
// (token, head) row, two row groups in flight per thread), and the zeroing is a separate flat
// sweep of 16-byte stores over the accumulator.
template <int D>
__global__ void __launch_bounds__(256) fat_bwd_prep_kernel(const uint4 *__restrict__ out,
                                                           const uint4 *__restrict__ dout,
                                                           float *__restrict__ dvec,
                                                           float4 *__restrict__ dq_acc,
                                                           float *__restrict__ dbias, int nbias,
                                                           int T, int H) {
  grid_dep_wait();    // the forward's outputs are complete (a no-op when launched without overlap)
  grid_dep_launch();  // the main backward grid may be scheduled (it waits for this one's writes)
  constexpr int LPR = D / 8;         // lanes per row, 8 bf16 each
  constexpr int RPW = 32 / LPR;      // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, part = lane % LPR;
  const long long nrows = (long long)T * H;
  const long long gtid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long warp0 = gtid >> 5, nwarps = nthreads >> 5;
  if (dbias && warp0 == 0)
    for (int i = lane; i < nbias; i += 32) dbias[i] = 0.f;
  auto dot8 = [](uint4 a, uint4 b) {
    const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&b);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(a2[i]), y = __bfloat1622float2(b2[i]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
    return acc;
  };
  // Row groups of RPW rows; each warp takes two groups per step so that four 16-byte loads per
  // lane are in flight.
  const long long ngroups = (nrows + RPW - 1) / RPW;
  for (long long g = warp0 * 2; g < ngroups; g += nwarps * 2) {
    const long long r0 = g * RPW + sub, r1 = (g + 1) * RPW + sub;
    const bool v0 = r0 < nrows, v1 = r1 < nrows;
    uint4 a0 = make_uint4(0, 0, 0, 0), b0 = a0, a1 = a0, b1 = a0;
    if (v0) { a0 = out[r0 * LPR + part]; b0 = dout[r0 * LPR + part]; }
    if (v1) { a1 = out[r1 * LPR + part]; b1 = dout[r1 * LPR + part]; }
    float s0 = dot8(a0, b0), s1 = dot8(a1, b1);
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
    }
    if (part == 0) {
      if (v0) dvec[(r0 % H) * (long long)T + r0 / H] = s0;
      if (v1) dvec[(r1 % H) * (long long)T + r1 / H] = s1;
    }
  }
  const long long n4 = nrows * (D / 4);
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  long long i = gtid;
  for (; i + 3 * nthreads < n4; i += 4 * nthreads) {
    dq_acc[i] = z;
    dq_acc[i + nthreads] = z;
    dq_acc[i + 2 * nthreads] = z;
    dq_acc[i + 3 * nthreads] = z;
  }
  for (; i < n4; i += nthreads) dq_acc[i] = z;
}

// dq = bf16(dq_acc * softmax_scale): eight accumulator values in, one 16-byte store out per
// thread step; n8 = element count / 8 (the element count is a multiple of 64).
__global__ void __launch_bounds__(256) fat_bwd_finish_kernel(const float4 *__restrict__ acc,
                                                             uint4 *__restrict__ dq, float scale,
                                                             long long n8) {
  grid_dep_wait();  // the accumulator is complete (a no-op when launched without overlap)
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  auto cvt = [scale](float4 a, float4 b) {
    uint4 o;
    o.x = pack_bf16x2(a.x * scale, a.y * scale);
    o.y = pack_bf16x2(a.z * scale, a.w * scale);
    o.z = pack_bf16x2(b.x * scale, b.y * scale);
    o.w = pack_bf16x2(b.z * scale, b.w * scale);
    return o;
  };
  for (; i + nthreads < n8; i += 2 * nthreads) {
    const float4 a0 = acc[2 * i], b0 = acc[2 * i + 1];
    const float4 a1 = acc[2 * (i + nthreads)], b1 = acc[2 * (i + nthreads) + 1];
    dq[i] = cvt(a0, b0);
    dq[i + nthreads] = cvt(a1, b1);
  }
  if (i < n8) dq[i] = cvt(acc[2 * i], acc[2 * i + 1]);
}

// ---- C ABI -------------------------------------------------------------------------------------
extern "C" {

const char *fat_attn_last_error_message(void) { return g_last_error; }

const char *fat_attn_strerror(int code) {
  switch (code) {
    case FAT_OK: return "ok";
    case FAT_EINVAL_NULL: return "a required pointer is NULL";
    case FAT_EINVAL_SHAPE: return "invalid shape, head_dim or pointer alignment";
    case FAT_EINVAL_BUCKETS: return "invalid T5 bucket arguments";
    case FAT_ECUDA: return "a CUDA call failed";
    case FAT_EUNSUPPORTED: return "unsupported argument combination";
    case FAT_EDEVICE: return "the device error word was set";
    default: return "unknown error code";
  }
}

int fat_attn_bucket_thresholds(int num_buckets, int max_distance, int bidirectional,
                               int32_t *thr, int *count, int *saturation) {
  if (!thr || !count || !saturation) return FAT_EINVAL_NULL;
  int nbh = 0;
  int rc = check_buckets(num_buckets, max_distance, bidirectional, &nbh);
  if (rc) return rc;
  return thresholds(nbh, max_distance, thr, count, saturation);
}

void fat_attn_debug_set_watchdog(long long timeout_ns, int flags) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timeout_ns = timeout_ns > 0 ? timeout_ns : kDefaultTimeoutNs;
  g_debug_flags = flags;
}

int fat_attn_get_device_error(void *stream, int *bits) {
  int *ep = nullptr;
  int rc = device_error_ptr(&ep);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FAT_ECUDA;
  if (cudaMemcpyAsync(&host, ep, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FAT_ECUDA;
  if (cudaMemsetAsync(ep, 0, sizeof(int), s) != cudaSuccess) return FAT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FAT_ECUDA;
  if (bits) *bits = host;
  return host ? FAT_EDEVICE : FAT_OK;
}

int fat_attn_fwd(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                 const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                 const float *alibi_slopes, const int32_t *cu_seqlens, int causal,
                 float softmax_scale, void *out, float *lse) {
  int rc = check_shape(sh);
  if (rc) return rc;
  if (!q || !k || !v || !cu_seqlens || !out) return FAT_EINVAL_NULL;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) ||
      misaligned(cu_seqlens) || misaligned(bias_table) || misaligned(alibi_slopes) ||
      misaligned(lse))
    return FAT_EINVAL_SHAPE;
  FwdParams p{};
  rc = fill_bias(&p.bias, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes);
  if (rc) return rc;
  if (fwd_smem_bytes(sh->head_dim, p.bias.lut_len) > (size_t)kSmemLimit) return FAT_EUNSUPPORTED;
  if (sh->total_tokens == 0 || sh->num_seqs == 0 || sh->max_seqlen == 0) return FAT_OK;
  rc = device_error_ptr(&p.err);
  if (rc) return rc;
  p.seq = SeqParams{cu_seqlens, sh->num_seqs, sh->num_heads, sh->total_tokens, sh->max_seqlen};
  p.causal = causal ? 1 : 0;
  p.scale_log2 = softmax_scale * kLog2e;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.lse = lse;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    p.timeout_ns = g_timeout_ns;
    p.debug_flags = g_debug_flags;
  }
  return cuda_rc(launch_fwd(p, sh->head_dim, sh->max_seqlen, q, k, v,
                            static_cast<cudaStream_t>(sh->stream)));
}

size_t fat_attn_bwd_workspace_size(const fat_shape_t *sh) {
  if (check_shape(sh)) return 0;
  const size_t T = (size_t)sh->total_tokens, H = (size_t)sh->num_heads, d = (size_t)sh->head_dim;
  const size_t a = (T * H * d * 4 + 255) & ~(size_t)255;
  const size_t b = (T * H * 4 + 255) & ~(size_t)255;
  return a + b;
}

namespace {
struct WorkspaceView {
  float *dq_acc;
  float *dvec;
};
int check_workspace(const fat_shape_t *sh, const void *ws, size_t bytes, WorkspaceView *view) {
  const size_t need = fat_attn_bwd_workspace_size(sh);
  if (!ws && need) return FAT_EINVAL_NULL;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return FAT_EINVAL_SHAPE;
  if (bytes < need) return FAT_EINVAL_SHAPE;
  const size_t T = (size_t)sh->total_tokens, H = (size_t)sh->num_heads, d = (size_t)sh->head_dim;
  view->dq_acc = static_cast<float *>(const_cast<void *>(ws));
  view->dvec = reinterpret_cast<float *>(static_cast<char *>(const_cast<void *>(ws)) +
                                         ((T * H * d * 4 + 255) & ~(size_t)255));
  return FAT_OK;
}
bool empty_problem(const fat_shape_t *sh) {
  return sh->total_tokens == 0 || sh->num_seqs == 0 || sh->max_seqlen == 0;
}
int launch_rc(const char *what) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return FAT_OK;
  set_last_error(what, (int)e, cudaGetErrorString(e));
  return FAT_ECUDA;
}
}  // namespace

namespace {
int bwd_preprocess_impl(const fat_shape_t *sh, const void *out, const void *dout, void *workspace,
                        size_t workspace_bytes, float *dbias_table, int num_buckets,
                        bool overlap_previous) {
  int rc = check_shape(sh);
  if (rc) return rc;
  if (!out || !dout) return FAT_EINVAL_NULL;
  if (misaligned(out) || misaligned(dout) || misaligned(dbias_table)) return FAT_EINVAL_SHAPE;
  if (dbias_table && (num_buckets < 2 || num_buckets > 256)) return FAT_EINVAL_BUCKETS;
  WorkspaceView ws{};
  rc = check_workspace(sh, workspace, workspace_bytes, &ws);
  if (rc) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(sh->stream);
  const int T = sh->total_tokens, H = sh->num_heads, d = sh->head_dim;
  const int nbias = dbias_table ? num_buckets * H : 0;
  if (T == 0) {
    if (!nbias) return FAT_OK;
    const cudaError_t e = cudaMemsetAsync(dbias_table, 0, sizeof(float) * nbias, stream);
    if (e != cudaSuccess) set_last_error("cudaMemsetAsync(dbias_table)", (int)e, cudaGetErrorString(e));
    return cuda_rc((int)e);
  }
  const long long rows = (long long)T * H;
  // Enough warps for every (token, head) row group, at most eight 256-thread blocks per SM.
  const int blocks = (int)std::min<long long>((rows + 63) / 64, 152LL * 8);
  const auto *o = static_cast<const uint4 *>(out);
  const auto *g = static_cast<const uint4 *>(dout);
  float4 *acc4 = reinterpret_cast<float4 *>(ws.dq_acc);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  if (overlap_previous) {  // it waits for the previous grid before touching memory
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e =
      d == 64 ? cudaLaunchKernelEx(&cfg, fat_bwd_prep_kernel<64>, o, g, ws.dvec, acc4, dbias_table,
                                   nbias, T, H)
              : cudaLaunchKernelEx(&cfg, fat_bwd_prep_kernel<128>, o, g, ws.dvec, acc4,
                                   dbias_table, nbias, T, H);
  if (e != cudaSuccess) {
    set_last_error("backward preprocess launch", (int)e, cudaGetErrorString(e));
    return FAT_ECUDA;
  }
  return launch_rc("backward preprocess launch");
}
}  // namespace

int fat_attn_bwd_preprocess(const fat_shape_t *sh, const void *out, const void *dout,
                            void *workspace, size_t workspace_bytes, float *dbias_table,
                            int num_buckets) {
  return bwd_preprocess_impl(sh, out, dout, workspace, workspace_bytes, dbias_table, num_buckets,
                             false);
}

namespace {
int bwd_main_impl(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                  const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                  const float *alibi_slopes, const int32_t *cu_seqlens, int causal,
                  float softmax_scale, const float *lse, const void *dout, void *workspace,
                  size_t workspace_bytes, void *dk, void *dv, float *dbias_table,
                  bool overlap_previous) {
  int rc = check_shape(sh);
  if (rc) return rc;
  if (!q || !k || !v || !cu_seqlens || !lse || !dout || !dk || !dv) return FAT_EINVAL_NULL;
  if (dbias_table && !bias_table) return FAT_EUNSUPPORTED;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(dout) || misaligned(dk) ||
      misaligned(dv) || misaligned(lse) || misaligned(cu_seqlens) || misaligned(bias_table) ||
      misaligned(alibi_slopes) || misaligned(dbias_table))
    return FAT_EINVAL_SHAPE;
  BwdParams p{};
  rc = fill_bias(&p.bias, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes);
  if (rc) return rc;
  if (bwd_smem_bytes(sh->head_dim, p.bias.lut_len) > (size_t)kSmemLimit) return FAT_EUNSUPPORTED;
  WorkspaceView ws{};
  rc = check_workspace(sh, workspace, workspace_bytes, &ws);
  if (rc) return rc;
  if (empty_problem(sh)) return FAT_OK;
  rc = device_error_ptr(&p.err);
  if (rc) return rc;
  p.seq = SeqParams{cu_seqlens, sh->num_seqs, sh->num_heads, sh->total_tokens, sh->max_seqlen};
  p.causal = causal ? 1 : 0;
  p.scale_log2 = softmax_scale * kLog2e;
  p.scale = softmax_scale;
  p.lse = lse;
  p.dvec = ws.dvec;
  p.dq_acc = ws.dq_acc;
  p.dk = static_cast<__nv_bfloat16 *>(dk);
  p.dv = static_cast<__nv_bfloat16 *>(dv);
  p.dbias = dbias_table;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    p.timeout_ns = g_timeout_ns;
    p.debug_flags = g_debug_flags;
  }
  return cuda_rc(launch_bwd(p, sh->head_dim, sh->max_seqlen, q, k, v, nullptr, dout,
                           static_cast<cudaStream_t>(sh->stream), overlap_previous));
}

int bwd_finalize_impl(const fat_shape_t *sh, const void *workspace, size_t workspace_bytes,
                      float softmax_scale, void *dq, bool overlap_previous) {
  int rc = check_shape(sh);
  if (rc) return rc;
  if (!dq) return FAT_EINVAL_NULL;
  if (misaligned(dq)) return FAT_EINVAL_SHAPE;
  WorkspaceView ws{};
  rc = check_workspace(sh, workspace, workspace_bytes, &ws);
  if (rc) return rc;
  const long long n8 = (long long)sh->total_tokens * sh->num_heads * sh->head_dim / 8;
  if (n8 == 0) return FAT_OK;
  const int blocks = (int)std::min<long long>((n8 + 255) / 256, 152LL * 8);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(sh->stream);
  if (overlap_previous) {  // programmatic dependent launch on the main backward grid
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fat_bwd_finish_kernel,
                                           reinterpret_cast<const float4 *>(ws.dq_acc),
                                           static_cast<uint4 *>(dq), softmax_scale, n8);
  if (e != cudaSuccess) {
    set_last_error("backward finalize launch", (int)e, cudaGetErrorString(e));
    return FAT_ECUDA;
  }
  return launch_rc("backward finalize launch");
}
}  // namespace

int fat_attn_bwd_main(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                      const float *bias_table, int num_buckets, int max_distance,
                      int bidirectional, const float *alibi_slopes, const int32_t *cu_seqlens,
                      int causal, float softmax_scale, const float *lse, const void *dout,
                      void *workspace, size_t workspace_bytes, void *dk, void *dv,
                      float *dbias_table) {
  return bwd_main_impl(sh, q, k, v, bias_table, num_buckets, max_distance, bidirectional,
                       alibi_slopes, cu_seqlens, causal, softmax_scale, lse, dout, workspace,
                       workspace_bytes, dk, dv, dbias_table, false);
}

int fat_attn_bwd_finalize(const fat_shape_t *sh, const void *workspace, size_t workspace_bytes,
                          float softmax_scale, void *dq) {
  return bwd_finalize_impl(sh, workspace, workspace_bytes, softmax_scale, dq, false);
}

}  // extern "C"

namespace fat {
int check_bwd_args(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                   const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                   const float *alibi_slopes, const int32_t *cu_seqlens, const void *out,
                   const float *lse, const void *dout, const void *dq, const void *dk,
                   const void *dv, const float *dbias_table) {
  int rc = check_shape(sh);
  if (rc) return rc;
  if (!q || !k || !v || !cu_seqlens || !out || !lse || !dout || !dq || !dk || !dv)
    return FAT_EINVAL_NULL;
  if (dbias_table && !bias_table) return FAT_EUNSUPPORTED;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(dout) ||
      misaligned(dq) || misaligned(dk) || misaligned(dv) || misaligned(lse) ||
      misaligned(cu_seqlens) || misaligned(bias_table) || misaligned(alibi_slopes) ||
      misaligned(dbias_table))
    return FAT_EINVAL_SHAPE;
  BiasParams b{};
  rc = fill_bias(&b, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes);
  if (rc) return rc;
  if (bwd_smem_bytes(sh->head_dim, b.lut_len) > (size_t)kSmemLimit) return FAT_EUNSUPPORTED;
  return FAT_OK;
}
}  // namespace fat

extern "C" {

int fat_attn_bwd(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                 const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                 const float *alibi_slopes, const int32_t *cu_seqlens, int causal,
                 float softmax_scale, const void *out, const float *lse, const void *dout,
                 void *workspace, size_t workspace_bytes, void *dq, void *dk, void *dv,
                 float *dbias_table) {
  // validate everything before enqueueing anything
  int rc = check_bwd_args(sh, q, k, v, bias_table, num_buckets, max_distance, bidirectional,
                          alibi_slopes, cu_seqlens, out, lse, dout, dq, dk, dv, dbias_table);
  if (rc) return rc;
  {
    WorkspaceView ws{};
    rc = check_workspace(sh, workspace, workspace_bytes, &ws);
    if (rc) return rc;
  }
  rc = bwd_preprocess_impl(sh, out, dout, workspace, workspace_bytes, dbias_table, num_buckets,
                           true);
  if (rc) return rc;
  // All three grids are launched as programmatic dependents of the grid before them: each is
  // scheduled while that grid drains and waits for its writes in-kernel (the preprocessing grid
  // before it touches memory; the main grid before it reads D or touches the accumulators).
  rc = bwd_main_impl(sh, q, k, v, bias_table, num_buckets, max_distance, bidirectional,
                     alibi_slopes, cu_seqlens, causal, softmax_scale, lse, dout, workspace,
                     workspace_bytes, dk, dv, dbias_table, true);
  if (rc) return rc;
  return bwd_finalize_impl(sh, workspace, workspace_bytes, softmax_scale, dq, true);
}

int fat_attn_debug_buckets(long long delta_lo, int n, int num_buckets, int max_distance,
                           int bidirectional, int32_t *out_dev, void *stream) {
  if (!out_dev) return FAT_EINVAL_NULL;
  if (n < 0) return FAT_EINVAL_SHAPE;
  if (delta_lo < -(1LL << 30) || delta_lo + n > (1LL << 30)) return FAT_EINVAL_SHAPE;
  BiasParams b{};
  static const float dummy = 0.f;
  int rc = fill_bias(&b, &dummy, num_buckets, max_distance, bidirectional, nullptr);
  if (rc) return rc;
  if (n == 0) return FAT_OK;
  return cuda_rc(launch_debug_buckets(b, delta_lo, n, out_dev, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace fat {
__global__ void fat_debug_buckets_kernel(const BiasParams b, long long lo, int n, int32_t *out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = t5_bucket_dev((int)(lo + i), b);
}
int launch_debug_buckets(const BiasParams &b, long long lo, int n, int32_t *out,
                         cudaStream_t stream) {
  fat_debug_buckets_kernel<<<(n + 255) / 256, 256, 0, stream>>>(b, lo, n, out);
  return (int)cudaGetLastError();
}
}  // namespace fat
