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

int thresholds_exact(int nbh, int md, int32_t *thr, int *count, int *sat) {
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

// The thresholds depend on (buckets per side, max distance) only, and their exact big-integer
// search costs tens of microseconds of host time: computed once per pair and kept (a few
// entries, replaced in turn), so a call pays a lookup.
int thresholds(int nbh, int md, int32_t *thr, int *count, int *sat) {
  struct Entry {
    int nbh, md, count, sat;
    int32_t thr[kMaxThresholds];
  };
  constexpr int kEntries = 16;
  static Entry cache[kEntries];
  static int used = 0, next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].nbh == nbh && cache[i].md == md) {
        std::copy(cache[i].thr, cache[i].thr + cache[i].count, thr);
        *count = cache[i].count;
        *sat = cache[i].sat;
        return FAT_OK;
      }
  }
  Entry e{};
  e.nbh = nbh;
  e.md = md;
  const int rc = thresholds_exact(nbh, md, e.thr, &e.count, &e.sat);
  if (rc) return rc;
  std::copy(e.thr, e.thr + e.count, thr);
  *count = e.count;
  *sat = e.sat;
  std::lock_guard<std::mutex> lk(mu);
  cache[next] = e;
  next = (next + 1) % kEntries;
  used = used < kEntries ? used + 1 : used;
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

int device_error_address(int **out) { return device_error_ptr(out); }

// Per (kernel, device): the largest dynamic shared-memory size already allowed, and whether the
// compiled register count times the block size holds the kernel's register re-balancing.
// Launchers call this before every launch; only the first call per size does any CUDA work.
int prepare_kernel(const void *fn, size_t smem, int nthreads, int regs_needed) {
  struct Entry {
    const void *fn;
    int dev;
    size_t smem;
    bool regs_ok;
  };
  static std::mutex mu;
  static Entry tab[256];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  std::lock_guard<std::mutex> lk(mu);
  Entry *en = nullptr;
  for (int i = 0; i < used; ++i)
    if (tab[i].fn == fn && tab[i].dev == dev) en = &tab[i];
  if (en && en->smem >= smem && en->regs_ok) return 0;
  if (!en) {
    if (used == 256) used = 0;  // more kernels x devices than any build has: start over
    en = &tab[used++];
    *en = Entry{fn, dev, 0, false};
  }
  if (!en->regs_ok) {
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) {
      set_last_error("cudaFuncGetAttributes", (int)e, cudaGetErrorString(e));
      return (int)e;
    }
    if (fa.numRegs * nthreads < regs_needed) {
      set_last_error("kernel register pool smaller than its warp-role split", fa.numRegs,
                     "no launch");
      return (int)cudaErrorInvalidConfiguration;
    }
    en->regs_ok = true;
  }
  if (en->smem < smem) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
      set_last_error("cudaFuncSetAttribute(max dynamic shared memory)", (int)e,
                     cudaGetErrorString(e));
      return (int)e;
    }
    en->smem = smem;
  }
  return 0;
}

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

int max_pair_ctas(const void *fn, size_t smem, int nthreads) {
  struct Entry {
    const void *fn;
    int dev;
    size_t smem;
    int ctas;
  };
  static std::mutex mu;
  static Entry tab[32];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < used; ++i)
    if (tab[i].fn == fn && tab[i].dev == dev && tab[i].smem == smem) return tab[i].ctas;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(nthreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();  // this query's own error: the caller launches without clusters
    n = 0;
  }
  if (used == 32) used = 0;
  tab[used++] = Entry{fn, dev, smem, 2 * n};
  return 2 * n;
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

namespace {
// Encoded tensor maps, keyed by everything they encode (address, sizes, box, element type), so a
// hit is byte-for-byte the map a fresh encode would give: no entry can go stale. Replacement is
// round-robin over 128 entries.
struct TmapKey {
  const void *ptr;
  int T, H, d, box_c, box_rows, fp32;
  bool operator==(const TmapKey &o) const {
    return ptr == o.ptr && T == o.T && H == o.H && d == o.d && box_c == o.box_c &&
           box_rows == o.box_rows && fp32 == o.fp32;
  }
};
constexpr int kTmapCache = 128;
std::mutex g_tmap_mu;
TmapKey g_tmap_key[kTmapCache];
CUtensorMap g_tmap_val[kTmapCache];
int g_tmap_used = 0, g_tmap_next = 0;

bool tmap_lookup(const TmapKey &k, CUtensorMap *map) {
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  for (int i = 0; i < g_tmap_used; ++i)
    if (g_tmap_key[i] == k) {
      *map = g_tmap_val[i];
      return true;
    }
  return false;
}
void tmap_store(const TmapKey &k, const CUtensorMap &map) {
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  const int i = g_tmap_used < kTmapCache ? g_tmap_used++ : (g_tmap_next++ % kTmapCache);
  g_tmap_key[i] = k;
  g_tmap_val[i] = map;
}
}  // namespace

int make_tmap_thd(CUtensorMap *map, const void *ptr, int T, int H, int d, int box_rows) {
  const TmapKey key{ptr, T, H, d, 64, box_rows, 0};
  if (tmap_lookup(key, map)) return 0;
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
  tmap_store(key, *map);
  return 0;
}

int make_tmap_thd_f32(CUtensorMap *map, const void *ptr, int T, int H, int d, int box_c,
                      int box_rows) {
  const TmapKey key{ptr, T, H, d, box_c, box_rows, 1};
  if (tmap_lookup(key, map)) return 0;
  if (!resolve_encode()) return -1;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4};
  const cuuint32_t box[3] = {(cuuint32_t)box_c, 1, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_c * 4 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled(fp32)", (int)r, "");
    return -1;
  }
  tmap_store(key, *map);
  return 0;
}

}  // namespace fat

using namespace fat;

// ---- preprocessing and finishing kernels of the backward -----------------------------------
// D[h, t] = sum_c dout[t, h, c] * out[t, h, c] (fp32), the fp32 accumulators zeroed (dQ, and
// dK, dV when query heads share key/value heads: one contiguous region of n4_zero float4), and
// the table gradient zeroed. Memory bound: each lane loads 16 bytes of out and of dout (D/8
// lanes per (token, head) row, two row groups in flight per thread), and the zeroing is a
// separate flat sweep of 16-byte stores.
template <int D>
__global__ void __launch_bounds__(256) fat_bwd_prep_kernel(const uint4 *__restrict__ out,
                                                           const uint4 *__restrict__ dout,
                                                           float *__restrict__ dvec,
                                                           float4 *__restrict__ acc,
                                                           long long n4_zero,
                                                           float4 *__restrict__ acc2,
                                                           long long n4_zero2,
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
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(a2[i]), y = __bfloat1622float2(b2[i]);
      s = fmaf(x.x, y.x, s);
      s = fmaf(x.y, y.y, s);
    }
    return s;
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
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  long long i = gtid;
  for (; i + 3 * nthreads < n4_zero; i += 4 * nthreads) {
    acc[i] = z;
    acc[i + nthreads] = z;
    acc[i + 2 * nthreads] = z;
    acc[i + 3 * nthreads] = z;
  }
  for (; i < n4_zero; i += nthreads) acc[i] = z;
  for (i = gtid; i < n4_zero2; i += nthreads) acc2[i] = z;
}

// out = bf16(acc * scale) over up to three segments (dQ; dK and dV when query heads share
// key/value heads): eight accumulator values in, one 16-byte store out per thread step; each
// segment's n8 = element count / 8 (element counts are multiples of 64).
struct FinishSegs {
  const float4 *acc[3];
  uint4 *out[3];
  float scale[3];
  long long n8[3];
  int nseg;
  // split last wave of the backward (documents of equal length Lk): tail CTA c holds the dK,
  // dV rows of key tile (tail_first + c) % nkb, head ((tail_first + c) / nkb) % H, document
  // (tail_first + c) / (nkb H), as [c][dK, dV][128][d] fp32 (dK already scaled)
  const float4 *tail_acc;
  uint4 *tail_dk, *tail_dv;
  long long tail_first;
  int ntail, nkb, H, d8, Lk;
};
__global__ void __launch_bounds__(256) fat_bwd_finish_kernel(const FinishSegs f) {
  grid_dep_wait();  // the accumulators are complete (a no-op when launched without overlap)
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (int sg = 0; sg < f.nseg; ++sg) {
    const float4 *acc = f.acc[sg];
    uint4 *dq = f.out[sg];
    const float scale = f.scale[sg];
    const long long n8 = f.n8[sg];
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
  const long long ntail8 = (long long)f.ntail * 2 * 128 * f.d8;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < ntail8;
       i += nthreads) {
    const int c8 = (int)(i % f.d8);
    const long long rest = i / f.d8;
    const int row = (int)(rest % 128);
    const int which = (int)((rest / 128) % 2);
    const long long c = rest / 256;
    const long long cta = f.tail_first + c;
    const int kb = (int)(cta % f.nkb), h = (int)((cta / f.nkb) % f.H);
    const long long doc = cta / ((long long)f.nkb * f.H);
    const int krow = kb * 128 + row;
    if (krow >= f.Lk) continue;
    const float4 *src = f.tail_acc + 2 * i;  // [c][which][row][d / 4], c8-th pair of float4
    uint4 o;
    const float4 a = src[0], b = src[1];
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    uint4 *dst = which ? f.tail_dv : f.tail_dk;
    dst[((doc * f.Lk + krow) * f.H + h) * f.d8 + c8] = o;
  }
}

// dK = dV = 0 for the keys of documents without queries (cross-attention): no backward item
// covers them. One block per document; the others exit at once.
__global__ void __launch_bounds__(256) fat_zero_unseen_keys_kernel(const int32_t *cu_q,
                                                                   const int32_t *cu_k, int Tk,
                                                                   int row_elems, uint4 *dk,
                                                                   uint4 *dv) {
  const int doc = blockIdx.x;
  const int q0 = __ldg(cu_q + doc), q1 = __ldg(cu_q + doc + 1);
  const int k0 = __ldg(cu_k + doc), k1 = __ldg(cu_k + doc + 1);
  if (q1 != q0 || k0 < 0 || k1 > Tk || k1 <= k0) return;
  const long long n16 = (long long)(k1 - k0) * row_elems / 8;  // 16-byte units
  const long long base = (long long)k0 * row_elems / 8;
  for (long long i = threadIdx.x; i < n16; i += blockDim.x) {
    dk[base + i] = make_uint4(0u, 0u, 0u, 0u);
    dv[base + i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---- the generalised problem every entry point is lowered to ------------------------------
namespace fat {
namespace {

struct XShape {
  int Tq, Tk, n, maxq, maxk, Hq, Hkv, d;
  cudaStream_t stream;
};

int to_xshape(const fat_shape_t *sh, XShape *x) {
  int rc = check_shape(sh);
  if (rc) return rc;
  *x = XShape{sh->total_tokens, sh->total_tokens, sh->num_seqs, sh->max_seqlen, sh->max_seqlen,
              sh->num_heads, sh->num_heads, sh->head_dim, static_cast<cudaStream_t>(sh->stream)};
  return FAT_OK;
}

int to_xshape(const fat_xshape_t *xs, XShape *x) {
  if (!xs) return FAT_EINVAL_NULL;
  if (xs->total_q < 0 || xs->total_k < 0 || xs->num_seqs < 0 || xs->max_seqlen_q < 0 ||
      xs->max_seqlen_k < 0 || xs->num_heads_q <= 0 || xs->num_heads_kv <= 0 ||
      xs->num_heads_q % xs->num_heads_kv != 0)
    return FAT_EINVAL_SHAPE;
  if (xs->head_dim != 64 && xs->head_dim != 128) return FAT_EINVAL_SHAPE;
  if ((long long)xs->total_q * xs->num_heads_q * xs->head_dim > (1LL << 40) ||
      (long long)xs->total_k * xs->num_heads_kv * xs->head_dim > (1LL << 40))
    return FAT_EINVAL_SHAPE;
  if (xs->num_heads_q > 65535 || xs->num_seqs > 65535) return FAT_EUNSUPPORTED;
  *x = XShape{xs->total_q, xs->total_k, xs->num_seqs, xs->max_seqlen_q, xs->max_seqlen_k,
              xs->num_heads_q, xs->num_heads_kv, xs->head_dim,
              static_cast<cudaStream_t>(xs->stream)};
  return FAT_OK;
}

SeqParams seq_params(const XShape &x, const int32_t *cu_q, const int32_t *cu_k) {
  SeqParams s{};
  s.cu_seqlens = cu_q;
  s.cu_seqlens_k = cu_k;
  s.num_seqs = x.n;
  s.num_heads = x.Hq;
  s.total_tokens = x.Tq;
  s.max_seqlen = x.maxq;
  s.num_heads_kv = x.Hkv;
  s.total_k = x.Tk;
  s.max_seqlen_k = x.maxk;
  s.group = x.Hq / x.Hkv;
  return s;
}

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// Split last wave of the backward's one-CTA-per-key-tile grid. When every document has the same
// length (sum of lengths = documents x bound) and the grid is not a whole number of waves of
// one CTA per SM, the CTAs of the partial last wave (at most half a wave) are each split into
// `splits` CTAs that share the key tile's query tiles, so that wave takes 1/splits of the time.
// (Used only without the causal mask, where every CTA carries the same work.)
struct TailPlan {
  long long first;  // id of the first split CTA
  int splits, ntail;
};
TailPlan bwd_tail_plan(const XShape &x) {
  TailPlan t{0, 0, 0};
  if (x.n <= 0 || x.maxq <= 0 || x.maxk <= 0 || !bwd_uses_tiles(x.d, x.maxk)) return t;
  if ((long long)x.n * x.maxq != x.Tq || (long long)x.n * x.maxk != x.Tk) return t;
  const int sms = sm_count();
  if (sms <= 0) return t;
  const long long items = (long long)((x.maxk + 127) / 128) * x.Hq * x.n;
  const long long whole = items / sms * sms, ntail = items - whole;
  const int bq = bwd_query_tile(x.d);
  const int nq = (x.maxq + bq - 1) / bq;
  if (ntail == 0 || ntail > sms / 2) return t;
  const int splits = (int)std::min<long long>(sms / ntail, nq / 2);
  if (splits < 2) return t;
  t.first = whole;
  t.splits = splits;
  t.ntail = (int)ntail;
  return t;
}

// Backward workspace: fp32 dQ accumulator [Tq, Hq, d]; when query heads share key/value heads,
// fp32 dK and dV accumulators [Tk, Hkv, d]; then D [Hq, Tq] (this prefix is the minimum a call
// accepts). When the shape has a split last wave (bwd_tail_plan) and its own key/value heads,
// the size reported adds fp32 dK and dV rows of those key tiles [tail CTA][2][128][d], used
// when the caller's workspace holds them. Each part 256-byte aligned; the preprocess zeroes the
// accumulators.
struct WsLayout {
  size_t dk, dv, dvec, base_total, tail, total;
};
WsLayout ws_layout(const XShape &x) {
  WsLayout l{};
  const size_t a = align256((size_t)x.Tq * x.Hq * x.d * 4);
  const size_t b = x.Hq != x.Hkv ? align256((size_t)x.Tk * x.Hkv * x.d * 4) : 0;
  const TailPlan t = x.Hq == x.Hkv ? bwd_tail_plan(x) : TailPlan{0, 0, 0};
  l.dk = a;
  l.dv = a + b;
  l.dvec = a + 2 * b;
  l.base_total = l.dvec + align256((size_t)x.Tq * x.Hq * 4);
  l.tail = l.base_total;
  l.total = l.tail + align256((size_t)t.ntail * 2 * 128 * x.d * 4);
  return l;
}

struct WorkspaceView {
  float *dq_acc, *dk_acc, *dv_acc, *tail_acc, *dvec;
  size_t zero_bytes, tail_bytes;  // accumulators to zero: [0, zero_bytes), tail_acc
};
int check_workspace(const XShape &x, const void *ws, size_t bytes, WorkspaceView *view) {
  const WsLayout l = ws_layout(x);
  if (!ws && l.base_total) return FAT_EINVAL_NULL;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return FAT_EINVAL_SHAPE;
  if (bytes < l.base_total) return FAT_EINVAL_SHAPE;
  char *base = static_cast<char *>(const_cast<void *>(ws));
  view->dq_acc = reinterpret_cast<float *>(base);
  view->dk_acc = x.Hq != x.Hkv ? reinterpret_cast<float *>(base + l.dk) : nullptr;
  view->dv_acc = x.Hq != x.Hkv ? reinterpret_cast<float *>(base + l.dv) : nullptr;
  const bool tail = l.total > l.tail && bytes >= l.total;
  view->tail_acc = tail ? reinterpret_cast<float *>(base + l.tail) : nullptr;
  view->tail_bytes = tail ? l.total - l.tail : 0;
  view->dvec = reinterpret_cast<float *>(base + l.dvec);
  view->zero_bytes = l.dvec;
  return FAT_OK;
}

int launch_rc(const char *what) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return FAT_OK;
  set_last_error(what, (int)e, cudaGetErrorString(e));
  return FAT_ECUDA;
}

void fill_runtime_knobs(long long *timeout_ns, int *debug_flags) {
  std::lock_guard<std::mutex> lk(g_mu);
  *timeout_ns = g_timeout_ns;
  *debug_flags = g_debug_flags;
}

// Split-key forward workspace: normalised partial outputs fp32 [splits, Tq, Hq, d], then
// partial lse fp32 [splits, Hq, Tq], each 256-byte aligned.
size_t splitkv_bytes(const XShape &x, int splits) {
  return align256((size_t)splits * x.Tq * x.Hq * x.d * 4) + align256((size_t)splits * x.Hq * x.Tq * 4);
}

// Rows of one few-row forward block: every query of a document times the query heads of a group.
long long decode_row_count(const XShape &x) { return (long long)x.maxq * (x.Hq / x.Hkv); }

// Number of key splits, each keeping at least two 128-key tiles, at most 64. Tiled forward:
// enough blocks for about two per SM when the rows alone give fewer. Few-row forward (blocks of
// (split, key/value head, document), two resident per SM): as many splits as fill one wave.
int auto_splits(const XShape &x) {
  const int sms = sm_count() > 0 ? sm_count() : 152;
  const int nkt = (x.maxk + 127) / 128;
  if (decode_row_count(x) <= 8) {
    const long long base = (long long)x.Hkv * x.n;
    if (base <= 0 || nkt < 4) return 1;
    long long want = (long long)decode_blocks_per_sm() * sms / base;
    want = std::min<long long>(want, nkt / 2);
    want = std::min<long long>(want, 64);
    return (int)std::max<long long>(want, 1);
  }
  const long long base = (long long)((x.maxq + 255) / 256) * x.Hq * x.n;
  if (base <= 0 || base >= sms || nkt < 4) return 1;
  long long want = (2LL * sms + base - 1) / base;
  want = std::min<long long>(want, nkt / 2);
  want = std::min<long long>(want, 64);
  return (int)std::max<long long>(want, 1);
}

// Split last wave of the forward grid (one CTA per 256 query rows x head x document, one CTA
// per SM): documents of equal length, no causal mask, a partial last wave of at most half the
// SMs; its CTAs are each split into `splits` key ranges (at least two key tiles each) whose
// partial rows a merge pass combines. bytes: the partial rows and lse the split needs.
struct FwdTail {
  long long first;
  int splits, ntail, gx;
  size_t o_bytes, bytes;
};
FwdTail fwd_tail_plan(const XShape &x) {
  FwdTail t{0, 0, 0, 0, 0, 0};
  if (x.n <= 0 || x.maxq <= 0 || x.maxk <= 0 || decode_row_count(x) <= 8) return t;
  if ((long long)x.n * x.maxq != x.Tq || (long long)x.n * x.maxk != x.Tk) return t;
  if (fwd_tiles_per_cta(x.d, x.maxq) == 1) return t;  // one-tile CTAs, two per SM: not planned
  const int sms = sm_count();
  if (sms <= 0) return t;
  const int gx = (x.maxq + 255) / 256;
  const long long items = (long long)gx * x.Hq * x.n;
  const long long whole = items / sms * sms, ntail = items - whole;
  const int nkv = (x.maxk + 127) / 128;
  if (ntail == 0 || ntail > sms / 2) return t;
  // at most 64 parts per CTA (the merge takes one or two per lane)
  const int splits = (int)std::min<long long>(std::min<long long>(sms / ntail, nkv / 2), 64);
  if (splits < 2) return t;
  t.first = whole;
  t.splits = splits;
  t.ntail = (int)ntail;
  t.gx = gx;
  t.o_bytes = align256((size_t)ntail * splits * 256 * x.d * 4);
  t.bytes = t.o_bytes + align256((size_t)ntail * splits * 256 * 4);
  return t;
}

int fwd_impl(const XShape &x, const void *q, const void *k, const void *v,
             const float *bias_table, int num_buckets, int max_distance, int bidirectional,
             const float *alibi_slopes, const int32_t *cu_q, const int32_t *cu_k, int causal,
             float softmax_scale, void *out, float *lse, int splits, void *workspace,
             size_t workspace_bytes) {
  if (!q || !k || !v || !cu_q || !cu_k || !out) return FAT_EINVAL_NULL;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(cu_q) ||
      misaligned(cu_k) || misaligned(bias_table) || misaligned(alibi_slopes) || misaligned(lse))
    return FAT_EINVAL_SHAPE;
  FwdParams p{};
  int rc = fill_bias(&p.bias, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes);
  if (rc) return rc;
  if (fwd_smem_bytes(x.d, p.bias.lut_len, 2) > (size_t)kSmemLimit) return FAT_EUNSUPPORTED;
  if (splits < 1 || splits > 64 || (long long)x.n * splits > 65535) return FAT_EUNSUPPORTED;
  if (splits > 1) {
    if (!workspace) return FAT_EINVAL_NULL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) ||
        workspace_bytes < splitkv_bytes(x, splits))
      return FAT_EINVAL_SHAPE;
  } else if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
    return FAT_EINVAL_SHAPE;
  }
  if (x.Tq == 0 || x.n == 0 || x.maxq == 0) return FAT_OK;
  rc = device_error_ptr(&p.err);
  if (rc) return rc;
  p.seq = seq_params(x, cu_q, cu_k);
  p.causal = causal ? 1 : 0;
  p.scale_log2 = softmax_scale * kLog2e;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.lse = lse;
  fill_runtime_knobs(&p.timeout_ns, &p.debug_flags);
  p.kv_splits = splits;
  const int nkt = (x.maxk + 127) / 128;
  p.split_tiles = splits == 1 ? (1 << 30) : (nkt + splits - 1) / splits;
  if (splits > 1) {
    char *base = static_cast<char *>(workspace);
    p.o_part = reinterpret_cast<float *>(base);
    p.lse_part = reinterpret_cast<float *>(
        base + align256((size_t)splits * x.Tq * x.Hq * x.d * 4));
  }
  const bool few_rows = decode_row_count(x) <= 8 &&
                        decode_eligible(x.d, (int)decode_row_count(x), x.Hq / x.Hkv, p.bias);
  if (splits == 1 && workspace && !causal && !few_rows) {
    const FwdTail t = fwd_tail_plan(x);
    if (t.splits > 0 && workspace_bytes >= t.bytes) {
      p.tail_first = t.first;
      p.tail_splits = t.splits;
      p.tail_gx = t.gx;
      p.tail_ntail = t.ntail;
      p.tail_o = static_cast<float *>(workspace);
      p.tail_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + t.o_bytes);
    }
  }
  rc = cuda_rc(few_rows ? launch_decode(p, x.d, q, k, v, x.stream)
                        : launch_fwd(p, x.d, q, k, v, x.stream));
  if (rc || splits == 1) return rc;
  return cuda_rc(launch_fwd_combine(p, x.d, x.stream));
}

int check_bwd_args_x(const XShape &x, const void *q, const void *k, const void *v,
                     const float *bias_table, int num_buckets, int max_distance,
                     int bidirectional, const float *alibi_slopes, const int32_t *cu_q,
                     const int32_t *cu_k, const void *out, const float *lse, const void *dout,
                     const void *dq, const void *dk, const void *dv,
                     const float *dbias_table) {
  if (!q || !k || !v || !cu_q || !cu_k || !out || !lse || !dout || !dq || !dk || !dv)
    return FAT_EINVAL_NULL;
  if (dbias_table && !bias_table) return FAT_EUNSUPPORTED;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out) || misaligned(dout) ||
      misaligned(dq) || misaligned(dk) || misaligned(dv) || misaligned(lse) ||
      misaligned(cu_q) || misaligned(cu_k) || misaligned(bias_table) ||
      misaligned(alibi_slopes) || misaligned(dbias_table))
    return FAT_EINVAL_SHAPE;
  BiasParams b{};
  int rc = fill_bias(&b, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes);
  if (rc) return rc;
  if (bwd_smem_bytes(x.d, b.lut_len) > (size_t)kSmemLimit) return FAT_EUNSUPPORTED;
  return FAT_OK;
}

int bwd_preprocess_impl(const XShape &x, const void *out, const void *dout, void *workspace,
                        size_t workspace_bytes, float *dbias_table, int num_buckets,
                        bool overlap_previous) {
  if (!out || !dout) return FAT_EINVAL_NULL;
  if (misaligned(out) || misaligned(dout) || misaligned(dbias_table)) return FAT_EINVAL_SHAPE;
  if (dbias_table && (num_buckets < 2 || num_buckets > 256)) return FAT_EINVAL_BUCKETS;
  WorkspaceView ws{};
  int rc = check_workspace(x, workspace, workspace_bytes, &ws);
  if (rc) return rc;
  const int T = x.Tq, H = x.Hq, d = x.d;
  const int nbias = dbias_table ? num_buckets * H : 0;
  const long long n4 = (long long)(ws.zero_bytes / 16);
  if (T == 0 && n4 == 0) {
    if (!nbias) return FAT_OK;
    const cudaError_t e = cudaMemsetAsync(dbias_table, 0, sizeof(float) * nbias, x.stream);
    if (e != cudaSuccess) set_last_error("cudaMemsetAsync(dbias_table)", (int)e, cudaGetErrorString(e));
    return cuda_rc((int)e);
  }
  const long long rows = (long long)T * H;
  // Enough warps for every (token, head) row group and the zeroing, at most eight 256-thread
  // blocks per SM.
  const long long want = std::max<long long>((rows + 63) / 64, (n4 + 1023) / 1024);
  const int blocks = (int)std::max<long long>(1, std::min<long long>(want, 152LL * 8));
  const auto *o = static_cast<const uint4 *>(out);
  const auto *g = static_cast<const uint4 *>(dout);
  float4 *acc4 = reinterpret_cast<float4 *>(ws.dq_acc);
  float4 *tail4 = reinterpret_cast<float4 *>(ws.tail_acc);
  const long long n4_tail = (long long)(ws.tail_bytes / 16);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = x.stream;
  if (overlap_previous) {  // it waits for the previous grid before touching memory
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e =
      d == 64 ? cudaLaunchKernelEx(&cfg, fat_bwd_prep_kernel<64>, o, g, ws.dvec, acc4, n4,
                                   tail4, n4_tail, dbias_table, nbias, T, H)
              : cudaLaunchKernelEx(&cfg, fat_bwd_prep_kernel<128>, o, g, ws.dvec, acc4, n4,
                                   tail4, n4_tail, dbias_table, nbias, T, H);
  if (e != cudaSuccess) {
    set_last_error("backward preprocess launch", (int)e, cudaGetErrorString(e));
    return FAT_ECUDA;
  }
  return launch_rc("backward preprocess launch");
}

int bwd_main_impl(const XShape &x, const void *q, const void *k, const void *v,
                  const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                  const float *alibi_slopes, const int32_t *cu_q, const int32_t *cu_k,
                  int causal, float softmax_scale, const float *lse, const void *dout,
                  void *workspace, size_t workspace_bytes, void *dk, void *dv,
                  float *dbias_table, bool overlap_previous, bool split_tail) {
  if (!q || !k || !v || !cu_q || !cu_k || !lse || !dout || !dk || !dv) return FAT_EINVAL_NULL;
  if (dbias_table && !bias_table) return FAT_EUNSUPPORTED;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(dout) || misaligned(dk) ||
      misaligned(dv) || misaligned(lse) || misaligned(cu_q) || misaligned(cu_k) ||
      misaligned(bias_table) || misaligned(alibi_slopes) || misaligned(dbias_table))
    return FAT_EINVAL_SHAPE;
  BwdParams p{};
  int rc = fill_bias(&p.bias, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes);
  if (rc) return rc;
  if (bwd_smem_bytes(x.d, p.bias.lut_len) > (size_t)kSmemLimit) return FAT_EUNSUPPORTED;
  WorkspaceView ws{};
  rc = check_workspace(x, workspace, workspace_bytes, &ws);
  if (rc) return rc;
  if (x.Tq == 0 || x.Tk == 0 || x.n == 0 || x.maxq == 0 || x.maxk == 0) return FAT_OK;
  rc = device_error_ptr(&p.err);
  if (rc) return rc;
  p.seq = seq_params(x, cu_q, cu_k);
  p.causal = causal ? 1 : 0;
  p.scale_log2 = softmax_scale * kLog2e;
  p.scale = softmax_scale;
  p.lse = lse;
  p.dvec = ws.dvec;
  p.dq_acc = ws.dq_acc;
  p.dk = static_cast<__nv_bfloat16 *>(dk);
  p.dv = static_cast<__nv_bfloat16 *>(dv);
  p.dk_acc = ws.dk_acc;
  p.dv_acc = ws.dv_acc;
  p.dbias = dbias_table;
  fill_runtime_knobs(&p.timeout_ns, &p.debug_flags);
  if (split_tail && !causal && (ws.tail_acc || ws.dk_acc)) {
    const TailPlan t = bwd_tail_plan(x);
    p.tail_first = t.first;
    p.tail_splits = t.splits;
    p.tail_acc = ws.tail_acc;
  }
  return cuda_rc(launch_bwd(p, x.d, q, k, v, dout, x.stream, overlap_previous));
}

int bwd_finalize_impl(const XShape &x, const void *workspace, size_t workspace_bytes,
                      float softmax_scale, void *dq, void *dk, void *dv, bool overlap_previous,
                      bool split_tail) {
  if (!dq) return FAT_EINVAL_NULL;
  if (misaligned(dq)) return FAT_EINVAL_SHAPE;
  WorkspaceView ws{};
  int rc = check_workspace(x, workspace, workspace_bytes, &ws);
  if (rc) return rc;
  FinishSegs f{};
  long long most = 0;
  auto add = [&](const float *acc, void *dst, float scale, long long n) {
    if (n == 0) return;
    f.acc[f.nseg] = reinterpret_cast<const float4 *>(acc);
    f.out[f.nseg] = static_cast<uint4 *>(dst);
    f.scale[f.nseg] = scale;
    f.n8[f.nseg] = n / 8;
    most = std::max(most, n / 8);
    ++f.nseg;
  };
  add(ws.dq_acc, dq, softmax_scale, (long long)x.Tq * x.Hq * x.d);
  if (ws.dk_acc) {  // query heads share key/value heads: dK (already scaled) and dV
    if (!dk || !dv) return FAT_EINVAL_NULL;
    if (misaligned(dk) || misaligned(dv)) return FAT_EINVAL_SHAPE;
    add(ws.dk_acc, dk, 1.0f, (long long)x.Tk * x.Hkv * x.d);
    add(ws.dv_acc, dv, 1.0f, (long long)x.Tk * x.Hkv * x.d);
  }
  if (split_tail && ws.tail_acc) {  // the split last wave's dK, dV rows
    if (!dk || !dv) return FAT_EINVAL_NULL;
    if (misaligned(dk) || misaligned(dv)) return FAT_EINVAL_SHAPE;
    const TailPlan t = bwd_tail_plan(x);
    f.tail_acc = reinterpret_cast<const float4 *>(ws.tail_acc);
    f.tail_dk = static_cast<uint4 *>(dk);
    f.tail_dv = static_cast<uint4 *>(dv);
    f.tail_first = t.first;
    f.ntail = t.ntail;
    f.nkb = (x.maxk + 127) / 128;
    f.H = x.Hq;
    f.d8 = x.d / 8;
    f.Lk = x.maxk;
    most = std::max(most, (long long)t.ntail * 2 * 128 * (x.d / 8));
  }
  if (f.nseg == 0 && f.ntail == 0) return FAT_OK;
  const int blocks = (int)std::min<long long>((most + 255) / 256, 152LL * 8);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = x.stream;
  if (overlap_previous) {  // programmatic dependent launch on the main backward grid
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fat_bwd_finish_kernel, f);
  if (e != cudaSuccess) {
    set_last_error("backward finalize launch", (int)e, cudaGetErrorString(e));
    return FAT_ECUDA;
  }
  return launch_rc("backward finalize launch");
}

int bwd_impl(const XShape &x, const void *q, const void *k, const void *v,
             const float *bias_table, int num_buckets, int max_distance, int bidirectional,
             const float *alibi_slopes, const int32_t *cu_q, const int32_t *cu_k, int causal,
             float softmax_scale, const void *out, const float *lse, const void *dout,
             void *workspace, size_t workspace_bytes, void *dq, void *dk, void *dv,
             float *dbias_table) {
  // validate everything before enqueueing anything
  int rc = check_bwd_args_x(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional,
                            alibi_slopes, cu_q, cu_k, out, lse, dout, dq, dk, dv, dbias_table);
  if (rc) return rc;
  {
    WorkspaceView ws{};
    rc = check_workspace(x, workspace, workspace_bytes, &ws);
    if (rc) return rc;
  }
  rc = bwd_preprocess_impl(x, out, dout, workspace, workspace_bytes, dbias_table, num_buckets,
                           true);
  if (rc) return rc;
  // All three grids are launched as programmatic dependents of the grid before them: each is
  // scheduled while that grid drains and waits for its writes in-kernel (the preprocessing grid
  // before it touches memory; the main grid before it reads D or touches the accumulators).
  rc = bwd_main_impl(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional,
                     alibi_slopes, cu_q, cu_k, causal, softmax_scale, lse, dout, workspace,
                     workspace_bytes, dk, dv, dbias_table, true, !causal);
  if (rc) return rc;
  rc = bwd_finalize_impl(x, workspace, workspace_bytes, softmax_scale, dq, dk, dv, true,
                         !causal);
  if (rc || cu_q == cu_k || x.Tk == 0 || x.n == 0) return rc;
  // own key sequences: keys of a document without queries get zero gradients
  fat_zero_unseen_keys_kernel<<<x.n, 256, 0, x.stream>>>(cu_q, cu_k, x.Tk, x.Hkv * x.d,
                                                         static_cast<uint4 *>(dk),
                                                         static_cast<uint4 *>(dv));
  return launch_rc("unseen-key zeroing launch");
}

}  // namespace

int check_bwd_args(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                   const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                   const float *alibi_slopes, const int32_t *cu_seqlens, const void *out,
                   const float *lse, const void *dout, const void *dq, const void *dk,
                   const void *dv, const float *dbias_table) {
  XShape x{};
  int rc = to_xshape(sh, &x);
  if (rc) return rc;
  return check_bwd_args_x(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional,
                          alibi_slopes, cu_seqlens, cu_seqlens, out, lse, dout, dq, dk, dv,
                          dbias_table);
}

}  // namespace fat

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
  XShape x{};
  int rc = to_xshape(sh, &x);
  if (rc) return rc;
  return fwd_impl(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes,
                  cu_seqlens, cu_seqlens, causal, softmax_scale, out, lse, 1, nullptr, 0);
}

size_t fat_attn_fwd_workspace_size(const fat_shape_t *sh) {
  XShape x{};
  if (to_xshape(sh, &x)) return 0;
  return fwd_tail_plan(x).bytes;
}

int fat_attn_fwd_ws(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                    const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                    const float *alibi_slopes, const int32_t *cu_seqlens, int causal,
                    float softmax_scale, void *out, float *lse, void *workspace,
                    size_t workspace_bytes) {
  XShape x{};
  int rc = to_xshape(sh, &x);
  if (rc) return rc;
  return fwd_impl(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes,
                  cu_seqlens, cu_seqlens, causal, softmax_scale, out, lse, 1, workspace,
                  workspace_bytes);
}

int fat_xattn_fwd(const fat_xshape_t *xs, const void *q, const void *k, const void *v,
                  const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                  const float *alibi_slopes, const int32_t *cu_seqlens_q,
                  const int32_t *cu_seqlens_k, int causal, float softmax_scale, void *out,
                  float *lse) {
  XShape x{};
  int rc = to_xshape(xs, &x);
  if (rc) return rc;
  return fwd_impl(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes,
                  cu_seqlens_q, cu_seqlens_k, causal, softmax_scale, out, lse, 1, nullptr, 0);
}

int fat_xattn_splitkv_num_splits(const fat_xshape_t *xs) {
  XShape x{};
  if (to_xshape(xs, &x)) return 1;
  return auto_splits(x);
}

size_t fat_xattn_splitkv_workspace_size(const fat_xshape_t *xs, int num_splits) {
  XShape x{};
  if (to_xshape(xs, &x) || num_splits < 1 || num_splits > 64) return 0;
  return num_splits == 1 ? 0 : splitkv_bytes(x, num_splits);
}

int fat_xattn_fwd_splitkv(const fat_xshape_t *xs, const void *q, const void *k, const void *v,
                          const float *bias_table, int num_buckets, int max_distance,
                          int bidirectional, const float *alibi_slopes,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int causal,
                          float softmax_scale, int num_splits, void *workspace,
                          size_t workspace_bytes, void *out, float *lse) {
  XShape x{};
  int rc = to_xshape(xs, &x);
  if (rc) return rc;
  return fwd_impl(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes,
                  cu_seqlens_q, cu_seqlens_k, causal, softmax_scale, out, lse, num_splits,
                  workspace, workspace_bytes);
}

size_t fat_attn_bwd_workspace_size(const fat_shape_t *sh) {
  XShape x{};
  if (to_xshape(sh, &x)) return 0;
  return ws_layout(x).total;
}

size_t fat_xattn_bwd_workspace_size(const fat_xshape_t *xs) {
  XShape x{};
  if (to_xshape(xs, &x)) return 0;
  return ws_layout(x).total;
}

int fat_attn_bwd_preprocess(const fat_shape_t *sh, const void *out, const void *dout,
                            void *workspace, size_t workspace_bytes, float *dbias_table,
                            int num_buckets) {
  XShape x{};
  int rc = to_xshape(sh, &x);
  if (rc) return rc;
  return bwd_preprocess_impl(x, out, dout, workspace, workspace_bytes, dbias_table, num_buckets,
                             false);
}

int fat_attn_bwd_main(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                      const float *bias_table, int num_buckets, int max_distance,
                      int bidirectional, const float *alibi_slopes, const int32_t *cu_seqlens,
                      int causal, float softmax_scale, const float *lse, const void *dout,
                      void *workspace, size_t workspace_bytes, void *dk, void *dv,
                      float *dbias_table) {
  XShape x{};
  int rc = to_xshape(sh, &x);
  if (rc) return rc;
  return bwd_main_impl(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional,
                       alibi_slopes, cu_seqlens, cu_seqlens, causal, softmax_scale, lse, dout,
                       workspace, workspace_bytes, dk, dv, dbias_table, false, false);
}

int fat_attn_bwd_finalize(const fat_shape_t *sh, const void *workspace, size_t workspace_bytes,
                          float softmax_scale, void *dq) {
  XShape x{};
  int rc = to_xshape(sh, &x);
  if (rc) return rc;
  return bwd_finalize_impl(x, workspace, workspace_bytes, softmax_scale, dq, nullptr, nullptr,
                           false, false);
}

int fat_attn_bwd(const fat_shape_t *sh, const void *q, const void *k, const void *v,
                 const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                 const float *alibi_slopes, const int32_t *cu_seqlens, int causal,
                 float softmax_scale, const void *out, const float *lse, const void *dout,
                 void *workspace, size_t workspace_bytes, void *dq, void *dk, void *dv,
                 float *dbias_table) {
  XShape x{};
  int rc = to_xshape(sh, &x);
  if (rc) return rc;
  return bwd_impl(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes,
                  cu_seqlens, cu_seqlens, causal, softmax_scale, out, lse, dout, workspace,
                  workspace_bytes, dq, dk, dv, dbias_table);
}

int fat_xattn_bwd(const fat_xshape_t *xs, const void *q, const void *k, const void *v,
                  const float *bias_table, int num_buckets, int max_distance, int bidirectional,
                  const float *alibi_slopes, const int32_t *cu_seqlens_q,
                  const int32_t *cu_seqlens_k, int causal, float softmax_scale, const void *out,
                  const float *lse, const void *dout, void *workspace, size_t workspace_bytes,
                  void *dq, void *dk, void *dv, float *dbias_table) {
  XShape x{};
  int rc = to_xshape(xs, &x);
  if (rc) return rc;
  return bwd_impl(x, q, k, v, bias_table, num_buckets, max_distance, bidirectional, alibi_slopes,
                  cu_seqlens_q, cu_seqlens_k, causal, softmax_scale, out, lse, dout, workspace,
                  workspace_bytes, dq, dk, dv, dbias_table);
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
// Both device bucket functions the kernels use: the staged binary search (bias tables) and the
// direct count (saturated sides, the few-row kernel); -1 where they disagree.
__global__ void fat_debug_buckets_kernel(const BiasParams b, long long lo, int n, int32_t *out) {
  __shared__ int thr_s[kMaxThresholds];
  for (int i = threadIdx.x; i < b.n_thr; i += blockDim.x) thr_s[i] = b.thr[i];
  __syncthreads();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const int direct = t5_bucket_dev((int)(lo + i), b);
    const int staged = t5_bucket_staged((int)(lo + i), b, thr_s);
    out[i] = direct == staged ? staged : -1;
  }
}
int launch_debug_buckets(const BiasParams &b, long long lo, int n, int32_t *out,
                         cudaStream_t stream) {
  fat_debug_buckets_kernel<<<(n + 255) / 256, 256, 0, stream>>>(b, lo, n, out);
  return (int)cudaGetLastError();
}
}  // namespace fat
