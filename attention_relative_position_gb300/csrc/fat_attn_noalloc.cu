// fat_attn_noalloc.cu -- the backward pass for callers that cannot allocate device memory.
//
// fat_attn_bwd needs a scratch workspace (the fp32 dQ accumulator and the row statistics D).
// Some callers cannot provide one: a host application that hands this library a fixed budget of
// caller-owned buffers and owns every allocation on the GPU, or a plug-in loaded into a framework
// whose allocator must not be bypassed and which gives plug-ins no allocation hook. For them this
// file keeps the scratch in a file-scope device array of fixed size, which every GPU that loads
// the library holds until the process exits, and runs the ordinary backward stages on it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fat_attn.h"
#include "fat_attn_internal.cuh"

namespace {

// The built-in scratch (size in include/fat_attn.h). Shared by every call on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FAT_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[128] = {nullptr};  // device address of the array, per device ordinal

// Device address of the scratch on the current device. The first call on a device looks it up
// (set-up, with that device current); later calls reuse it. The address stays valid as long as
// the device's primary context does: resetting the device after the first call is unsupported.
int scratch_on_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    fat::set_last_error("fat_attn_bwd_noalloc: cudaGetDevice", (int)e, cudaGetErrorString(e));
    return FAT_ECUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      fat::set_last_error("fat_attn_bwd_noalloc: cudaGetSymbolAddress(scratch)", (int)e,
                          cudaGetErrorString(e));
      return FAT_ECUDA;
    }
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return FAT_OK;
}

}  // namespace

extern "C" int fat_attn_bwd_noalloc(const fat_shape_t *sh, const void *q, const void *k,
                                    const void *v, const float *bias_table, int num_buckets,
                                    int max_distance, int bidirectional,
                                    const float *alibi_slopes, const int32_t *cu_seqlens,
                                    int causal, float softmax_scale, const void *out,
                                    const float *lse, const void *dout, void *dq, void *dk,
                                    void *dv, float *dbias_table) {
  // the same argument checks as fat_attn_bwd first, so that errors come out as they would there
  int rc = fat::check_bwd_args(sh, q, k, v, bias_table, num_buckets, max_distance, bidirectional,
                               alibi_slopes, cu_seqlens, out, lse, dout, dq, dk, dv,
                               dbias_table);
  if (rc) return rc;
  const size_t need = fat_attn_bwd_workspace_size(sh);
  if (need > (size_t)FAT_NOALLOC_SCRATCH_BYTES) {
    fat::set_last_error("fat_attn_bwd_noalloc: the problem needs more scratch than the built-in "
                        "array holds (bytes needed)",
                        (int)(need > 0x7fffffffu ? 0x7fffffff : need),
                        "use fat_attn_bwd with a caller-provided workspace");
    return FAT_EUNSUPPORTED;
  }
  void *scratch = nullptr;
  rc = scratch_on_current_device(&scratch);
  if (rc) return rc;
  return fat_attn_bwd(sh, q, k, v, bias_table, num_buckets, max_distance, bidirectional,
                      alibi_slopes, cu_seqlens, causal, softmax_scale, out, lse, dout, scratch,
                      (size_t)FAT_NOALLOC_SCRATCH_BYTES, dq, dk, dv, dbias_table);
}
