// ds4a_index_topk_noalloc: the indexer top-k with its scratch in a static
// device array instead of a caller-provided workspace, for callers that
// cannot allocate device memory (see the declaration in ds4a.h).
#include <mutex>

#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

// The scratch area. In host code `g_scratch` names a host-side stand-in, not
// a device address: only the pointer from cudaGetSymbolAddress may be handed
// to a kernel.
static __device__ __align__(256) unsigned char g_scratch[DS4A_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_dev[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" ds4a_status ds4a_index_topk_noalloc(const ds4a_layer_cache *cache, uint32_t pos0,
                                               uint32_t T, const void *q_idx, const void *w,
                                               uint32_t n_heads, uint32_t top_k, int32_t *topk,
                                               ds4a_stream_t stream) {
  // the checks of ds4a_index_topk first, so that a malformed call gets the
  // same status from both entry points; then the scratch size
  const ds4a_status st = ds4a::index_topk_check(cache, pos0, T, q_idx, w, n_heads, top_k, topk);
  if (st) return st;
  const size_t need = ds4a_workspace_bytes(DS4A_CALL_INDEX_TOPK, cache, T, n_heads, top_k);
  if (need > DS4A_STATIC_SCRATCH_BYTES) return DS4A_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (ds4a::note_error(scratch_address(&scratch)) != cudaSuccess) return DS4A_ERR_CUDA;
  return ds4a_index_topk(cache, pos0, T, q_idx, w, n_heads, top_k, topk, scratch,
                         DS4A_STATIC_SCRATCH_BYTES, stream);
}

extern "C" ds4a_status ds4a_noalloc_status(uint32_t *count) {
  void *scratch = nullptr;
  if (ds4a::note_error(scratch_address(&scratch)) != cudaSuccess) return DS4A_ERR_CUDA;
  return ds4a_workspace_status(scratch, DS4A_STATIC_SCRATCH_BYTES, count);
}
