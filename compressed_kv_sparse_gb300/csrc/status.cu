// Host read-back of the error word that the bounded device waits write, and a
// self-test of those waits. Every wait of the tensor-core kernels gives up
// after a time limit, adds 1 to the error word at byte offset 0 of the call's
// workspace and lets its thread block wind down (tc.cuh), so a stuck call
// returns with its outputs invalid instead of hanging the device; these calls
// let the host see that it happened.
#include "internal.h"
#include "tc.cuh"

namespace ds4a {
namespace {

// One block waits on a barrier phase that nothing completes: the barrier
// expects one arrival and no thread arrives. Nothing asynchronous (copy or
// MMA) is issued, so giving up leaves nothing in flight.
__global__ void wait_selftest_kernel(int *err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const ErrWord ew{err, *(volatile int *)err};
  const bool ok = __all_sync(0xffffffffu, mbar_wait_for(&bar, 0, ew, limit_ns));
  (void)ok;
}

}  // namespace
}  // namespace ds4a

extern "C" {

ds4a_status ds4a_workspace_status(const void *ws, size_t ws_bytes, uint32_t *count) {
  if (!ws || ws_bytes < sizeof(int)) return DS4A_ERR_WORKSPACE;
  int v = 0;
  // device (or managed) memory: a 4-byte copy; host memory (a mapped or
  // pinned workspace, or a host copy of the word): read in place
  cudaPointerAttributes at;
  const bool known = cudaPointerGetAttributes(&at, ws) == cudaSuccess;
  if (!known) (void)cudaGetLastError();
  if (known && (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)) {
    if (ds4a::note_error(cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
      return DS4A_ERR_CUDA;
  } else {
    v = *static_cast<const volatile int *>(ws);
  }
  if (count) *count = (uint32_t)v;
  return v ? DS4A_ERR_TIMEOUT : DS4A_OK;
}

ds4a_status ds4a_workspace_clear_status(void *ws, size_t ws_bytes, ds4a_stream_t stream) {
  if (!ws || ws_bytes < sizeof(int)) return DS4A_ERR_WORKSPACE;
  const cudaError_t e =
      cudaMemsetAsync(ws, 0, sizeof(int), reinterpret_cast<cudaStream_t>(stream));
  return ds4a::note_error(e) == cudaSuccess ? DS4A_OK : DS4A_ERR_CUDA;
}

ds4a_status ds4a_wait_selftest(void *ws, size_t ws_bytes, uint32_t limit_us,
                               ds4a_stream_t stream) {
  if (!ws || ws_bytes < sizeof(int)) return DS4A_ERR_WORKSPACE;
  if (limit_us == 0 || limit_us > 1000000u) return DS4A_ERR_ARG;
  ds4a::wait_selftest_kernel<<<1, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<int *>(ws), (uint64_t)limit_us * 1000u);
  ds4a::note_launches(1);
  return ds4a::note_error(cudaGetLastError()) == cudaSuccess ? DS4A_OK : DS4A_ERR_CUDA;
}

}  // extern "C"
