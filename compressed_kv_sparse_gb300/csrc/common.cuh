// Device helpers shared by the ds4a kernels (element access, reductions).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace ds4a {

// Programmatic dependent launch. Kernels launched with launch_pdl may start
// while the previous kernel in the stream is still running: each calls
// pdl_wait() (the previous grid has completed and its writes are visible)
// before its first global memory access, then pdl_trigger() so that the next
// kernel can be scheduled as soon as SMs free up.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Position of sequence b's first token in this call: its own (ragged decode,
// seq_pos non-NULL) or the call's pos0.
__device__ __forceinline__ uint32_t seq_base(const uint32_t *seq_pos, uint32_t pos0, uint32_t b) {
  return seq_pos ? __ldg(seq_pos + b) : pos0;
}

__device__ __forceinline__ float ld_f32(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_f32(const __nv_bfloat16 *p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_elem(float *p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, size_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}
// Round an fp32 value to the storage type and back (exact for fp32).
__device__ __forceinline__ float round_to(float v, const float *) { return v; }
__device__ __forceinline__ float round_to(float v, const __nv_bfloat16 *) {
  return __bfloat162float(__float2bfloat16_rn(v));
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

// Block-wide sum; every thread gets the result. `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float *red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
}

// Block-wide max; every thread gets the result. `red` holds >= 32 floats.
__device__ __forceinline__ float block_max(float v, float *red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_max(t);
}

// An upper bound of the Euclidean norm from partial sums of scaled squares:
// the values were multiplied by 2^-e (e = exponent of the largest |value|,
// exact) before squaring, so squares of tiny magnitudes do not underflow.
// `ss_scaled` = sum of the scaled squares (>= 0.25 when the largest value is
// nonzero); the result is scaled back and widened by 2^-16 for the fp32
// roundings of at most a few hundred terms.
__device__ __forceinline__ float norm_from_scaled(float ss_scaled, int e) {
  return ldexpf(sqrtf(ss_scaled), e) * (1.0f + 0x1p-16f);
}

}  // namespace ds4a
