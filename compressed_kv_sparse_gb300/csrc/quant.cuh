// Step 8 of the compressor: block-scaled FP8 (E4M3) and FP4 (E2M1) round
// trips and the Walsh-Hadamard transform ("【#3】ds4.c を読み解く" §4 step 8,
// §9: attention rows take an E4M3 round trip on their non-RoPE dims, indexer
// rows and the indexer query a 128-point Hadamard plus an FP4 round trip).
//
// The arithmetic is fixed so that every scale and code is reproducible:
// * a block of values takes the scale 2^k, k the smallest integer >= -127 with
//   amax <= qmax * 2^k (qmax = 448 for E4M3, 6 for E2M1), read off the bits of
//   amax; x * 2^-k and code * 2^k are exact;
// * a value r (|r| <= qmax) becomes the nearest format value, ties to the even
//   code: r over its quantum (2^(e - mantissa bits) for r of exponent e, the
//   subnormal quantum below the smallest normal) is rounded half to even;
// * the Hadamard is the radix-2 butterfly over stages h = 1, 2, ..., n/2, each
//   pair (a at i, b at i + h, i & h == 0) becoming (a + b, a - b) in fp32, then
//   a multiplication by c = 1/sqrt(n) rounded to fp32.
// Blocks: 64 consecutive non-RoPE dims (FP8), 32 transformed values (FP4).
#pragma once
#include "common.cuh"

namespace ds4a {

struct QFmt {
  uint32_t max_frac;   // fraction bits of the largest finite value
  int max_exp;         // its exponent
  int man_bits;        // mantissa bits
  int min_normal_exp;  // exponent of the smallest normal
};
constexpr QFmt kE4M3{0x600000u, 8, 3, -6};   // 448 = 1.75 * 2^8
constexpr QFmt kE2M1{0x400000u, 2, 1, 0};    // 6 = 1.5 * 2^2

// 2^e for -127 <= e <= 127 (2^-127 is an fp32 subnormal).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Smallest k >= -127 with amax <= qmax * 2^k.
__device__ __forceinline__ int block_scale_exp(float amax, QFmt f) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (b < 0x00800000u) return -127;   // zero or subnormal: within qmax * 2^-127
  const int e = (int)(b >> 23) - 127;
  const int k = e - f.max_exp + ((b & 0x7FFFFFu) > f.max_frac ? 1 : 0);
  return k < -127 ? -127 : k;
}

// Nearest format value to r (|r| <= the format's largest value), ties to even.
__device__ __forceinline__ float round_fmt(float r, QFmt f) {
  const float a = fabsf(r);
  const int e = (int)(__float_as_uint(a) >> 23) - 127;
  const int qe = (e < f.min_normal_exp ? f.min_normal_exp : e) - f.man_bits;
  const float n = rintf(__fmul_rn(a, pow2f(-qe)));
  return copysignf(__fmul_rn(n, pow2f(qe)), r);
}

__device__ __forceinline__ float quant_dequant(float x, int k, QFmt f) {
  return __fmul_rn(round_fmt(__fmul_rn(x, pow2f(-k)), f), pow2f(k));
}

// In-place unnormalised Walsh-Hadamard transform of buf[0, n) in shared
// memory. Every thread of the block calls it after buf is written and a
// barrier has passed; it ends with a barrier.
__device__ __forceinline__ void fwht_smem(float *buf, uint32_t n) {
  for (uint32_t h = 1; h < n; h <<= 1) {
    for (uint32_t t = threadIdx.x; t < n / 2; t += blockDim.x) {
      const uint32_t i = (t / h) * 2 * h + (t % h);
      const float a = buf[i], b = buf[i + h];
      buf[i] = __fadd_rn(a, b);
      buf[i + h] = __fsub_rn(a, b);
    }
    __syncthreads();
  }
}

// FP4 QAT round trip of buf[0, n) in place (n a power of two >= 32):
// z = c H x, E2M1 per 32 values, x' = c H z'. Same calling rules as
// fwht_smem; blockDim.x is a multiple of 32.
__device__ __forceinline__ void fp4_qat_smem(float *buf, uint32_t n, float c) {
  fwht_smem(buf, n);
  const uint32_t lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (uint32_t b = threadIdx.x >> 5; b < n / 32; b += nw) {   // warp-uniform
    const float z = __fmul_rn(buf[b * 32 + lane], c);
    const int k = block_scale_exp(warp_max(fabsf(z)), kE2M1);
    buf[b * 32 + lane] = quant_dequant(z, k, kE2M1);
  }
  __syncthreads();
  fwht_smem(buf, n);
  for (uint32_t d = threadIdx.x; d < n; d += blockDim.x) buf[d] = __fmul_rn(buf[d], c);
  __syncthreads();
}

// The same round trip on a row held by an aligned group of G lanes (G = n / 8,
// a power of two, 4 <= G <= 32), eight consecutive values per lane: v[j] is
// value 8u + j, u the lane's index in the group; `mask` holds the group.
__device__ __forceinline__ void fp4_qat_lanes8(float (&v)[8], uint32_t u, uint32_t G,
                                               uint32_t mask, float c) {
  auto fwht = [&]() {
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (!(j & h)) {
          const float a = v[j], b = v[j + h];
          v[j] = __fadd_rn(a, b);
          v[j + h] = __fsub_rn(a, b);
        }
    for (uint32_t m = 1; m < G; m <<= 1)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float o = __shfl_xor_sync(mask, v[j], m);
        v[j] = (u & m) ? __fsub_rn(o, v[j]) : __fadd_rn(v[j], o);
      }
  };
  fwht();
  float am = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = __fmul_rn(v[j], c);
    am = fmaxf(am, fabsf(v[j]));
  }
  am = fmaxf(am, __shfl_xor_sync(mask, am, 1));   // 32 values = 4 lanes
  am = fmaxf(am, __shfl_xor_sync(mask, am, 2));
  const int k = block_scale_exp(am, kE2M1);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = quant_dequant(v[j], k, kE2M1);
  fwht();
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], c);
}

}  // namespace ds4a
