// Selection helpers of the indexer top-k (shared by the select kernels and
// the fused decode scorer): order-preserving score keys, block scans, the
// radix select with ties to the lower index, and the exact fp32 score recipe
// ("【#3】ds4.c を読み解く" §6 indexer) for rows whose tensor-core score is too
// close to the cut to decide.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"

namespace ds4a {
namespace {

constexpr uint32_t kHistBins = 4096;    // bins of the top 12 bits of a score key

// Order-preserving unsigned key of an fp32 score (+0 and -0 share a key).
__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint32_t score_key(float f) {
  if (f == 0.f) f = 0.f;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix of a 0/1 flag; returns the prefix, adds the
// block total to *total. Uses warp ballots; `wsum` holds 32 ints.
__device__ __forceinline__ uint32_t block_flag_scan(bool flag, uint32_t *wsum,
                                                    uint32_t *total) {
  const uint32_t lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t bal = __ballot_sync(0xffffffffu, flag);
  const uint32_t in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) wsum[wid] = __popc(bal);
  __syncthreads();
  if (wid == 0) {
    const uint32_t nw = blockDim.x >> 5;
    uint32_t v = lane < nw ? wsum[lane] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= (uint32_t)o) incl += n;
    }
    if (lane < nw) wsum[lane] = incl - v;
    if (lane == 31) wsum[32] = incl;
  }
  __syncthreads();
  const uint32_t r = wsum[wid] + in_warp;
  const uint32_t tot = wsum[32];
  __syncthreads();
  *total = tot;
  return r;
}

// k-th largest of key(s), s < n, by an 8-bit radix select. Returns the key
// and, in *need, how many rows with exactly that key belong to the top k.
// With last_shift = 8 or 16 it stops after three or two digits and returns
// the lowest key with the k-th largest key's top 24 or 16 bits (at least k
// keys are >= it).
template <typename KeyF>
__device__ uint32_t radix_kth(KeyF key, uint32_t n, uint32_t k, uint32_t *hist, uint32_t *sel,
                              uint32_t *need_out, int last_shift = 0) {
  uint32_t prefix = 0, mask = 0, need = k;
  for (int shift = 24; shift >= last_shift; shift -= 8) {
    for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    // warp-aggregated: lanes with the same digit add once (keys of similar
    // magnitude share their top digits, so per-lane atomics would serialise)
    for (uint32_t base = 0; base < n; base += blockDim.x) {
      const uint32_t s = base + threadIdx.x;
      uint32_t bin = 256u;
      if (s < n) {
        const uint32_t kk = key(s);
        if ((kk & mask) == prefix) bin = (kk >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (bin < 256u && (threadIdx.x & 31) == (uint32_t)(__ffs(peers) - 1))
        atomicAdd(&hist[bin], (uint32_t)__popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // digit holding the need-th largest key: lane l covers digits
      // 255 - 8l .. 248 - 8l; a scan over lanes runs from the top digit down
      const uint32_t lane = threadIdx.x;
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        tot += c[j];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= (uint32_t)o) incl += v;
      }
      uint32_t cum = incl - tot;
      if (cum < need && incl >= need) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cum + c[j] >= need) {
            sel[0] = 255 - 8 * lane - j;
            sel[1] = cum;
            break;
          }
          cum += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= sel[0] << shift;
    mask |= 255u << shift;
    need -= sel[1];
    __syncthreads();
  }
  *need_out = need;
  return prefix;
}

// Write, in ascending order of s, every s with key > kth and the first
// `need` with key == kth (ties to the lower index); out[pos] = map(s).
template <typename KeyF, typename MapF>
__device__ void ordered_emit(KeyF key, uint32_t n, uint32_t kth, uint32_t need, uint32_t k,
                             int32_t *out, uint32_t *wsum, MapF map) {
  uint32_t eq_seen = 0, out_pos = 0;
  for (uint32_t base = 0; base < n; base += blockDim.x) {
    const uint32_t s = base + threadIdx.x;
    const uint32_t kk = s < n ? key(s) : 0u;
    const bool gt = s < n && kk > kth;
    const bool eq = s < n && kk == kth;
    uint32_t eq_tot, sel_tot;
    const uint32_t eq_rank = eq_seen + block_flag_scan(eq, wsum, &eq_tot);
    const bool take = gt || (eq && eq_rank < need);
    const uint32_t pos = out_pos + block_flag_scan(take, wsum, &sel_tot);
    if (take && pos < k) out[pos] = (int32_t)map(s);
    eq_seen += eq_tot;
    out_pos += sel_tot;
  }
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr float kRel = 2.4e-7f;        // slack for the rounding of the bound arithmetic
constexpr uint32_t kQB = 132;          // row stride (bf16) of q' in shared memory: the 8-byte
                                        // loads of 16 lanes at 16 rows hit 32 distinct banks

// Block-wide exclusive prefix sum of v (every thread gets its prefix and the
// total). `wsum` holds 33 words.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *wsum, uint32_t *total) {
  const uint32_t lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= (uint32_t)o) incl += n;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const uint32_t nw = blockDim.x >> 5;
    const uint32_t x = lane < nw ? wsum[lane] : 0u;
    uint32_t in2 = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, in2, o);
      if (lane >= (uint32_t)o) in2 += n;
    }
    if (lane < nw) wsum[lane] = in2 - x;
    if (lane == 31) wsum[32] = in2;
  }
  __syncthreads();
  const uint32_t r = wsum[wid] + incl - v;
  *total = wsum[32];
  __syncthreads();
  return r;
}

// Unbiased exponent of a nonzero fp32 value; subnormals report -140 (below
// any of their magnitudes), inf / NaN 128.
__device__ __forceinline__ int exp_of(float x) {
  const int f = (int)((__float_as_uint(x) >> 23) & 0xFFu);
  return f == 0 ? -140 : f - 127;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// The exact recipe adds fl(q * k) to the running dot product in ascending d.
// For two bf16 factors the product has at most 16 significant bits, so
// fl(q * k) = q * k unless it is subnormal or overflows, and then
// fma(q, k, acc) rounds exactly like acc + fl(q * k). The exponent ranges of
// q' (eq_min, eq_max, over nonzero entries) and of the key rows decide which
// form is used.
__device__ __forceinline__ bool fma_exact(int eq_min, int eq_max, int ek_min, int ek_max) {
  return eq_min + ek_min >= -126 && eq_max + ek_max <= 125;
}

// Exponent range of the nonzero entries among four key values, over the warp.
__device__ __forceinline__ void key_exp_range(const float (&kk)[4], int &emin, int &emax) {
  emin = 1000;
  emax = -1000;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (kk[e] != 0.f) {
      emin = min(emin, exp_of(kk[e]));
      emax = max(emax, exp_of(kk[e]));
    }
  }
  emin = warp_min_i(emin);
  emax = warp_max_i(emax);
}

__device__ __forceinline__ void bf16x4(uint2 v, float &a, float &b, float &c, float &d) {
  a = __uint_as_float(v.x << 16);
  b = __uint_as_float(v.x & 0xFFFF0000u);
  c = __uint_as_float(v.y << 16);
  d = __uint_as_float(v.y & 0xFFFF0000u);
}

// Exact recipe for key row `kr` against the 64 x 128 query in shared memory
// (one warp, two heads per lane); lane 0 returns the score.
__device__ __forceinline__ float rescore_row(const __nv_bfloat16 *qsm, const float *wsh, float *kb,
                                             float *rel, const __nv_bfloat16 *kr, uint32_t lane,
                                             int eq_min, int eq_max) {
  __syncwarp();
  int emin, emax;
  {
    float kk[4];
    bf16x4(*reinterpret_cast<const uint2 *>(kr + 4 * lane), kk[0], kk[1], kk[2], kk[3]);
    *reinterpret_cast<float4 *>(kb + 4 * lane) = make_float4(kk[0], kk[1], kk[2], kk[3]);
    key_exp_range(kk, emin, emax);
  }
  const bool exact = fma_exact(eq_min, eq_max, emin, emax);
  __syncwarp();
  const float4 *k4 = reinterpret_cast<const float4 *>(kb);
#pragma unroll
  for (uint32_t j = 0; j < 2; ++j) {
    const uint32_t h = lane + 32 * j;
    const uint2 *q2 = reinterpret_cast<const uint2 *>(qsm + (size_t)h * kQB);
    float acc = 0.f;
#pragma unroll 4
    for (uint32_t c = 0; c < 32; ++c) {
      float q0, q1, q2v, q3;
      bf16x4(q2[c], q0, q1, q2v, q3);
      const float4 k = k4[c];
      if (exact) {
        acc = fmaf(q0, k.x, acc);
        acc = fmaf(q1, k.y, acc);
        acc = fmaf(q2v, k.z, acc);
        acc = fmaf(q3, k.w, acc);
      } else {
        acc = __fadd_rn(acc, __fmul_rn(q0, k.x));
        acc = __fadd_rn(acc, __fmul_rn(q1, k.y));
        acc = __fadd_rn(acc, __fmul_rn(q2v, k.z));
        acc = __fadd_rn(acc, __fmul_rn(q3, k.w));
      }
    }
    rel[h] = acc > 0.f ? acc : 0.f;
  }
  __syncwarp();
  float tot = 0.f;
  if (lane == 0) {
#pragma unroll 16
    for (uint32_t h = 0; h < 64; ++h) tot = __fadd_rn(tot, __fmul_rn(wsh[h], rel[h]));
  }
  return tot;
}

// Per-head ReLU dots of RPP band rows (fp32 keys at k4, RPP x 128) against
// head h of q': one q' load serves RPP rows. `exact`: every product is exact,
// so the fused form rounds like the separate one.
template <int RPP>
__device__ __forceinline__ void band_dots(const uint2 *q2, const float4 *k4, bool exact,
                                          float (&acc)[RPP]) {
#pragma unroll
  for (int rr = 0; rr < RPP; ++rr) acc[rr] = 0.f;
  constexpr int kUnroll = RPP >= 4 ? 2 : 4;
  if (exact) {
#pragma unroll kUnroll
    for (uint32_t c = 0; c < 32; ++c) {
      float q0, q1, q2v, q3;
      bf16x4(q2[c], q0, q1, q2v, q3);
#pragma unroll
      for (int rr = 0; rr < RPP; ++rr) {
        const float4 k = k4[rr * 32 + c];
        acc[rr] = fmaf(q0, k.x, acc[rr]);
        acc[rr] = fmaf(q1, k.y, acc[rr]);
        acc[rr] = fmaf(q2v, k.z, acc[rr]);
        acc[rr] = fmaf(q3, k.w, acc[rr]);
      }
    }
  } else {
#pragma unroll 2
    for (uint32_t c = 0; c < 32; ++c) {
      float q0, q1, q2v, q3;
      bf16x4(q2[c], q0, q1, q2v, q3);
#pragma unroll
      for (int rr = 0; rr < RPP; ++rr) {
        const float4 k = k4[rr * 32 + c];
        acc[rr] = __fadd_rn(acc[rr], __fmul_rn(q0, k.x));
        acc[rr] = __fadd_rn(acc[rr], __fmul_rn(q1, k.y));
        acc[rr] = __fadd_rn(acc[rr], __fmul_rn(q2v, k.z));
        acc[rr] = __fadd_rn(acc[rr], __fmul_rn(q3, k.w));
      }
    }
  }
}

// Exact recipe for the band rows (whole block, NW warps), in rounds of 2 NW
// rows: every key row of the round is loaded first (two per warp, both loads
// in flight before either converts) as fp32 into `kbuf` [2 NW][128], with the
// row's exponent range; then thread t takes head t % 64 of the row group
// t / 64 (two rows with 1024 threads, four with 256: one q' load serves the
// group, and every lane of a warp reads the same keys) and writes their ReLU
// dots to `relb` [2 NW][64]; then one thread per row sums w_h ReLU(dot_h) in
// ascending h. Results replace cS[band[i]].
template <int NW>
__device__ __forceinline__ void rescore_band(const __nv_bfloat16 *qsm, const float *wsh,
                                             float *kbuf, float *relb, const uint32_t *band,
                                             uint32_t nband, const uint32_t *cidx, float *cS,
                                             const __nv_bfloat16 *keys, const RowMap &map,
                                             uint32_t b, uint32_t *rexact,
                                             int eq_min, int eq_max) {
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t RPR = 2 * NW, NT = 32 * NW;
  for (uint32_t base = 0; base < nband; base += RPR) {
    const uint32_t nr = min(RPR, nband - base);
    uint2 kv[2];
#pragma unroll
    for (uint32_t t = 0; t < 2; ++t) {
      const uint32_t rr = warp + NW * t;
      if (rr < nr)   // warp-uniform
        kv[t] = *reinterpret_cast<const uint2 *>(keys + map.row_of(b, cidx[band[base + rr]]) * 128 +
                                                 4 * lane);
    }
#pragma unroll
    for (uint32_t t = 0; t < 2; ++t) {
      const uint32_t rr = warp + NW * t;
      if (rr < nr) {   // warp-uniform
        float kk[4];
        bf16x4(kv[t], kk[0], kk[1], kk[2], kk[3]);
        *reinterpret_cast<float4 *>(kbuf + rr * 128 + 4 * lane) =
            make_float4(kk[0], kk[1], kk[2], kk[3]);
        int emin, emax;
        key_exp_range(kk, emin, emax);
        if (lane == 0) rexact[rr] = fma_exact(eq_min, eq_max, emin, emax) ? 1u : 0u;
      }
    }
    __syncthreads();
    // (row group, head): rows RPP g .. RPP g + RPP - 1 of the round against
    // head h (RPP = 4 where that leaves one item per thread: four
    // independent chains instead of two items in turn)
    constexpr uint32_t RPP = NT >= 1024 ? 2 : 4;
    const uint32_t n_grp = (nr + RPP - 1) / RPP;
    for (uint32_t it = threadIdx.x; it < n_grp * 64; it += NT) {
      const uint32_t rp = it >> 6, h = it & 63, r0 = RPP * rp;
      const uint2 *q2 = reinterpret_cast<const uint2 *>(qsm + (size_t)h * kQB);
      const float4 *k4 = reinterpret_cast<const float4 *>(kbuf + r0 * 128);
      // (rows past the round's last read stale keys: never stored)
      const uint32_t nv = min(RPP, nr - r0);
      bool exact = true;
#pragma unroll
      for (uint32_t rr = 0; rr < RPP; ++rr) exact = exact && (rr >= nv || rexact[r0 + rr] != 0u);
      float acc[RPP];
      band_dots<RPP>(q2, k4, exact, acc);
#pragma unroll
      for (uint32_t rr = 0; rr < RPP; ++rr)
        if (rr < nv) relb[(r0 + rr) * 64 + h] = acc[rr] > 0.f ? acc[rr] : 0.f;
    }
    __syncthreads();
    if (threadIdx.x < nr) {
      const float *rl = relb + threadIdx.x * 64;
      float tot = 0.f;
#pragma unroll 16
      for (uint32_t hh = 0; hh < 64; ++hh) tot = __fadd_rn(tot, __fmul_rn(wsh[hh], rl[hh]));
      cS[band[base + threadIdx.x]] = tot;
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace ds4a
