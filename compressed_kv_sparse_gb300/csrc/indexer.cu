// Ratio-4 indexer: score visible compressed index rows and keep the top k
// ("【#3】ds4.c を読み解く" §6 indexer, §7 visible rows; vLLM DeepSeek V4 page,
// DSA top-k).
//
// Score (fp32, fixed order, one rounding per operation, no fused multiply-add):
//   dot_h = (((q'_h0 k_0) + q'_h1 k_1) + ...)  ascending d
//   I     = (((w_0 relu(dot_0)) + w_1 relu(dot_1)) + ...)  ascending h, from +0
// with q' the indexer query rotated at its position in fp32 and rounded to the
// storage dtype. The selection is exact for this score: ties go to the lower
// row index and the kept rows come out in ascending order.
//
// fp32 layers: rotate the queries, score every visible row with the exact
// recipe (one thread per row, keys staged in shared memory), then a per-query
// radix select (8-bit digits over an order-preserving key) and an ordered
// compaction.
// bf16 layers (64 heads x 128 dims): rotate the queries to bf16, score every
// visible row on the tensor cores (indexer_tc.cu: approximate scores S~ and
// key norms), then a certified selection per query: with tau~ the k-th largest
// S~ and e_s = c * A_t * ||k_s|| a bound on |S~ - S| (A_t = sum_h |w_h| ||q'_h||,
// c from the accumulation lengths), rows with S~ - e_s > tau~ + E are certainly
// kept, rows with S~ + e_s < tau~ - E certainly dropped (E = max e_s), and the
// rows in between are rescored with the exact recipe before the final exact
// radix select. The kept set is therefore the exact one.
#include <cmath>

#include "common.cuh"

namespace ds4a {
namespace {

constexpr int kRowsPerBlock = 128;
constexpr int kSelectThreads = 1024;

__host__ __device__ inline uint32_t round_up8(uint32_t x) { return (x + 7u) & ~7u; }

// Workspace layout: qrot [B*T][Di][Hpad] fp32, then scores [B*T][comp_cap] fp32.
struct IndexWs {
  float *qrot, *scores;
};
__host__ __device__ inline IndexWs index_ws_split(void *ws, uint32_t nq, uint32_t Hi,
                                                  uint32_t Di) {
  float *base = static_cast<float *>(ws);
  const size_t qsz = (size_t)nq * Di * round_up8(Hi);
  return IndexWs{base, base + ((qsz + 63) & ~(size_t)63)};
}

// Workspace of bf16 layers: err word, A_t [nq], qbf [nq][Hi][Di] bf16,
// norms [B][comp_cap], scores [nq][comp_cap] (fp32, rewritten in place as the
// exact selection keys).
struct TcWs {
  int *err;
  float *at, *norms, *scores;
  __nv_bfloat16 *qbf;
};
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline TcWs tc_ws_split(void *ws, uint32_t nq, uint32_t B, uint32_t Hi, uint32_t Di,
                        uint32_t comp_cap, size_t *total) {
  uint8_t *base = static_cast<uint8_t *>(ws);
  size_t off = 0;
  TcWs w;
  w.err = reinterpret_cast<int *>(base + off);
  off = align_up(off + 16, 256);
  w.at = reinterpret_cast<float *>(base + off);
  off = align_up(off + (size_t)nq * 4, 1024);
  w.qbf = reinterpret_cast<__nv_bfloat16 *>(base + off);
  off = align_up(off + (size_t)nq * Hi * Di * 2, 256);
  w.norms = reinterpret_cast<float *>(base + off);
  off = align_up(off + (size_t)B * comp_cap * 4, 256);
  w.scores = reinterpret_cast<float *>(base + off);
  off += (size_t)nq * comp_cap * 4;
  if (total) *total = off;
  return w;
}

// bf16 layers: q' = rotated query rounded to bf16 (fp32 recipe), and
// A_t = sum_h |w_h| ||q'_h||. Block 0 also clears the error word.
__global__ void index_qbf_kernel(IndexArgs a, __nv_bfloat16 *qbf, float *at, int *err) {
  __shared__ float red[32];
  const uint32_t qi = blockIdx.x, t = qi % a.T, p = a.pos0 + t;
  const uint32_t Hi = a.n_heads, Di = a.dim, n_nope = Di - a.rot;
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q_idx) + (size_t)qi * Hi * Di;
  const __nv_bfloat16 *w = static_cast<const __nv_bfloat16 *>(a.w) + (size_t)qi * Hi;
  __nv_bfloat16 *dst = qbf + (size_t)qi * Hi * Di;
  if (qi == 0 && threadIdx.x == 0) *err = 0;
  float part = 0.f;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (uint32_t h = warp; h < Hi; h += nw) {
    float ss = 0.f;
    for (uint32_t c = 2 * lane; c < Di; c += 64) {
      float x0 = __bfloat162float(q[(size_t)h * Di + c]);
      float x1 = __bfloat162float(q[(size_t)h * Di + c + 1]);
      if (c >= n_nope) {
        const uint32_t fi = (c - n_nope) / 2;
        const float co = a.cos[(size_t)p * (a.rot / 2) + fi];
        const float si = a.sin[(size_t)p * (a.rot / 2) + fi];
        const float r0 = __fsub_rn(__fmul_rn(x0, co), __fmul_rn(x1, si));
        const float r1 = __fadd_rn(__fmul_rn(x0, si), __fmul_rn(x1, co));
        x0 = __bfloat162float(__float2bfloat16_rn(r0));
        x1 = __bfloat162float(__float2bfloat16_rn(r1));
      }
      dst[(size_t)h * Di + c] = __float2bfloat16_rn(x0);
      dst[(size_t)h * Di + c + 1] = __float2bfloat16_rn(x1);
      ss = fmaf(x0, x0, fmaf(x1, x1, ss));
    }
    ss = warp_sum(ss);
    part += fabsf(__bfloat162float(w[h])) * sqrtf(ss);
  }
  if (lane == 0) red[warp] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (uint32_t i = 0; i < nw; ++i) tot += red[i];
    at[qi] = tot;
  }
}

template <typename T>
__global__ void index_qrot_kernel(IndexArgs a, float *qrot) {
  const uint32_t qi = blockIdx.x, t = qi % a.T, p = a.pos0 + t;
  const uint32_t Hi = a.n_heads, Di = a.dim, Hp = round_up8(Hi), n_nope = Di - a.rot;
  const T *q = static_cast<const T *>(a.q_idx) + (size_t)qi * Hi * Di;
  float *dst = qrot + (size_t)qi * Di * Hp;
  const T *tag = nullptr;
  for (uint32_t pr = threadIdx.x; pr < Hp * Di / 2; pr += blockDim.x) {
    const uint32_t h = pr / (Di / 2), c = 2 * (pr % (Di / 2));
    float x0 = 0.f, x1 = 0.f;
    if (h < Hi) {
      x0 = ld_f32(q, (size_t)h * Di + c);
      x1 = ld_f32(q, (size_t)h * Di + c + 1);
      if (c >= n_nope) {
        const uint32_t fi = (c - n_nope) / 2;
        const float co = a.cos[(size_t)p * (a.rot / 2) + fi];
        const float si = a.sin[(size_t)p * (a.rot / 2) + fi];
        const float r0 = __fsub_rn(__fmul_rn(x0, co), __fmul_rn(x1, si));
        const float r1 = __fadd_rn(__fmul_rn(x0, si), __fmul_rn(x1, co));
        x0 = round_to(r0, tag);
        x1 = round_to(r1, tag);
      }
    }
    dst[(size_t)c * Hp + h] = x0;
    dst[(size_t)(c + 1) * Hp + h] = x1;
  }
}

template <typename T>
__global__ void __launch_bounds__(kRowsPerBlock)
    index_score_exact_kernel(IndexArgs a, const float *qrot, float *scores) {
  extern __shared__ float4 smem4[];
  const uint32_t qi = blockIdx.y, b = qi / a.T, t = qi % a.T, p = a.pos0 + t;
  const uint32_t vis = min((p + 1) / 4, a.n_comp);
  const uint32_t row0 = blockIdx.x * kRowsPerBlock;
  if (vis <= a.top_k || row0 >= vis) return;
  const uint32_t Hi = a.n_heads, Di = a.dim, Hp = round_up8(Hi), ks_stride = Di + 1;
  float *qs = reinterpret_cast<float *>(smem4);  // [Di][Hp]
  float *ws = qs + (size_t)Di * Hp;              // [Hp]
  float *ks = ws + Hp;                           // [rows][Di + 1]
  const float *qsrc = qrot + (size_t)qi * Di * Hp;
  for (uint32_t i = threadIdx.x; i < Di * Hp; i += blockDim.x) qs[i] = qsrc[i];
  const T *w = static_cast<const T *>(a.w) + (size_t)qi * Hi;
  for (uint32_t h = threadIdx.x; h < Hp; h += blockDim.x) ws[h] = h < Hi ? ld_f32(w, h) : 0.f;
  const T *keys = static_cast<const T *>(a.keys) + (size_t)b * a.comp_cap * Di;
  const uint32_t nrow = min((uint32_t)kRowsPerBlock, vis - row0);
  for (uint32_t i = threadIdx.x; i < nrow * Di; i += blockDim.x) {
    const uint32_t r = i / Di, d = i % Di;
    ks[(size_t)r * ks_stride + d] = ld_f32(keys, (size_t)(row0 + r) * Di + d);
  }
  __syncthreads();
  const uint32_t s = threadIdx.x;
  if (s >= nrow) return;
  const float *kr = ks + (size_t)s * ks_stride;
  float tot = 0.f;
  for (uint32_t hc = 0; hc < Hp; hc += 8) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (uint32_t d = 0; d < Di; ++d) {
      const float kd = kr[d];
      const float4 qa = *reinterpret_cast<const float4 *>(qs + (size_t)d * Hp + hc);
      const float4 qb = *reinterpret_cast<const float4 *>(qs + (size_t)d * Hp + hc + 4);
      acc[0] = __fadd_rn(acc[0], __fmul_rn(qa.x, kd));
      acc[1] = __fadd_rn(acc[1], __fmul_rn(qa.y, kd));
      acc[2] = __fadd_rn(acc[2], __fmul_rn(qa.z, kd));
      acc[3] = __fadd_rn(acc[3], __fmul_rn(qa.w, kd));
      acc[4] = __fadd_rn(acc[4], __fmul_rn(qb.x, kd));
      acc[5] = __fadd_rn(acc[5], __fmul_rn(qb.y, kd));
      acc[6] = __fadd_rn(acc[6], __fmul_rn(qb.z, kd));
      acc[7] = __fadd_rn(acc[7], __fmul_rn(qb.w, kd));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (hc + j < Hi) {
        const float r = acc[j] > 0.f ? acc[j] : 0.f;
        tot = __fadd_rn(tot, __fmul_rn(ws[hc + j], r));
      }
    }
  }
  scores[(size_t)qi * a.comp_cap + row0 + s] = tot;
}

// Order-preserving unsigned key of an fp32 score (+0 and -0 share a key).
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
template <typename KeyF>
__device__ uint32_t radix_kth(KeyF key, uint32_t n, uint32_t k, uint32_t *hist, uint32_t *sel,
                              uint32_t *need_out) {
  uint32_t prefix = 0, mask = 0, need = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (uint32_t s = threadIdx.x; s < n; s += blockDim.x) {
      const uint32_t kk = key(s);
      if ((kk & mask) == prefix) atomicAdd(&hist[(kk >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t cum = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (cum + hist[d] >= need) break;
        cum += hist[d];
      }
      sel[0] = (uint32_t)d;
      sel[1] = cum;
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

// Write, in ascending row order, every row with key > kth and the first
// `need` rows with key == kth (ties to the lower index).
template <typename KeyF>
__device__ void ordered_emit(KeyF key, uint32_t n, uint32_t kth, uint32_t need, uint32_t k,
                             int32_t *out, uint32_t *wsum) {
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
    if (take && pos < k) out[pos] = (int32_t)s;
    eq_seen += eq_tot;
    out_pos += sel_tot;
  }
}

__global__ void __launch_bounds__(kSelectThreads)
    topk_select_kernel(IndexArgs a, const float *scores) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wsum[33];
  __shared__ uint32_t sel[2];
  const uint32_t qi = blockIdx.x, t = qi % a.T, p = a.pos0 + t;
  const uint32_t vis = min((p + 1) / 4, a.n_comp), k = a.top_k;
  int32_t *out = a.topk + (size_t)qi * k;
  if (vis <= k) {
    for (uint32_t j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < vis ? (int32_t)j : -1;
    return;
  }
  const float *sc = scores + (size_t)qi * a.comp_cap;
  auto key = [&](uint32_t s) { return score_key(sc[s]); };
  uint32_t need;
  const uint32_t kth = radix_kth(key, vis, k, hist, sel, &need);
  ordered_emit(key, vis, kth, need, k, out, wsum);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr uint32_t kBandCap = 4096;

// Certified selection for bf16 layers (see the file comment). `cb` bounds the
// relative accumulation error; scores are rewritten in place as exact keys.
__global__ void __launch_bounds__(kSelectThreads)
    topk_certified_kernel(IndexArgs a, TcWs w, float cb) {
  extern __shared__ float4 dyn4[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wsum[33];
  __shared__ uint32_t sel[2];
  __shared__ uint32_t s_nband, s_maxbits;
  const uint32_t Hi = a.n_heads, Di = a.dim;
  float *qT = reinterpret_cast<float *>(dyn4);          // [Di][Hi]
  float *wsh = qT + (size_t)Di * Hi;                    // [Hi]
  float *kbuf = wsh + ((Hi + 3) & ~3u);                 // [32 warps][Di]
  uint32_t *band = reinterpret_cast<uint32_t *>(kbuf + 32 * Di);  // [kBandCap]

  const uint32_t qi = blockIdx.x, b = qi / a.T, t = qi % a.T, p = a.pos0 + t;
  const uint32_t vis = min((p + 1) / 4, a.n_comp), k = a.top_k;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t *out = a.topk + (size_t)qi * k;
  if (vis <= k) {
    for (uint32_t j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < vis ? (int32_t)j : -1;
    return;
  }
  if (*(volatile int *)w.err) {   // the scorer gave up: no valid scores
    for (uint32_t j = threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
    return;
  }
  float *sc = w.scores + (size_t)qi * a.comp_cap;
  const float *nr = w.norms + (size_t)b * a.comp_cap;
  if (threadIdx.x == 0) {
    s_nband = 0;
    s_maxbits = 0;
  }
  __syncthreads();
  float mx = 0.f;
  for (uint32_t s = threadIdx.x; s < vis; s += blockDim.x) mx = fmaxf(mx, nr[s]);
  mx = warp_max(mx);
  if (lane == 0) atomicMax(&s_maxbits, __float_as_uint(mx));
  // approximate k-th largest score
  uint32_t need;
  const float tau =
      key_to_float(radix_kth([&](uint32_t s) { return score_key(sc[s]); }, vis, k, hist, sel, &need));
  const float A = w.at[qi] * cb;
  const float E = A * __uint_as_float(s_maxbits);
  const float hi_cut = tau + E + fabsf(tau) * 2.4e-7f;
  const float lo_cut = tau - E - fabsf(tau) * 2.4e-7f;
  // classify: certainly in -> +inf, certainly out -> -inf, band rows keep S~
  for (uint32_t s = threadIdx.x; s < vis; s += blockDim.x) {
    const float S = sc[s];
    const float e = A * nr[s] + fabsf(S) * 2.4e-7f;
    if (S - e > hi_cut) {
      sc[s] = INFINITY;
    } else if (S + e < lo_cut) {
      sc[s] = -INFINITY;
    } else {
      const uint32_t i = atomicAdd(&s_nband, 1u);
      if (i < kBandCap) band[i] = s;
    }
  }
  // exact-recipe operands: q'^T, w
  const __nv_bfloat16 *qb = w.qbf + (size_t)qi * Hi * Di;
  for (uint32_t i = threadIdx.x; i < Hi * Di; i += blockDim.x) {
    const uint32_t h = i / Di, d = i % Di;
    qT[(size_t)d * Hi + h] = __bfloat162float(qb[i]);
  }
  const __nv_bfloat16 *wq = static_cast<const __nv_bfloat16 *>(a.w) + (size_t)qi * Hi;
  for (uint32_t h = threadIdx.x; h < Hi; h += blockDim.x) wsh[h] = __bfloat162float(wq[h]);
  __syncthreads();
  const __nv_bfloat16 *keys = static_cast<const __nv_bfloat16 *>(a.keys) + (size_t)b * a.comp_cap * Di;
  float *kb = kbuf + (size_t)warp * Di;
  auto rescore = [&](uint32_t s) {
    const __nv_bfloat16 *kr = keys + (size_t)s * Di;
    for (uint32_t d = lane; d < Di; d += 32) kb[d] = __bfloat162float(kr[d]);
    __syncwarp();
    float rel[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t h = lane + 32 * j;
      float acc = 0.f;
      if (h < Hi)
        for (uint32_t d = 0; d < Di; ++d) acc = __fadd_rn(acc, __fmul_rn(qT[(size_t)d * Hi + h], kb[d]));
      rel[j] = acc > 0.f ? acc : 0.f;
    }
    float tot = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      for (uint32_t l = 0; l < 32; ++l) {
        const float r = __shfl_sync(0xffffffffu, rel[j], l);
        const uint32_t h = 32 * j + l;
        if (h < Hi) tot = __fadd_rn(tot, __fmul_rn(wsh[h], r));
      }
    }
    __syncwarp();
    if (lane == 0) sc[s] = tot;
  };
  const uint32_t nband = s_nband;
  if (nband <= kBandCap) {
    for (uint32_t i = warp; i < nband; i += blockDim.x / 32) rescore(band[i]);
  } else {
    for (uint32_t s = warp; s < vis; s += blockDim.x / 32) {
      const float v = sc[s];
      if (v != INFINITY && v != -INFINITY) rescore(s);
    }
  }
  __syncthreads();
  auto key = [&](uint32_t s) { return score_key(sc[s]); };
  const uint32_t kth = radix_kth(key, vis, k, hist, sel, &need);
  ordered_emit(key, vis, kth, need, k, out, wsum);
}

template <typename T>
cudaError_t launch_index_exact(const IndexArgs &a, cudaStream_t s) {
  const uint32_t nq = a.batch * a.T;
  IndexWs w = index_ws_split(a.ws, nq, a.n_heads, a.dim);
  index_qrot_kernel<T><<<nq, 256, 0, s>>>(a, w.qrot);
  note_launches(1);
  const uint32_t Hp = round_up8(a.n_heads);
  const size_t smem = ((size_t)a.dim * Hp + Hp + (size_t)kRowsPerBlock * (a.dim + 1)) * 4;
  static int smem_set = 0;
  cudaError_t e = ensure_smem(index_score_exact_kernel<T>, smem, &smem_set);
  if (e != cudaSuccess) return e;
  const uint32_t vis_max = min((a.pos0 + a.T) / 4, a.n_comp);
  if (vis_max > a.top_k) {
    dim3 grid((vis_max + kRowsPerBlock - 1) / kRowsPerBlock, nq);
    index_score_exact_kernel<T><<<grid, kRowsPerBlock, smem, s>>>(a, w.qrot, w.scores);
    note_launches(1);
  }
  topk_select_kernel<<<nq, kSelectThreads, 0, s>>>(a, w.scores);
  note_launches(1);
  return cudaGetLastError();
}

// gamma_n = n u / (1 - n u), u = 2^-24: bound of n roundings in fp32.
inline double gamma_n(double n) {
  const double u = std::ldexp(1.0, -24);
  return n * u / (1.0 - n * u);
}

cudaError_t launch_index_tc(const IndexArgs &a, cudaStream_t s) {
  const uint32_t nq = a.batch * a.T;
  TcWs w = tc_ws_split(a.ws, nq, a.batch, a.n_heads, a.dim, a.comp_cap, nullptr);
  index_qbf_kernel<<<nq, 256, 0, s>>>(a, w.qbf, w.at, w.err);
  note_launches(1);
  const uint32_t vis_max = min((a.pos0 + a.T) / 4, a.n_comp);
  if (vis_max > a.top_k) {
    IndexTcArgs t;
    t.batch = a.batch;
    t.T = a.T;
    t.pos0 = a.pos0;
    t.comp_cap = a.comp_cap;
    t.n_comp = a.n_comp;
    t.keys = a.keys;
    t.qbf = w.qbf;
    t.w = a.w;
    t.scores = w.scores;
    t.norms = w.norms;
    t.err = w.err;
    cudaError_t e = launch_index_score_tc(t, s);
    if (e != cudaSuccess) return e;
  }
  // |S~ - S| <= cb * A_t * ||k_s||: the exact recipe (Di products, Hi weighted
  // terms) and the tensor-core accumulation (taken as at most 4 Di fp32
  // roundings) plus the fp32 epilogue; widened for the fp32 norms.
  const double cb = (gamma_n(a.dim + a.n_heads + 1) + gamma_n(4.0 * a.dim + a.n_heads + 1)) *
                    (1.0 + std::ldexp(1.0, -8));
  const size_t smem = ((size_t)a.dim * a.n_heads + ((a.n_heads + 3) & ~3u) + 32 * (size_t)a.dim) * 4 +
                      kBandCap * 4;
  static int smem_set = 0;
  cudaError_t e = ensure_smem(topk_certified_kernel, smem, &smem_set);
  if (e != cudaSuccess) return e;
  topk_certified_kernel<<<nq, kSelectThreads, smem, s>>>(a, w, (float)cb);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

size_t index_ws_bytes(int dtype, uint32_t batch, uint32_t T, uint32_t n_heads, uint32_t dim,
                      uint32_t comp_cap) {
  const size_t nq = (size_t)batch * T;
  if (dtype == DS4A_BF16 && index_tc_supported(n_heads, dim)) {
    size_t total = 0;
    tc_ws_split(nullptr, (uint32_t)nq, batch, n_heads, dim, comp_cap, &total);
    return total;
  }
  const size_t qsz = nq * dim * round_up8(n_heads);
  return (((qsz + 63) & ~(size_t)63) + nq * comp_cap) * sizeof(float);
}

cudaError_t launch_index_topk(const IndexArgs &a, cudaStream_t s) {
  if (a.dtype == DS4A_BF16) {
    if (index_tc_supported(a.n_heads, a.dim)) return launch_index_tc(a, s);
    return launch_index_exact<__nv_bfloat16>(a, s);
  }
  return launch_index_exact<float>(a, s);
}

}  // namespace ds4a
