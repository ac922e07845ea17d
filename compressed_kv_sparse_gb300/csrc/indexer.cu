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

#include "quant.cuh"
#include "select.cuh"
#include "tc.cuh"

namespace ds4a {
namespace {

constexpr int kRowsPerBlock = 128;
constexpr int kSelectThreads = 1024;

__host__ __device__ inline uint32_t round_up8(uint32_t x) { return (x + 7u) & ~7u; }

// Workspace layout: the error word (int32, then padding to 256 bytes; this
// path has no device waits, so the query rotation only zeroes it), qrot
// [B*T][Di][Hpad] fp32, then scores [B*T][comp_cap] fp32.
constexpr size_t kExactWsHeader = 256;
struct IndexWs {
  int *err;
  float *qrot, *scores;
};
__host__ __device__ inline IndexWs index_ws_split(void *ws, uint32_t nq, uint32_t Hi,
                                                  uint32_t Di) {
  float *base = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kExactWsHeader);
  const size_t qsz = (size_t)nq * Di * round_up8(Hi);
  return IndexWs{static_cast<int *>(ws), base, base + ((qsz + 63) & ~(size_t)63)};
}

// Workspace of bf16 layers: err word, qbf [nq][Hi][Di] bf16, scores
// [nq][comp_cap rounded up to 32] (fp32) and per-query histograms of the
// scores' top 12 key bits [nq][4096]. The row norms of the error bound live
// in the cache (written when rows are appended).
struct TcWs {
  int *err;
  float *scores;        // [nq][sstride]
  __nv_bfloat16 *qbf;
  uint32_t *hist;
  float *qnorm;         // [nq][Hi] upper bound of ||q'_h||
  uint32_t *qexp;       // [nq][Hi] exponent range of the nonzero entries of q'_h:
                        // int16 minimum | int16 maximum << 16 (1000 | -1000: all zero)
  uint32_t sstride;     // floats per query row of scores: comp_cap rounded up to 32
};
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline TcWs tc_ws_split(void *ws, uint32_t nq, uint32_t B, uint32_t Hi, uint32_t Di,
                        uint32_t comp_cap, size_t *total) {
  uint8_t *base = static_cast<uint8_t *>(ws);
  size_t off = 0;
  TcWs w;
  w.err = reinterpret_cast<int *>(base + off);
  off = align_up(off + 16, 1024);
  w.qbf = reinterpret_cast<__nv_bfloat16 *>(base + off);
  off = align_up(off + (size_t)nq * Hi * Di * 2, 256);
  w.sstride = (comp_cap + 31u) & ~31u;   // 128-byte aligned rows (bulk copies)
  w.scores = reinterpret_cast<float *>(base + off);
  off = align_up(off + (size_t)nq * w.sstride * 4, 256);
  w.hist = reinterpret_cast<uint32_t *>(base + off);
  off = align_up(off + (size_t)nq * kHistBins * 4, 256);
  w.qnorm = reinterpret_cast<float *>(base + off);
  off = align_up(off + (size_t)nq * Hi * 4, 256);
  w.qexp = reinterpret_cast<uint32_t *>(base + off);
  off += (size_t)nq * Hi * 4;
  if (total) *total = off;
  return w;
}

// bf16 layers: q' = rotated query rounded to bf16 (fp32 recipe), one thread
// per `per` dims (a 16-byte unit of 8, or a pair when the query is not 16-byte
// aligned); the same grid clears the call's error word and, when the scorer
// builds them, the key histograms. With the FP4 QAT round
// trip, units are always 8 dims (loaded one by one when `vec` is false) and
// the Di / 8 lanes of a head row run the transform together.
__global__ void index_qbf_kernel(IndexArgs a, TcWs w, bool clear_hist, bool vec) {
  pdl_wait();
  pdl_trigger();
  // one thread per 8 dims: a head row of Di = 128 dims is an aligned group of
  // 16 lanes
  constexpr uint32_t per = 8;
  const uint32_t Hi = a.n_heads, Di = a.dim, n_nope = Di - a.rot;
  const uint32_t nq = a.batch * a.T;
  const uint32_t upr = Di / per;                  // lanes per head row
  const uint32_t n_units = nq * Hi * upr;         // a multiple of 32
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0) *w.err = 0;
  if (clear_hist && i < nq * (kHistBins / 4))
    reinterpret_cast<uint4 *>(w.hist)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (i >= n_units) return;
  const uint32_t row = i / upr, c0 = (i - row * upr) * per;   // row = query * Hi + head
  const uint32_t p = seq_base(a.seq_pos, a.pos0, (row / Hi) / a.T) + (row / Hi) % a.T;
  const uint32_t lane = threadIdx.x & 31;
  // the 8 bf16 inputs as pairs (16-byte loads when aligned)
  uint32_t w4[4];
  if (vec) {
    const uint4 q4 = reinterpret_cast<const uint4 *>(a.q_idx)[i];
    w4[0] = q4.x;
    w4[1] = q4.y;
    w4[2] = q4.z;
    w4[3] = q4.w;
  } else {
    const uint16_t *q = static_cast<const uint16_t *>(a.q_idx) + (size_t)i * per;
#pragma unroll
    for (int e = 0; e < 4; ++e) w4[e] = (uint32_t)q[2 * e] | ((uint32_t)q[2 * e + 1] << 16);
  }
  if (a.qat) {   // uniform
    float v[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = __uint_as_float(w4[e] << 16);
      v[2 * e + 1] = __uint_as_float(w4[e] & 0xFFFF0000u);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t c = c0 + 2 * e;
      if (c < n_nope) continue;
      const uint32_t fi = (c - n_nope) / 2;
      const float co = a.cos[(size_t)p * (a.rot / 2) + fi];
      const float si = a.sin[(size_t)p * (a.rot / 2) + fi];
      const float x0 = v[2 * e], x1 = v[2 * e + 1];
      v[2 * e] = __fsub_rn(__fmul_rn(x0, co), __fmul_rn(x1, si));
      v[2 * e + 1] = __fadd_rn(__fmul_rn(x0, si), __fmul_rn(x1, co));
    }
    const uint32_t mask = ((1u << upr) - 1u) << (lane & ~(upr - 1u));
    fp4_qat_lanes8(v, lane & (upr - 1u), upr, mask, a.had_c);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 r = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
      w4[e] = *reinterpret_cast<const uint32_t *>(&r);
    }
  } else if (c0 + per > n_nope) {
    // rotate the pairs that lie in the tail
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t c = c0 + 2 * e;
      if (c < n_nope) continue;
      const float x0 = __uint_as_float(w4[e] << 16), x1 = __uint_as_float(w4[e] & 0xFFFF0000u);
      const uint32_t fi = (c - n_nope) / 2;
      const float co = a.cos[(size_t)p * (a.rot / 2) + fi];
      const float si = a.sin[(size_t)p * (a.rot / 2) + fi];
      const float r0 = __fsub_rn(__fmul_rn(x0, co), __fmul_rn(x1, si));
      const float r1 = __fadd_rn(__fmul_rn(x0, si), __fmul_rn(x1, co));
      const __nv_bfloat162 r = __floats2bfloat162_rn(r0, r1);
      w4[e] = *reinterpret_cast<const uint32_t *>(&r);
    }
  }
  reinterpret_cast<uint4 *>(w.qbf)[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  // per head row of the stored q': an upper bound of its Euclidean norm (from
  // squares scaled by 2^-e, e the exponent of its largest |value|, so tiny
  // magnitudes do not underflow) and the exponent range of its nonzero
  // entries, for the selection's error bound and exactness test
  // (the exponent range is that of the smallest nonzero and the largest
  // magnitude: the exponent grows with the magnitude)
  float x[8], mx = 0.f, mn = INFINITY;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = __uint_as_float(w4[e] << 16);
    x[2 * e + 1] = __uint_as_float(w4[e] & 0xFFFF0000u);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float ax = fabsf(x[e]);
    mx = fmaxf(mx, ax);
    mn = fminf(mn, ax > 0.f ? ax : INFINITY);
  }
#pragma unroll
  for (uint32_t o = upr / 2; o > 0; o >>= 1) {   // within the 16-lane group
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  // mx = f 2^eh with f in [0.5, 1); scaling by 2^-eh is one multiply,
  // rounded like ldexpf, while 2^-eh is a normal fp32 value (biased exponent
  // of mx in 1 .. 252), else ldexpf
  int eh = 0;
  float ss = 0.f;
  const uint32_t mb = __float_as_uint(mx) >> 23;   // biased exponent (mx >= 0)
  if (mb >= 1u && mb <= 252u) {
    eh = (int)mb - 126;
    const float sc = __uint_as_float((uint32_t)(127 - eh) << 23);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float y = x[e] * sc;
      ss = fmaf(y, y, ss);
    }
  } else if (mx > 0.f) {
    frexpf(mx, &eh);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float y = ldexpf(x[e], -eh);
      ss = fmaf(y, y, ss);
    }
  }
#pragma unroll
  for (uint32_t o = upr / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((lane & (upr - 1u)) == 0) {
    const int emin = mx > 0.f ? exp_of(mn) : 1000, emax = mx > 0.f ? exp_of(mx) : -1000;
    w.qnorm[row] = mx > 0.f ? norm_from_scaled(ss, eh) : 0.f;
    w.qexp[row] = ((uint32_t)emin & 0xFFFFu) | ((uint32_t)emax << 16);
  }
}

template <typename T>
__global__ void index_qrot_kernel(IndexArgs a, float *qrot, int *err) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *err = 0;
  const uint32_t qi = blockIdx.x, t = qi % a.T, p = seq_base(a.seq_pos, a.pos0, qi / a.T) + t;
  const uint32_t Hi = a.n_heads, Di = a.dim, Hp = round_up8(Hi), n_nope = Di - a.rot;
  const T *q = static_cast<const T *>(a.q_idx) + (size_t)qi * Hi * Di;
  float *dst = qrot + (size_t)qi * Di * Hp;
  const T *tag = nullptr;
  if (a.qat) {   // uniform: one head at a time through shared memory
    __shared__ float buf[256];
    for (uint32_t h = 0; h < Hp; ++h) {
      if (h >= Hi) {
        for (uint32_t c = threadIdx.x; c < Di; c += blockDim.x) dst[(size_t)c * Hp + h] = 0.f;
        continue;
      }
      for (uint32_t pr = threadIdx.x; pr < Di / 2; pr += blockDim.x) {
        const uint32_t c = 2 * pr;
        float x0 = ld_f32(q, (size_t)h * Di + c), x1 = ld_f32(q, (size_t)h * Di + c + 1);
        if (c >= n_nope) {
          const uint32_t fi = (c - n_nope) / 2;
          const float co = a.cos[(size_t)p * (a.rot / 2) + fi];
          const float si = a.sin[(size_t)p * (a.rot / 2) + fi];
          const float r0 = __fsub_rn(__fmul_rn(x0, co), __fmul_rn(x1, si));
          const float r1 = __fadd_rn(__fmul_rn(x0, si), __fmul_rn(x1, co));
          x0 = r0;
          x1 = r1;
        }
        buf[c] = x0;
        buf[c + 1] = x1;
      }
      __syncthreads();
      fp4_qat_smem(buf, Di, a.had_c);
      for (uint32_t c = threadIdx.x; c < Di; c += blockDim.x)
        dst[(size_t)c * Hp + h] = round_to(buf[c], tag);
      __syncthreads();
    }
    return;
  }
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
  const uint32_t qi = blockIdx.y, b = qi / a.T, t = qi % a.T;
  const uint32_t p = seq_base(a.seq_pos, a.pos0, b) + t;
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
  const T *keys = static_cast<const T *>(a.keys);
  const uint32_t nrow = min((uint32_t)kRowsPerBlock, vis - row0);
  for (uint32_t i = threadIdx.x; i < nrow * Di; i += blockDim.x) {
    const uint32_t r = i / Di, d = i % Di;
    ks[(size_t)r * ks_stride + d] = ld_f32(keys, a.map.row_of(b, row0 + r) * Di + d);
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

__global__ void __launch_bounds__(kSelectThreads)
    topk_select_kernel(IndexArgs a, const float *scores) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wsum[33];
  __shared__ uint32_t sel[2];
  const uint32_t qi = blockIdx.x, t = qi % a.T, p = seq_base(a.seq_pos, a.pos0, qi / a.T) + t;
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
  ordered_emit(key, vis, kth, need, k, out, wsum, [](uint32_t x) { return x; });
}

// Select kernel configurations: 1024 threads when several blocks share a
// query (decode), 256 when each query has one block (prefill, large batches;
// four blocks per SM then overlap their latency chains).
template <int NT>
struct SelCfg {
  static constexpr int NW = NT / 32;                  // warps
  static constexpr int BPT = 4096 / NT;               // histogram bins per thread
  static constexpr int RPR = 2 * NW;                  // band rows per rescoring round
  static constexpr uint32_t CAP = NT == 1024 ? 4096u : 1536u;   // candidates in smem
  static constexpr uint32_t BANDCAP = CAP < 2048u ? CAP : 2048u;
  static constexpr size_t kScratch =
      (size_t)(4096 * 4 > RPR * 192 * 4 ? (4096 * 4 > BANDCAP * 8 ? 4096 * 4 : BANDCAP * 8)
                                        : (RPR * 192 * 4 > BANDCAP * 8 ? RPR * 192 * 4
                                                                      : BANDCAP * 8));
  static size_t smem(uint32_t comp_cap) {
    const size_t words = (comp_cap + 31) / 32;
    return 64 * kQB * 2 + 64 * 4 + kScratch + 3 * (size_t)CAP * 4 + words * 4;
  }
};

// Blocks per query: one wave of 1024-thread blocks (one per SM), at most 16.
inline uint32_t select_groups(uint32_t nq) {
  uint32_t g = (uint32_t)num_sms() / (nq ? nq : 1);
  return g < 1 ? 1 : (g > 8 ? 8 : g);
}

// Certified selection for bf16 layers (64 heads x 128 dims).
//
// Every row's exact score lies in [L_s, U_s] = [S~_s - e_s, S~_s + e_s] with
// e_s = A ||k_s|| (+ rounding slack), A = c * sum_h |w_h| ||q'_h||. The score
// kernel counted the top 12 key bits of S~ per query; the bin holding the k-th
// largest gives theta_S with at least k rows S~ >= theta_S, so with
// E = A max ||k|| and theta = theta_S - E (- slack) at least k rows have
// L_s >= theta, and every row with U_s < theta is beaten by k rows. The G
// blocks of a query form a thread-block cluster: each filters its share of
// the rows into the candidate lists of the cluster's first block
// (distributed shared memory), bounding every row's error with the largest
// row norm (a superset of the rows with U_s >= theta; one block per query
// takes theta_S from a sample of the scores instead). After one cluster
// barrier that block gives each candidate its own bound from its norm and
// runs the certified selection on the candidates: tau~ = k-th largest S~,
// rows with L_s > tau~ + E are in, rows with U_s < tau~ - E are out, the rest
// are rescored with the exact recipe and the final selection is exact (ties
// to the lower index). If the candidates overflow, the same selection runs
// over every visible row in place.
template <int NT>
__global__ void __launch_bounds__(NT, NT == 256 ? 4 : 1)
    topk_select_tc_kernel(IndexArgs a, TcWs w, float cb, uint32_t G) {
  using SC = SelCfg<NT>;
  constexpr uint32_t CAP = SC::CAP;
  extern __shared__ float4 dyn4[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wsum[33];
  __shared__ uint32_t sel[2];
  // bin of the k-th key, last-block flag, band count, tie / in count, keys above
  // the bin, second-level bin
  __shared__ uint32_t s_misc[6];
  __shared__ float s_red[32], s_wabs[32];
  __shared__ int s_qexp[2];        // exponent range of the nonzero q' entries
  __shared__ uint32_t s_rexact[SC::RPR];  // band round: fma is exact for the row
  __nv_bfloat16 *qsm = reinterpret_cast<__nv_bfloat16 *>(dyn4);   // [64][kQB]
  float *wsh = reinterpret_cast<float *>(qsm + 64 * kQB);           // [64]
  // scratch, used in turn by: the second-level histogram [4096]; the band
  // rescoring's keys [RPR][128] and ReLU dots [RPR][64]; the band values and
  // rows [BANDCAP] + [BANDCAP]
  float *scratch = wsh + 64;
  float *kbuf = scratch, *relb = scratch + SC::RPR * 128;
  uint32_t *cidx = reinterpret_cast<uint32_t *>(scratch + SC::kScratch / 4);   // [CAP]
  float *cS = reinterpret_cast<float *>(cidx + CAP);                           // [CAP]
  float *ce = cS + CAP;                                                        // [CAP]
  uint32_t *bitmap = reinterpret_cast<uint32_t *>(ce + CAP);   // [comp_cap / 32]

  const uint32_t Hi = 64, Di = 128;
  const uint32_t qi = blockIdx.x / G, g = blockIdx.x % G;
  const uint32_t b = qi / a.T, p = seq_base(a.seq_pos, a.pos0, b) + qi % a.T;
  const uint32_t vis = min((p + 1) / 4, a.n_comp), k = a.top_k;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t *out = a.topk + (size_t)qi * k;
  if (vis <= k) {
    pdl_wait();
    pdl_trigger();
    if (g == 0)
      for (uint32_t j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < vis ? (int32_t)j : -1;
    return;
  }
  float *sc = w.scores + (size_t)qi * w.sstride;
  const float *nr = a.norms;   // row r of this sequence: nr[a.map.row_of(b, r)]
  const float *nr_c = a.map.table ? nullptr : a.norms + (size_t)b * a.comp_cap;   // contiguous
  const __nv_bfloat16 *qb = w.qbf + (size_t)qi * Hi * Di;
  const __nv_bfloat16 *wq = static_cast<const __nv_bfloat16 *>(a.w) + (size_t)qi * Hi;

  // A = c * sum_h |w_h| ||q'_h|| and the exponent range of the nonzero
  // entries of q', from the per-head norms and ranges the query rotation
  // wrote (warps 0 and 1, one head per lane); q' rows to shared memory
  if (threadIdx.x == 0) {
    s_qexp[0] = 1000;
    s_qexp[1] = -1000;
  }
  __syncthreads();
  if (warp < 2) {
    const uint32_t h = threadIdx.x;
    const float wv = __bfloat162float(wq[h]), wa = fabsf(wv);
    const uint32_t ex = w.qexp[(size_t)qi * Hi + h];
    const float part = warp_sum(wa * w.qnorm[(size_t)qi * Hi + h]);
    const float wabs = warp_sum(wa);
    const int emin = warp_min_i((int)(int16_t)(ex & 0xFFFFu));
    const int emax = warp_max_i((int)(int16_t)(ex >> 16));
    if (lane == 0) {
      s_red[warp] = part;
      s_wabs[warp] = wabs;
      atomicMin(&s_qexp[0], emin);
      atomicMax(&s_qexp[1], emax);
    }
    wsh[h] = wv;
  }
  // (asynchronous: the rows are first read by the rescoring, after the
  // waits at the start of the selection)
  for (uint32_t i = threadIdx.x; i < Hi * (Di / 4); i += NT) {
    const uint32_t h = i / (Di / 4), c = 4 * (i % (Di / 4));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(qsm + (size_t)h * kQB + c)),
                 "l"(qb + (size_t)h * Di + c)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  // everything above read only what was written two or more launches back
  // (q', head weights, row norms); the scores and histograms need the scorer
  pdl_wait();
  pdl_trigger();
  // did the scorer give up? (tested once the threshold's loads are in flight)
  const int scorer_err = *(volatile int *)w.err;
  // theta_S: at least k rows have S~ >= theta_S. Several blocks per query:
  // the lower edge of the scorer's histogram bin holding the k-th largest.
  // One block per query: a value of an evenly strided sample of the scores at
  // a rank that leaves ~1.6 k rows above it; the filter below counts the rows
  // at or above it exactly, and too few sends the block to the full pass.
  if (threadIdx.x == 0) {
    s_misc[2] = 0;   // candidates (several blocks: the cluster's count, in its first block)
    s_misc[3] = 0;   // rows with S~ >= theta_S (one block per query)
  }
  // several blocks per query form a cluster: every block appends its
  // candidates to the first block's lists, whose count is zeroed above
  if (G > 1) cluster_arrive();
  float theta_s;
  if (G > 1) {
    const uint32_t *hq = w.hist + (size_t)qi * kHistBins;
    uint32_t cb4[SC::BPT], loc = 0;
#pragma unroll
    for (uint32_t j = 0; j < (uint32_t)SC::BPT; ++j) {
      cb4[j] = hq[kHistBins - 1 - (SC::BPT * threadIdx.x + j)];
      loc += cb4[j];
    }
    uint32_t tot;
    uint32_t cum = block_excl_scan(loc, wsum, &tot);   // also syncs s_red / wsh / qsm
    if (cum < k && cum + loc >= k) {
#pragma unroll
      for (uint32_t j = 0; j < (uint32_t)SC::BPT; ++j) {
        if (cum + cb4[j] >= k) {
          s_misc[0] = kHistBins - 1 - (SC::BPT * threadIdx.x + j);
          s_misc[4] = cum;
          break;
        }
        cum += cb4[j];
      }
    }
    __syncthreads();
    theta_s = key_to_float(s_misc[0] << 20);
  } else {
    constexpr uint32_t kSampleCap = (uint32_t)(SC::kScratch / 4);
    const uint32_t stride = max(16u, (vis + kSampleCap - 1) / kSampleCap);
    const uint32_t ns = vis / stride;   // >= 32: vis > k >= 512
    float *smp = scratch;
    for (uint32_t j = threadIdx.x; j < ns; j += blockDim.x) smp[j] = sc[j * stride + stride / 2];
    __syncthreads();   // (also syncs s_red / wsh / qsm)
    // (the sample's rank-r value has ~stride * r rows above it, give or take
    // ~stride * sqrt(r): 1.6 k leaves about three of those above k, so the
    // exact count rarely sends the block to the full pass)
    const uint32_t rs = min(ns, ((k + stride - 1) / stride) * 8 / 5 + 8);
    uint32_t need_s;
    // (three digits: the lower edge of the 24-bit key bin of that value,
    // a relative 2^-15 below it at most)
    theta_s = key_to_float(radix_kth([&](uint32_t j) { return score_key(smp[j]); }, ns, rs,
                                     hist, sel, &need_s, 8));
  }
  if (scorer_err) {   // no scores: no list
    if (g == 0)
      for (uint32_t j = threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
    return;
  }
  __syncthreads();
  float At = 0.f, Wt = 0.f;
  for (uint32_t i = 0; i < 2; ++i) {
    At += s_red[i];
    Wt += s_wabs[i];
  }
  const float A = At * (1.0f + 1e-5f) * cb;
  // absolute term for underflow: tensor-core products and partial sums that
  // flush to zero (each off by < 2^-126) and the subnormal roundings of both
  // computations, for 4 Di operations per head dot and 4 Hi per score
  const float eta = (4.0f * (float)Di * Wt * (1.0f + 1e-5f) + 4.0f * (float)Hi) * 0x1p-126f;
  const float E = A * __uint_as_float(a.norm_max[b]) + eta;
  const int eq_min = s_qexp[0], eq_max = s_qexp[1];
  const float theta = theta_s - E - fabsf(theta_s) * (2.0f * kRel);
  auto err_of = [&](float S, float nm) { return A * nm + fabsf(S) * kRel + eta; };

  // ---- this block's share of the rows: candidates with U >= theta, gathered
  // in shared memory (four rows per thread loaded before any is classified):
  // the block's own lists, or, with several blocks per query, the lists of
  // the cluster's first block (slots from its count, stores through
  // distributed shared memory), which then finishes alone
  if (G > 1) cluster_wait();
  const uint32_t c_cnt = mapa_shared(smem_u32(&s_misc[2]), 0);
  const uint32_t c_idx = mapa_shared(smem_u32(cidx), 0), c_S = mapa_shared(smem_u32(cS), 0);
  {
    const uint32_t per = ((vis + G * 32 - 1) / (G * 32)) * 32;
    const uint32_t r0 = g * per, r1 = min(vis, r0 + per);
    // four consecutive rows per thread and step (one 16-byte load where the
    // four are whole: the score rows are 16-byte aligned), three steps in
    // flight. The test bounds each row's error with the largest row norm (a
    // superset of the rows with U >= theta, no norm loads); the candidates'
    // own bounds follow from their norms below.
    constexpr uint32_t J = 3;
    uint32_t n_ge = 0;   // rows with S~ >= theta_S (one block per query)
    for (uint32_t pass = r0; pass < r1; pass += J * 4 * NT) {
      float Sv[J][4];
#pragma unroll
      for (uint32_t j = 0; j < J; ++j) {
        const uint32_t rb = pass + 4 * (j * NT + threadIdx.x);
        if (rb + 4 <= r1) {
          const float4 s4 = *reinterpret_cast<const float4 *>(sc + rb);
          Sv[j][0] = s4.x;
          Sv[j][1] = s4.y;
          Sv[j][2] = s4.z;
          Sv[j][3] = s4.w;
        } else {
#pragma unroll
          for (uint32_t u = 0; u < 4; ++u) Sv[j][u] = rb + u < r1 ? sc[rb + u] : 0.f;
        }
      }
#pragma unroll
      for (uint32_t j = 0; j < J; ++j) {
#pragma unroll
        for (uint32_t u = 0; u < 4; ++u) {
          const uint32_t r = pass + 4 * (j * NT + threadIdx.x) + u;
          const bool ok = r < r1;
          const float S = Sv[j][u];
          const bool c = ok && S + (E + fabsf(S) * kRel) >= theta;
          n_ge += (ok && S >= theta_s) ? 1u : 0u;
          const uint32_t bal = __ballot_sync(0xffffffffu, c);
          if (bal) {
            uint32_t slot = 0;
            if (lane == 0)
              slot = G > 1 ? atom_add_cluster(c_cnt, (uint32_t)__popc(bal))
                           : atomicAdd(&s_misc[2], (uint32_t)__popc(bal));
            slot = __shfl_sync(0xffffffffu, slot, 0) + __popc(bal & ((1u << lane) - 1u));
            if (c && slot < CAP) {
              if (NT == 1024) {   // (only this width runs several blocks per query)
                st_cluster_u32(c_idx + 4 * slot, r);
                st_cluster_u32(c_S + 4 * slot, __float_as_uint(S));
              } else {
                cidx[slot] = r;
                cS[slot] = S;
              }
            }
          }
        }
      }
    }
    if (G == 1) {
      n_ge = warp_sum_u32(n_ge);
      if (lane == 0 && n_ge) atomicAdd(&s_misc[3], n_ge);
    }
  }
  if (G > 1) {
    // every block's candidates are in the first block's lists: it finishes
    cluster_arrive();
    cluster_wait();
    if (g != 0) return;
  } else {
    __syncthreads();
  }

  const __nv_bfloat16 *keys = static_cast<const __nv_bfloat16 *>(a.keys);   // rows via a.map
  float *kb = kbuf + warp * 128, *rel = relb + warp * 64;
  const uint32_t nc = s_misc[2];
  const bool fast = nc <= CAP && (G == 1 ? s_misc[3] >= k : true);
  uint32_t need;
  asm volatile("cp.async.wait_all;" ::: "memory");   // (this thread's q' rows)
  if (fast) {
    // each candidate's own error bound, from its row norm (read by the
    // classification, several barriers on)
    for (uint32_t j = threadIdx.x; j < nc; j += blockDim.x) {
      const uint32_t r = cidx[j];
      ce[j] = err_of(cS[j], nr_c ? nr_c[r] : nr[a.map.row_of(b, r)]);
    }
    // ---- certified selection on the candidates
    if (threadIdx.x == 0) s_misc[5] = 0u;
    __syncthreads();
    const uint32_t words = (vis + 31) / 32;
    for (uint32_t i = threadIdx.x; i < words; i += blockDim.x) bitmap[i] = 0u;
    if (G == 1) {
      // every row with S~ >= theta_S (at least k) is a candidate, so the k-th
      // largest S~ is the candidates' k-th: its 12-bit key bin b* and the
      // count above it from a histogram of the candidates
      uint32_t *h1 = reinterpret_cast<uint32_t *>(scratch);   // [4096]
      for (uint32_t i = threadIdx.x; i < kHistBins; i += blockDim.x) h1[i] = 0u;
      __syncthreads();
      for (uint32_t j = threadIdx.x; j < nc; j += blockDim.x)
        atomicAdd(&h1[score_key(cS[j]) >> 20], 1u);
      __syncthreads();
      uint32_t cb4[SC::BPT], loc = 0;
#pragma unroll
      for (uint32_t j = 0; j < (uint32_t)SC::BPT; ++j) {
        cb4[j] = h1[kHistBins - 1 - (SC::BPT * threadIdx.x + j)];
        loc += cb4[j];
      }
      uint32_t tot;
      uint32_t cum = block_excl_scan(loc, wsum, &tot);
      if (cum < k && cum + loc >= k) {
#pragma unroll
        for (uint32_t j = 0; j < (uint32_t)SC::BPT; ++j) {
          if (cum + cb4[j] >= k) {
            s_misc[0] = kHistBins - 1 - (SC::BPT * threadIdx.x + j);
            s_misc[4] = cum;
            break;
          }
          cum += cb4[j];
        }
      }
      __syncthreads();
    }
    // the k-th largest S~ lies in 12-bit key bin b* with `above` keys over it;
    // a histogram of the next 12 key bits of the candidates in b* narrows it
    // to one 24-bit key interval [t_lo, t_hi] (every row of b* is a candidate)
    uint32_t *h2 = reinterpret_cast<uint32_t *>(kbuf);   // [4096], free until rescoring
    for (uint32_t i = threadIdx.x; i < kHistBins; i += blockDim.x) h2[i] = 0u;
    __syncthreads();
    const bool cand_ok = s_misc[5] == 0u;
    __syncthreads();
    if (threadIdx.x == 0) s_misc[5] = 0xffffffffu;
    __syncthreads();
    const uint32_t bstar = s_misc[0], need_b = k - s_misc[4];
    for (uint32_t j = threadIdx.x; j < nc; j += blockDim.x) {
      const uint32_t kk = score_key(cS[j]);
      if ((kk >> 20) == bstar) atomicAdd(&h2[(kk >> 8) & (kHistBins - 1)], 1u);
    }
    __syncthreads();
    {
      uint32_t cb4[SC::BPT], loc = 0;
#pragma unroll
      for (uint32_t j = 0; j < (uint32_t)SC::BPT; ++j) {
        cb4[j] = h2[kHistBins - 1 - (SC::BPT * threadIdx.x + j)];
        loc += cb4[j];
      }
      uint32_t tot;
      uint32_t cum = block_excl_scan(loc, wsum, &tot);
      if (cum < need_b && cum + loc >= need_b) {
#pragma unroll
        for (uint32_t j = 0; j < (uint32_t)SC::BPT; ++j) {
          if (cum + cb4[j] >= need_b) {
            s_misc[5] = kHistBins - 1 - (SC::BPT * threadIdx.x + j);
            break;
          }
          cum += cb4[j];
        }
      }
    }
    __syncthreads();
    bool ok = cand_ok && s_misc[5] != 0xffffffffu;
    const uint32_t kpre = (bstar << 20) | (s_misc[5] << 8);
    const float t_lo = key_to_float(kpre), t_hi = key_to_float(kpre | 0xffu);
    // rows with L > t_hi + E beat the exact k-th score, rows with U < t_lo - E
    // are beaten by k rows; only the band between can hold or tie the k-th
    const float hi_cut = t_hi + E + fabsf(t_hi) * kRel;
    const float lo_cut = t_lo - E - fabsf(t_lo) * kRel;
    if (threadIdx.x == 0) {
      s_misc[1] = 0;   // band compaction slots (the ticket flag is no longer read)
      s_misc[2] = 0;
      s_misc[3] = 0;
    }
    __syncthreads();
    uint32_t cls = 0;   // 2 bits per candidate of this thread: 1 in, 2 band
    static_assert(CAP / NT <= 16, "two class bits per candidate of a thread");
    if (ok) {
      for (uint32_t j = threadIdx.x, u = 0; j < nc; j += blockDim.x, ++u) {
        const float S = cS[j], e = ce[j];
        if (S - e > hi_cut) {
          cls |= 1u << (2 * u);
          atomicOr(&bitmap[cidx[j] >> 5], 1u << (cidx[j] & 31));
        } else if (S + e >= lo_cut) {
          cls |= 2u << (2 * u);
        }
      }
      const uint32_t n_in = __popc(cls & 0x55555555u), n_band = __popc(cls & 0xaaaaaaaau);
      const uint32_t wi = warp_sum_u32(n_in), wb = warp_sum_u32(n_band);
      if (lane == 0) {
        if (wi) atomicAdd(&s_misc[3], wi);
        if (wb) atomicAdd(&s_misc[2], wb);
      }
    }
    __syncthreads();   // ce is free from here: it holds the band's candidate slots
    const uint32_t nband = s_misc[2], n_in = s_misc[3];
    ok = ok && n_in <= k && k - n_in <= nband && nband <= SC::BANDCAP;
    if (ok) {
      // (s_misc[2] keeps the band count every thread read above: the slots
      // come from a counter zeroed before that read's barrier)
      uint32_t *band = reinterpret_cast<uint32_t *>(ce);
      for (uint32_t j = threadIdx.x, u = 0; j < nc; j += blockDim.x, ++u)
        if ((cls >> (2 * u)) & 2u) band[atomicAdd(&s_misc[1], 1u)] = j;
      __syncthreads();
      // exact scores of the band
      rescore_band<SC::NW>(qsm, wsh, kbuf, relb, band, nband, cidx, cS, keys, a.map, b, s_rexact,
                           eq_min, eq_max);
      float *bV = scratch;
      uint32_t *bI = reinterpret_cast<uint32_t *>(scratch + SC::BANDCAP);
      for (uint32_t i = threadIdx.x; i < nband; i += blockDim.x) {
        bV[i] = cS[band[i]];
        bI[i] = cidx[band[i]];
      }
      __syncthreads();
      // the k - n_in best of the band by (exact score desc, row asc)
      const uint32_t want = k - n_in;
      for (uint32_t i = warp; i < nband; i += SC::NW) {   // one warp per band row
        const float V = bV[i];
        const uint32_t idx = bI[i];
        uint32_t rank = 0;
        for (uint32_t t = lane; t < nband; t += 32) {
          const float Vt = bV[t];
          rank += (Vt > V || (Vt == V && bI[t] < idx)) ? 1u : 0u;
        }
        rank = warp_sum_u32(rank);
        if (lane == 0 && rank < want) atomicOr(&bitmap[idx >> 5], 1u << (idx & 31));
      }
      __syncthreads();
      // ascending output from the bitmap
      const uint32_t per_t = (words + blockDim.x - 1) / blockDim.x;
      const uint32_t w0 = threadIdx.x * per_t, w1 = min(words, w0 + per_t);
      uint32_t cnt = 0;
      for (uint32_t i = w0; i < w1; ++i) cnt += __popc(bitmap[i]);
      uint32_t tot;
      uint32_t pos = block_excl_scan(cnt, wsum, &tot);
      for (uint32_t i = w0; i < w1; ++i) {
        uint32_t m = bitmap[i];
        while (m) {
          const uint32_t bit = __ffs(m) - 1;
          if (pos < k) out[pos] = (int32_t)(i * 32 + bit);
          ++pos;
          m &= m - 1;
        }
      }
      for (uint32_t j = tot + threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
      return;
    }
    // inconsistent counts (never expected): the in-place selection below
    // recomputes everything from the scores
    __syncthreads();
  }

  // ---- fallback: the same certified selection over every visible row
  const float tau = key_to_float(
      radix_kth([&](uint32_t s) { return score_key(sc[s]); }, vis, k, hist, sel, &need));
  const float hi_cut = tau + E + fabsf(tau) * kRel;
  const float lo_cut = tau - E - fabsf(tau) * kRel;
  uint32_t *band = cidx;
  if (threadIdx.x == 0) s_misc[2] = 0;
  __syncthreads();
  for (uint32_t s = threadIdx.x; s < vis; s += blockDim.x) {
    const float S = sc[s];
    const float e = err_of(S, nr[a.map.row_of(b, s)]);
    if (S - e > hi_cut) {
      sc[s] = INFINITY;
    } else if (S + e < lo_cut) {
      sc[s] = -INFINITY;
    } else {
      const uint32_t i = atomicAdd(&s_misc[2], 1u);
      if (i < CAP) band[i] = s;
    }
  }
  __syncthreads();
  const uint32_t nband = s_misc[2];
  if (nband <= CAP) {
    for (uint32_t i = warp; i < nband; i += SC::NW) {
      const uint32_t s = band[i];
      const float V = rescore_row(qsm, wsh, kb, rel, keys + a.map.row_of(b, s) * Di, lane, eq_min,
                                  eq_max);
      if (lane == 0) sc[s] = V;
    }
  } else {
    for (uint32_t s = warp; s < vis; s += SC::NW) {
      const float v = sc[s];
      if (v == INFINITY || v == -INFINITY) continue;
      const float V = rescore_row(qsm, wsh, kb, rel, keys + a.map.row_of(b, s) * Di, lane, eq_min,
                                  eq_max);
      if (lane == 0) sc[s] = V;
    }
  }
  __syncthreads();
  auto key = [&](uint32_t s) { return score_key(sc[s]); };
  const uint32_t kth = radix_kth(key, vis, k, hist, sel, &need);
  ordered_emit(key, vis, kth, need, k, out, wsum, [](uint32_t x) { return x; });
}

template <typename T>
cudaError_t launch_index_exact(const IndexArgs &a, cudaStream_t s) {
  const uint32_t nq = a.batch * a.T;
  IndexWs w = index_ws_split(a.ws, nq, a.n_heads, a.dim);
  index_qrot_kernel<T><<<nq, 256, 0, s>>>(a, w.qrot, w.err);
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
  // q' in units of 8 dims (one 16-byte load each when the query is 16-byte
  // aligned, else eight 2-byte loads)
  const bool vec = reinterpret_cast<uintptr_t>(a.q_idx) % 16 == 0;
  const uint32_t per = 8;
  if ((size_t)nq * a.n_heads * a.dim >= (1ull << 31)) return cudaErrorInvalidValue;
  // the scorer builds key histograms when several select blocks share a
  // query; with one block per query the selection samples its threshold
  const bool scorer_hist = select_groups(nq) > 1;
  size_t nthreads = (size_t)nq * a.n_heads * a.dim / per;
  if (scorer_hist && (size_t)nq * (kHistBins / 4) > nthreads) nthreads = (size_t)nq * (kHistBins / 4);
  if (nthreads == 0) nthreads = 1;
  cudaError_t eq = launch_pdl(index_qbf_kernel, dim3((unsigned)((nthreads + 255) / 256)),
                              dim3(256), 0, s, a, w, scorer_hist, vec);
  if (eq != cudaSuccess) return eq;
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
    t.score_stride = w.sstride;
    t.hist = scorer_hist ? w.hist : nullptr;
    t.err = w.err;
    t.map = a.map;
    t.seq_pos = a.seq_pos;
    cudaError_t e = launch_index_score_tc(t, s);
    if (e != cudaSuccess) return e;
  }
  // |S~ - S| <= cb * A_t * ||k_s||: the exact recipe (Di products, Hi weighted
  // terms) and the tensor-core accumulation (taken as at most 4 Di fp32
  // roundings) plus the fp32 epilogue; widened for the fp32 norms.
  const double cb = (gamma_n(a.dim + a.n_heads + 1) + gamma_n(4.0 * a.dim + a.n_heads + 1)) *
                    (1.0 + std::ldexp(1.0, -8));
  const uint32_t G = select_groups(nq);
  if (G == 1) {
    const size_t smem = SelCfg<256>::smem(a.comp_cap);
    static int smem_set = 0;
    cudaError_t e = ensure_smem(topk_select_tc_kernel<256>, smem, &smem_set);
    if (e != cudaSuccess) return e;
    // four blocks per SM: the largest shared-memory carveout
    static int carve = 0;
    if (!carve) {
      e = cudaFuncSetAttribute(topk_select_tc_kernel<256>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      carve = 1;
    }
    e = launch_pdl(topk_select_tc_kernel<256>, dim3(nq), dim3(256), smem, s, a, w, (float)cb, G);
    if (e != cudaSuccess) return e;
  } else {
    const size_t smem = SelCfg<1024>::smem(a.comp_cap);
    static int smem_set = 0;
    cudaError_t e = ensure_smem(topk_select_tc_kernel<1024>, smem, &smem_set);
    if (e != cudaSuccess) return e;
    // the G blocks of a query form a cluster (their candidates go to the
    // first block's shared memory)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = G;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(nq * G);
    cfg.blockDim = dim3(1024);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, topk_select_tc_kernel<1024>, a, w, (float)cb, G);
    if (e != cudaSuccess) return e;
  }
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
  return kExactWsHeader + (((qsz + 63) & ~(size_t)63) + nq * comp_cap) * sizeof(float);
}

cudaError_t launch_index_topk(const IndexArgs &a, cudaStream_t s) {
  if (a.dtype == DS4A_BF16) {
    if (index_tc_supported(a.n_heads, a.dim)) return launch_index_tc(a, s);
    return launch_index_exact<__nv_bfloat16>(a, s);
  }
  return launch_index_exact<float>(a, s);
}

}  // namespace ds4a
