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
// Three launches: rotate the queries into the workspace, score every visible
// row (one thread per row, 128 rows per block, keys staged in shared memory),
// then a per-query radix select (8-bit digits over an order-preserving key)
// followed by an ordered compaction.
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

__global__ void __launch_bounds__(kSelectThreads)
    topk_select_kernel(IndexArgs a, const float *scores) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wsum[33];
  __shared__ uint32_t sel_digit, sel_before;
  const uint32_t qi = blockIdx.x, t = qi % a.T, p = a.pos0 + t;
  const uint32_t vis = min((p + 1) / 4, a.n_comp), k = a.top_k;
  int32_t *out = a.topk + (size_t)qi * k;
  if (vis <= k) {
    for (uint32_t j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < vis ? (int32_t)j : -1;
    return;
  }
  const float *sc = scores + (size_t)qi * a.comp_cap;
  uint32_t prefix = 0, mask = 0, need = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (uint32_t i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (uint32_t s = threadIdx.x; s < vis; s += blockDim.x) {
      const uint32_t key = score_key(sc[s]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t cum = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (cum + hist[d] >= need) break;
        cum += hist[d];
      }
      sel_digit = (uint32_t)d;
      sel_before = cum;
    }
    __syncthreads();
    prefix |= sel_digit << shift;
    mask |= 255u << shift;
    need -= sel_before;
    __syncthreads();
  }
  // prefix = key of the k-th largest score; take every larger key and the
  // first `need` equal keys in index order.
  uint32_t eq_seen = 0, out_pos = 0;
  for (uint32_t base = 0; base < vis; base += blockDim.x) {
    const uint32_t s = base + threadIdx.x;
    const uint32_t key = s < vis ? score_key(sc[s]) : 0u;
    const bool gt = s < vis && key > prefix;
    const bool eq = s < vis && key == prefix;
    uint32_t eq_tot, sel_tot;
    const uint32_t eq_rank = eq_seen + block_flag_scan(eq, wsum, &eq_tot);
    const bool sel = gt || (eq && eq_rank < need);
    const uint32_t pos = out_pos + block_flag_scan(sel, wsum, &sel_tot);
    if (sel && pos < k) out[pos] = (int32_t)s;
    eq_seen += eq_tot;
    out_pos += sel_tot;
  }
}

template <typename T>
cudaError_t launch_index_t(const IndexArgs &a, cudaStream_t s) {
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

}  // namespace

size_t index_ws_bytes(uint32_t batch, uint32_t T, uint32_t n_heads, uint32_t dim,
                      uint32_t comp_cap) {
  const size_t nq = (size_t)batch * T;
  const size_t qsz = nq * dim * round_up8(n_heads);
  return (((qsz + 63) & ~(size_t)63) + nq * comp_cap) * sizeof(float);
}

cudaError_t launch_index_topk(const IndexArgs &a, cudaStream_t s) {
  return a.dtype == DS4A_BF16 ? launch_index_t<__nv_bfloat16>(a, s) : launch_index_t<float>(a, s);
}

}  // namespace ds4a
