// Sparse attention over the raw window plus compressed rows, K = V
// ("【#3】ds4.c を読み解く" §7 mixed attention; vLLM DeepSeek V4 page: shared
// K = V with inverse RoPE on the output, c4a / c128a, 128-token window).
//
// For the query at position p the attended rows are, in this order,
//   window:     positions max(0, p - cap_raw + 1) .. p  (ring slot p % cap_raw,
//               or the chunk's own rows for positions >= pos0 in a prefill)
//   compressed: ratio 4: the top-k list (entries < 0 skipped, the list ends at
//               the first entry >= floor((p+1)/4)); ratio 128: rows
//               0 .. floor((p+1)/128) - 1; ratio 0: none
// under one softmax with the given scale; the output tail is rotated by -p.
//
// Flash-decode structure: a block owns one query, a group of heads and a
// contiguous range (split) of the row list; it streams the rows through
// shared memory in tiles, keeps an online softmax per head and accumulates
// P V with the same tile (K = V, loaded once). Decode splits the row list so
// that enough blocks run; partial (m, l, o) are merged by a second kernel that
// also applies the inverse rotation. Prefill has one split per query and
// finishes in place.
#include "common.cuh"

namespace ds4a {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxOut = 16;  // outputs (head, dim) per thread: HG * D <= 4096

struct Plan {
  uint32_t tile, split_rows, n_splits, hg, n_hg, rows_max;
};

__host__ __device__ inline uint32_t rows_max(uint32_t ratio, uint32_t cap_raw,
                                             uint32_t comp_cap, uint32_t top_k) {
  return cap_raw + (ratio == 4 ? top_k : ratio == 128 ? comp_cap : 0);
}

// Rows of any query of a call whose last position is at most pos_end - 1
// (the window, then the listed or visible compressed rows): at most
// rows_max, and tighter once the position is known.
inline uint32_t rows_at(uint32_t ratio, uint32_t cap_raw, uint32_t comp_cap, uint32_t top_k,
                        uint32_t n_comp, uint64_t pos_end) {
  const uint32_t w = (uint32_t)(pos_end < cap_raw ? pos_end : cap_raw);
  uint64_t c = 0;
  if (ratio == 4) c = pos_end / 4 < top_k ? pos_end / 4 : top_k;
  else if (ratio == 128) c = pos_end / 128;
  if (ratio && c > n_comp) c = n_comp;
  const uint64_t r = (uint64_t)w + c;
  const uint32_t bound = rows_max(ratio, cap_raw, comp_cap, top_k);
  return r < bound ? (uint32_t)r : bound;
}

inline Plan make_plan(uint32_t ratio, uint32_t batch, uint32_t T, uint32_t H, uint32_t D,
                      uint32_t cap_raw, uint32_t comp_cap, uint32_t top_k) {
  Plan pl;
  pl.tile = 16384 / D;
  if (pl.tile > 128) pl.tile = 128;
  if (pl.tile < 8) pl.tile = 8;
  pl.hg = 4096 / D;
  if (pl.hg > H) pl.hg = H;
  if (pl.hg > 8) pl.hg = 8;
  while (H % pl.hg) --pl.hg;
  pl.n_hg = H / pl.hg;
  pl.rows_max = rows_max(ratio, cap_raw, comp_cap, top_k);
  const uint64_t nq = (uint64_t)batch * T;
  if (nq >= 256) {
    pl.split_rows = pl.rows_max;
    pl.n_splits = 1;
  } else {
    pl.split_rows = 2 * pl.tile;
    pl.n_splits = (pl.rows_max + pl.split_rows - 1) / pl.split_rows;
  }
  return pl;
}

inline size_t smem_bytes(const Plan &pl, uint32_t D) {
  return ((size_t)pl.hg * D + (size_t)pl.tile * (D + 4) + (size_t)pl.hg * pl.tile +
          4 * pl.hg) * sizeof(float) + (size_t)pl.tile * sizeof(long long) + 16;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    attn_kernel(AttnArgs a, Plan pl, float *part) {
  extern __shared__ float4 smem4[];
  const uint32_t D = a.head_dim, H = a.n_heads, HG = pl.hg, S = pl.tile, ks_stride = D + 4;
  float *qs = reinterpret_cast<float *>(smem4);        // [HG][D]
  float *ks = qs + (size_t)HG * D;                     // [S][D+4]
  float *ps = ks + (size_t)S * ks_stride;              // [HG][S]
  float *mrow = ps + (size_t)HG * S;                   // [HG] running max
  float *lrow = mrow + HG;                             // [HG] running sum
  float *alpha = lrow + HG;                            // [HG] rescale of this tile
  long long *roff = reinterpret_cast<long long *>(alpha + 2 * HG);  // [S] row offsets (-1 masked)
  __shared__ uint32_t s_nlist;

  const uint32_t qi = blockIdx.z, b = qi / a.T, t = qi % a.T;
  const uint32_t p = seq_base(a.seq_pos, a.pos0, b) + t;
  const uint32_t h0 = blockIdx.y * HG, split = blockIdx.x;
  const uint32_t n_w = min(p + 1, a.cap_raw);
  const int32_t *tk = a.topk ? a.topk + (size_t)qi * a.top_k : nullptr;

  // length of the compressed part of the list
  if (threadIdx.x == 0) s_nlist = 0xffffffffu;
  __syncthreads();
  uint32_t n_list = 0;
  if (a.ratio == 4) {
    const uint32_t vis = min((p + 1) / 4, a.n_comp);
    for (uint32_t j = threadIdx.x; j < a.top_k; j += blockDim.x)
      if (tk[j] >= 0 && (uint32_t)tk[j] >= vis) atomicMin(&s_nlist, j);
    __syncthreads();
    n_list = min(s_nlist, a.top_k);
  } else if (a.ratio == 128) {
    n_list = min((p + 1) / 128, a.n_comp);
  }
  const uint32_t N = n_w + n_list;
  const uint32_t r_begin = split * pl.split_rows;
  const uint32_t r_end = min(N, r_begin + pl.split_rows);

  // rotated queries of this head group
  const T *q = static_cast<const T *>(a.q) + ((size_t)qi * H + h0) * D;
  const uint32_t n_nope = D - a.n_rot;
  for (uint32_t pr = threadIdx.x; pr < HG * D / 2; pr += blockDim.x) {
    const uint32_t h = pr / (D / 2), c = 2 * (pr % (D / 2));
    float x0 = ld_f32(q, (size_t)h * D + c), x1 = ld_f32(q, (size_t)h * D + c + 1);
    if (c >= n_nope) {
      const uint32_t fi = (c - n_nope) / 2;
      const float co = a.cos[(size_t)p * (a.n_rot / 2) + fi];
      const float si = a.sin[(size_t)p * (a.n_rot / 2) + fi];
      const float r0 = x0 * co - x1 * si, r1 = x0 * si + x1 * co;
      x0 = r0;
      x1 = r1;
    }
    qs[(size_t)h * D + c] = x0;
    qs[(size_t)h * D + c + 1] = x1;
  }
  if (threadIdx.x < HG) {
    mrow[threadIdx.x] = -INFINITY;
    lrow[threadIdx.x] = 0.f;
  }
  float acc[kMaxOut];
#pragma unroll
  for (int j = 0; j < kMaxOut; ++j) acc[j] = 0.f;
  const uint32_t n_out = (HG * D + blockDim.x - 1) / blockDim.x;

  const T *ring = static_cast<const T *>(a.ring) + (size_t)b * a.cap_raw * D;
  const T *chunk = a.chunk ? static_cast<const T *>(a.chunk) + (size_t)b * a.T * D : nullptr;
  const T *comp = static_cast<const T *>(a.comp);   // pool base: rows via a.map
  const uint32_t lane = threadIdx.x & 31, wid = threadIdx.x >> 5;

  for (uint32_t r0 = r_begin; r0 < r_end; r0 += S) {
    const uint32_t nr = min(S, r_end - r0);
    __syncthreads();  // previous tile fully consumed
    // row offsets (elements from the per-sequence base; chunk rows are tagged)
    for (uint32_t r = threadIdx.x; r < S; r += blockDim.x) {
      long long off = -1;
      const uint32_t g = r0 + r;
      if (r < nr) {
        if (g < n_w) {
          const uint32_t pos = p - n_w + 1 + g;
          if (chunk && pos >= p - t)   // (p - t: this sequence's first chunk position)
            off = (1ll << 62) | (long long)(pos - (p - t)) * D;
          else
            off = (long long)(pos % a.cap_raw) * D;
        } else {
          const uint32_t j = g - n_w;
          const int32_t idx = a.ratio == 4 ? tk[j] : (int32_t)j;
          if (idx >= 0) off = (1ll << 61) | (long long)(a.map.row_of(b, (uint32_t)idx) * D);
        }
      }
      roff[r] = off;
    }
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < S * D; i += blockDim.x) {
      const uint32_t r = i / D, d = i % D;
      const long long off = roff[r];
      float v = 0.f;
      if (off >= 0) {
        if (off & (1ll << 62))
          v = ld_f32(chunk, (size_t)(off & ((1ll << 61) - 1)) + d);
        else if (off & (1ll << 61))
          v = ld_f32(comp, (size_t)(off & ((1ll << 61) - 1)) + d);
        else
          v = ld_f32(ring, (size_t)off + d);
      }
      ks[(size_t)r * ks_stride + d] = v;
    }
    __syncthreads();
    // scores
    for (uint32_t pr = threadIdx.x; pr < HG * S; pr += blockDim.x) {
      const uint32_t h = pr / S, r = pr % S;
      float s = -INFINITY;
      if (roff[r] >= 0) {
        const float4 *qv = reinterpret_cast<const float4 *>(qs + (size_t)h * D);
        const float4 *kv = reinterpret_cast<const float4 *>(ks + (size_t)r * ks_stride);
        float dot = 0.f;
        for (uint32_t d4 = 0; d4 < D / 4; ++d4) {
          const float4 x = qv[d4], y = kv[d4];
          dot += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
        }
        s = dot * a.scale;
      }
      ps[(size_t)h * S + r] = s;
    }
    __syncthreads();
    // online softmax, one warp per head
    for (uint32_t h = wid; h < HG; h += blockDim.x / 32) {
      float mx = -INFINITY;
      for (uint32_t r = lane; r < S; r += 32) mx = fmaxf(mx, ps[(size_t)h * S + r]);
      mx = warp_max(mx);
      const float m_old = mrow[h];
      const float m_new = fmaxf(m_old, mx);
      float sum = 0.f;
      for (uint32_t r = lane; r < S; r += 32) {
        const float s = ps[(size_t)h * S + r];
        const float e = (m_new == -INFINITY || s == -INFINITY) ? 0.f : expf(s - m_new);
        ps[(size_t)h * S + r] = e;
        sum += e;
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        const float al = (m_old == -INFINITY) ? (m_new == -INFINITY ? 1.f : 0.f)
                                              : expf(m_old - m_new);
        alpha[h] = al;
        lrow[h] = lrow[h] * al + sum;
        mrow[h] = m_new;
      }
    }
    __syncthreads();
    // o = o * alpha + P V
#pragma unroll
    for (int j = 0; j < kMaxOut; ++j) {
      if ((uint32_t)j >= n_out) break;
      const uint32_t idx = threadIdx.x + j * blockDim.x;
      if (idx >= HG * D) break;
      const uint32_t h = idx / D, d = idx % D;
      float o = acc[j] * alpha[h];
      const float *pr = ps + (size_t)h * S;
      for (uint32_t r = 0; r < nr; ++r) o += pr[r] * ks[(size_t)r * ks_stride + d];
      acc[j] = o;
    }
  }
  __syncthreads();

  if (pl.n_splits == 1) {
    T *out = static_cast<T *>(a.out) + ((size_t)qi * H + h0) * D;
#pragma unroll
    for (int j = 0; j < kMaxOut; ++j) {
      if ((uint32_t)j >= n_out) break;
      const uint32_t idx = threadIdx.x + j * blockDim.x;
      const bool live = idx < HG * D;
      const uint32_t h = live ? idx / D : 0, d = live ? idx % D : 0;
      float o = live ? acc[j] / lrow[h] : 0.f;
      const float other = __shfl_xor_sync(0xffffffffu, o, 1);
      if (live && d >= n_nope) {
        const uint32_t fi = (d - n_nope) / 2;
        const float co = a.cos[(size_t)p * (a.n_rot / 2) + fi];
        const float si = a.sin[(size_t)p * (a.n_rot / 2) + fi];
        // rotate by -p: (x0, x1) -> (x0 c + x1 s, -x0 s + x1 c)
        o = (d & 1) ? (-other * si + o * co) : (o * co + other * si);
      }
      if (live) st_elem(out, (size_t)h * D + d, o);
    }
    return;
  }
  // partials: o [qi][split][H][D], then (m, l) [qi][split][H][2]
  const size_t nq = (size_t)a.batch * a.T;
  float *po = part + ((size_t)qi * pl.n_splits + split) * H * D;
  float *pml = part + nq * pl.n_splits * H * D + ((size_t)qi * pl.n_splits + split) * H * 2;
#pragma unroll
  for (int j = 0; j < kMaxOut; ++j) {
    if ((uint32_t)j >= n_out) break;
    const uint32_t idx = threadIdx.x + j * blockDim.x;
    if (idx >= HG * D) break;
    po[(size_t)(h0 + idx / D) * D + idx % D] = acc[j];
  }
  if (threadIdx.x < HG) {
    pml[(h0 + threadIdx.x) * 2] = mrow[threadIdx.x];
    pml[(h0 + threadIdx.x) * 2 + 1] = lrow[threadIdx.x];
  }
}

template <typename T>
__global__ void attn_merge_kernel(AttnArgs a, Plan pl, const float *part) {
  const uint32_t h = blockIdx.x, qi = blockIdx.y, t = qi % a.T;
  const uint32_t p = seq_base(a.seq_pos, a.pos0, qi / a.T) + t;
  const uint32_t D = a.head_dim, H = a.n_heads, ns = pl.n_splits, n_nope = D - a.n_rot;
  const size_t nq = (size_t)a.batch * a.T;
  const float *pml = part + nq * ns * H * D + (size_t)qi * ns * H * 2;
  float M = -INFINITY;
  for (uint32_t s = 0; s < ns; ++s) M = fmaxf(M, pml[((size_t)s * H + h) * 2]);
  float L = 0.f;
  for (uint32_t s = 0; s < ns; ++s) {
    const float m = pml[((size_t)s * H + h) * 2];
    if (m != -INFINITY) L += pml[((size_t)s * H + h) * 2 + 1] * expf(m - M);
  }
  T *out = static_cast<T *>(a.out) + ((size_t)qi * H + h) * D;
  for (uint32_t j = threadIdx.x; j < D / 2; j += blockDim.x) {
    const uint32_t c = 2 * j;
    float o0 = 0.f, o1 = 0.f;
    for (uint32_t s = 0; s < ns; ++s) {
      const float m = pml[((size_t)s * H + h) * 2];
      if (m == -INFINITY) continue;
      const float f = expf(m - M);
      const float *po = part + (((size_t)qi * ns + s) * H + h) * D;
      o0 += f * po[c];
      o1 += f * po[c + 1];
    }
    o0 /= L;
    o1 /= L;
    if (c >= n_nope) {
      const uint32_t fi = (c - n_nope) / 2;
      const float co = a.cos[(size_t)p * (a.n_rot / 2) + fi];
      const float si = a.sin[(size_t)p * (a.n_rot / 2) + fi];
      const float r0 = o0 * co + o1 * si, r1 = -o0 * si + o1 * co;
      o0 = r0;
      o1 = r1;
    }
    st_elem(out, c, o0);
    st_elem(out, c + 1, o1);
  }
}

template <typename T>
__global__ void ring_commit_kernel(const T *chunk, T *ring, uint32_t T_len, uint32_t pos0,
                                   const uint32_t *seq_pos, uint32_t cap, uint32_t D, uint32_t n) {
  const uint32_t t = T_len - n + blockIdx.x, b = blockIdx.y;
  const uint32_t p = seq_base(seq_pos, pos0, b) + t;
  const T *src = chunk + ((size_t)b * T_len + t) * D;
  T *dst = ring + ((size_t)b * cap + p % cap) * D;
  for (uint32_t d = threadIdx.x; d < D; d += blockDim.x) dst[d] = src[d];
}

template <typename T>
cudaError_t launch_attention_t(const AttnArgs &a, cudaStream_t s) {
  const Plan pl = make_plan(a.ratio, a.batch, a.T, a.n_heads, a.head_dim, a.cap_raw,
                            a.comp_cap, a.top_k);
  const size_t smem = smem_bytes(pl, a.head_dim);
  static int smem_set = 0;
  cudaError_t e = ensure_smem(attn_kernel<T>, smem, &smem_set);
  if (e != cudaSuccess) return e;
  // (the first 256 bytes: the error word of the workspace; this path has no
  // device waits and leaves it alone)
  float *part = a.ws ? reinterpret_cast<float *>(static_cast<uint8_t *>(a.ws) + 256) : nullptr;
  dim3 grid(pl.n_splits, pl.n_hg, a.batch * a.T);
  attn_kernel<T><<<grid, kThreads, smem, s>>>(a, pl, part);
  note_launches(1);
  if (pl.n_splits > 1) {
    attn_merge_kernel<T><<<dim3(a.n_heads, a.batch * a.T), 128, 0, s>>>(a, pl, part);
    note_launches(1);
  }
  return cudaGetLastError();
}

// bf16 Flash shape: tcgen05 kernel (decode merges its splits inside a
// thread-block cluster); word 0 of the workspace is its error word (never
// reset: a launch compares it with its value at the start).
cudaError_t launch_attention_tc_path(const AttnArgs &a, cudaStream_t s) {
  // decode: the row bound at the call's position (the workspace is sized
  // for the shape's bound, which is never smaller)
  const uint32_t rmax = a.T == 1 ? rows_at(a.ratio, a.cap_raw, a.comp_cap, a.top_k, a.n_comp,
                                           (uint64_t)a.pos0 + 1)
                                 : rows_max(a.ratio, a.cap_raw, a.comp_cap, a.top_k);
  return launch_attention_tc(a, rmax, static_cast<int *>(a.ws), s);
}

}  // namespace

size_t attn_ws_bytes(int dtype, uint32_t ratio, uint32_t batch, uint32_t T, uint32_t n_heads,
                     uint32_t head_dim, uint32_t n_rot, uint32_t cap_raw, uint32_t comp_cap,
                     uint32_t top_k) {
  if (attn_tc_supported(dtype, n_heads, head_dim, n_rot))
    return attn_tc_ws_bytes(batch, T, rows_max(ratio, cap_raw, comp_cap, top_k));
  const Plan pl = make_plan(ratio, batch, T, n_heads, head_dim, cap_raw, comp_cap, top_k);
  if (pl.n_splits == 1) return 0;
  return 256 + (size_t)batch * T * pl.n_splits * n_heads * (head_dim + 2) * sizeof(float);
}

uint32_t attn_decode_cluster(int dtype, uint32_t ratio, uint32_t batch, uint32_t n_heads,
                             uint32_t head_dim, uint32_t n_rot, uint32_t cap_raw,
                             uint32_t comp_cap, uint32_t top_k, uint32_t n_comp,
                             uint64_t pos_end) {
  if (!attn_tc_supported(dtype, n_heads, head_dim, n_rot)) return 0;
  return attn_tc_decode_cluster(rows_at(ratio, cap_raw, comp_cap, top_k, n_comp, pos_end), batch);
}

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s) {
  if (attn_tc_supported(a.dtype, a.n_heads, a.head_dim, a.n_rot))
    return launch_attention_tc_path(a, s);
  return a.dtype == DS4A_BF16 ? launch_attention_t<__nv_bfloat16>(a, s)
                              : launch_attention_t<float>(a, s);
}

cudaError_t launch_ring_commit(int dtype, uint32_t batch, uint32_t T, uint32_t pos0,
                               const uint32_t *seq_pos, uint32_t cap_raw, uint32_t head_dim,
                               const void *chunk, void *ring, cudaStream_t s) {
  const uint32_t n = T < cap_raw ? T : cap_raw;
  if (!n) return cudaSuccess;
  note_launches(1);
  if (dtype == DS4A_BF16)
    ring_commit_kernel<__nv_bfloat16><<<dim3(n, batch), 128, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(chunk), static_cast<__nv_bfloat16 *>(ring), T, pos0,
        seq_pos, cap_raw, head_dim, n);
  else
    ring_commit_kernel<float><<<dim3(n, batch), 128, 0, s>>>(
        static_cast<const float *>(chunk), static_cast<float *>(ring), T, pos0, seq_pos,
        cap_raw, head_dim, n);
  return cudaGetLastError();
}

}  // namespace ds4a
