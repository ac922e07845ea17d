// Raw-window insert and KV compressor ("【#3】ds4.c を読み解く" §4 compressor
// steps, §5 ratio-4 frontier, §8 tail RoPE; vLLM DeepSeek V4 page: c4a pools
// 8 tokens at stride 4, c128a 128 tokens at stride 128).
//
// One fused, elementwise pass per call. A thread owns one (or two) adjacent
// channel pairs of a row, so the rotation pair, the per-channel pooling over
// the window slots and the state writes of a channel all stay in one thread;
// only the RMS of the pooled row needs a block reduction.
//
// Decode (T = 1): one launch, grid (B, 1 + lanes). Block y = 0 rotates the raw
// row into the ring (absent when the raw rows are not part of the call, y0 = 1);
// block y = 1 + l stores the token into lane l's state and,
// at a ratio boundary, pools, normalises, rotates and appends the compressed
// row, then (ratio 4) moves slots 4..7 to 0..3.
// Chunk (T > 1): every compressed row completed inside the chunk is built in
// parallel, one block per row, reading window tokens from the chunk inputs or,
// for tokens before pos0, from the state as it was before the chunk; a second
// launch then writes the state as the token-by-token process would leave it.
#include "quant.cuh"
#include "tc.cuh"

namespace ds4a {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxQatWidth = 256;      // indexer rows with the FP4 round trip
constexpr float kRmsEps = 1e-6f;
constexpr int kMaxPairsPerThread = 2;  // width <= 1024

struct SlotVal {
  float kv, score;
};

// Pool window slots per channel, RMS-normalise, rotate at `pos`, apply the
// lane's step-8 round trip (if any) and store row i of the lane. get(s, c)
// returns slot s of channel c (score without APE, -inf when empty). Called by
// every thread of the block (uniform).
template <typename T, typename Get>
__device__ void pool_norm_rope_store(const LaneArgs &L, uint32_t W, uint32_t b, uint32_t i,
                                     uint32_t pos, Get get, float *red) {
  const T *ape = static_cast<const T *>(L.ape);
  const T *gamma = static_cast<const T *>(L.gamma);
  T *comp = static_cast<T *>(L.comp);
  const uint32_t width = L.width, npair = width / 2, n_nope = width - L.n_rot;
  float y[kMaxPairsPerThread][2];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerThread; ++k) {
    const uint32_t j = threadIdx.x + k * blockDim.x;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float out = 0.f;
      if (j < npair) {
        const uint32_t c = 2 * j + e;
        float m = -INFINITY;
        for (uint32_t s = 0; s < W; ++s) {
          const float sig = get(s, c).score + ld_f32(ape, (size_t)s * width + c);
          m = fmaxf(m, sig);
        }
        if (m != -INFINITY) {
          float den = 0.f, num = 0.f;
          for (uint32_t s = 0; s < W; ++s) {
            const SlotVal v = get(s, c);
            const float w = expf(v.score + ld_f32(ape, (size_t)s * width + c) - m);
            if (w > 0.f) {
              den += w;
              num += w * v.kv;
            }
          }
          out = den > 0.f ? num / den : 0.f;
        }
      }
      y[k][e] = out;
      ss += out * out;
    }
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)width + kRmsEps);
  size_t prow;
  const bool mapped = L.map.phys(b, i, prow);   // uniform; unmapped: computed, not stored
  T *row = comp + prow * width;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerThread; ++k) {
    const uint32_t j = threadIdx.x + k * blockDim.x;
    if (j >= npair) continue;
    const uint32_t c = 2 * j;
    float a = ld_f32(gamma, c) * (y[k][0] * inv);
    float bb = ld_f32(gamma, c + 1) * (y[k][1] * inv);
    if (c >= n_nope) {
      const uint32_t fi = (c - n_nope) / 2;
      const float co = L.cos[(size_t)pos * (L.n_rot / 2) + fi];
      const float si = L.sin[(size_t)pos * (L.n_rot / 2) + fi];
      const float ra = a * co - bb * si;
      const float rb = a * si + bb * co;
      a = ra;
      bb = rb;
    }
    y[k][0] = a;
    y[k][1] = bb;
  }
  // step 8 (uniform branch): FP8 on the non-RoPE dims, one warp per 64-dim
  // block (thread j holds dims 2j, 2j + 1), or the FP4 QAT round trip of the
  // whole row through shared memory
  if (L.quant == 1) {
#pragma unroll
    for (int k = 0; k < kMaxPairsPerThread; ++k) {
      const uint32_t j = threadIdx.x + k * blockDim.x, c = 2 * j;
      const bool in = j < npair && c < n_nope;
      const float am = warp_max(in ? fmaxf(fabsf(y[k][0]), fabsf(y[k][1])) : 0.f);
      const int ke = block_scale_exp(am, kE4M3);
      if (in) {
        y[k][0] = quant_dequant(y[k][0], ke, kE4M3);
        y[k][1] = quant_dequant(y[k][1], ke, kE4M3);
      }
    }
  } else if (L.quant == 2) {
    __shared__ float qbuf[kMaxQatWidth];
#pragma unroll
    for (int k = 0; k < kMaxPairsPerThread; ++k) {
      const uint32_t j = threadIdx.x + k * blockDim.x;
      if (j < npair) {
        qbuf[2 * j] = y[k][0];
        qbuf[2 * j + 1] = y[k][1];
      }
    }
    __syncthreads();
    fp4_qat_smem(qbuf, width, L.had_c);
#pragma unroll
    for (int k = 0; k < kMaxPairsPerThread; ++k) {
      const uint32_t j = threadIdx.x + k * blockDim.x;
      if (j < npair) {
        y[k][0] = qbuf[2 * j];
        y[k][1] = qbuf[2 * j + 1];
      }
    }
  }
  float st[kMaxPairsPerThread][2];   // the stored (rounded) values, for the row norm
  float mx = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxPairsPerThread; ++k) {
    const uint32_t j = threadIdx.x + k * blockDim.x;
    if (j >= npair) continue;
    const uint32_t c = 2 * j;
    if (mapped) {
      st_elem(row, c, y[k][0]);
      st_elem(row, c + 1, y[k][1]);
    }
    st[k][0] = round_to(y[k][0], row);
    st[k][1] = round_to(y[k][1], row);
    mx = fmaxf(mx, fmaxf(fabsf(st[k][0]), fabsf(st[k][1])));
  }
  if (L.norm) {   // uniform: the indexer lane records the row's norm
    mx = block_max(mx, red);
    int e = 0;
    if (mx > 0.f) frexpf(mx, &e);
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxPairsPerThread; ++k) {
      const uint32_t j = threadIdx.x + k * blockDim.x;
      if (j < npair) {
        const float y0 = ldexpf(st[k][0], -e), y1 = ldexpf(st[k][1], -e);
        ss = fmaf(y0, y0, fmaf(y1, y1, ss));
      }
    }
    ss = block_sum(ss, red);
    if (threadIdx.x == 0 && mapped) {
      const float nm = mx > 0.f ? norm_from_scaled(ss, e) : 0.f;
      L.norm[prow] = nm;
      atomicMax(&L.norm_max[b], __float_as_uint(nm));
    }
  }
}

// Euclidean norm of stored indexer rows (rebuild after the caller wrote rows):
// one warp per row, the same widening as at append time.
template <typename T>
__global__ void index_norms_kernel(const T *rows, RowMap map, uint32_t dim, uint32_t n_rows,
                                   float *norm, uint32_t *norm_max) {
  const uint32_t b = blockIdx.y, lane = threadIdx.x & 31;
  const uint32_t r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= n_rows) return;
  size_t prow;
  if (!map.phys(b, r, prow)) return;   // warp-uniform
  const T *row = rows + prow * dim;
  float mx = 0.f;
  for (uint32_t c = lane; c < dim; c += 32) mx = fmaxf(mx, fabsf(ld_f32(row, c)));
  mx = warp_max(mx);
  int e = 0;
  if (mx > 0.f) frexpf(mx, &e);
  float ss = 0.f;
  for (uint32_t c = lane; c < dim; c += 32) {
    const float y = ldexpf(ld_f32(row, c), -e);
    ss = fmaf(y, y, ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) {
    const float nm = mx > 0.f ? norm_from_scaled(ss, e) : 0.f;
    norm[prow] = nm;
    atomicMax(&norm_max[b], __float_as_uint(nm));
  }
}

// Rotate one raw row (tail pairs) from src into dst.
template <typename T>
__device__ void raw_row(const T *src, T *dst, uint32_t D, uint32_t n_rot, uint32_t pos,
                        const float *cos, const float *sin) {
  const uint32_t n_nope = D - n_rot;
  for (uint32_t j = threadIdx.x; j < D / 2; j += blockDim.x) {
    const uint32_t c = 2 * j;
    float a = ld_f32(src, c), bb = ld_f32(src, c + 1);
    if (c >= n_nope) {
      const uint32_t fi = (c - n_nope) / 2;
      const float co = cos[(size_t)pos * (n_rot / 2) + fi];
      const float si = sin[(size_t)pos * (n_rot / 2) + fi];
      const float ra = a * co - bb * si;
      const float rb = a * si + bb * co;
      a = ra;
      bb = rb;
    }
    st_elem(dst, c, a);
    st_elem(dst, c + 1, bb);
  }
}

// One lane's decode step in one block: store the token into its window slot
// and, at a ratio boundary, pool, normalise, rotate and append the row, then
// (ratio 4) move slots 4..7 to 0..3.
template <typename T>
__device__ void lane_step_block(const AppendArgs &a, const LaneArgs &L, uint32_t b, uint32_t p,
                                float *red) {
  const uint32_t r = a.ratio, W = a.window, width = L.width;
  const uint32_t slot = r == 4 ? 4 + p % 4 : p % r;
  const T *cand = static_cast<const T *>(L.cand) + (size_t)b * width;
  const T *score = static_cast<const T *>(L.score) + (size_t)b * width;
  float *skv = L.state_kv + (size_t)b * W * width;
  float *ssc = L.state_score + (size_t)b * W * width;
  for (uint32_t c = threadIdx.x; c < width; c += blockDim.x) {
    skv[(size_t)slot * width + c] = ld_f32(cand, c);
    ssc[(size_t)slot * width + c] = ld_f32(score, c);
  }
  if ((p + 1) % r != 0) return;  // uniform over the block
  const uint32_t i = (p + 1) / r - 1;
  auto get = [&](uint32_t s, uint32_t c) {
    return SlotVal{skv[(size_t)s * width + c], ssc[(size_t)s * width + c]};
  };
  // The store above gives thread t channel t; the pool gives it channels 2t
  // and 2t + 1, written by other threads: make the stores visible first.
  __syncthreads();
  pool_norm_rope_store<T>(L, W, b, i, i * r, get, red);
  if (r == 4) {
    __syncthreads();  // every pool read of slots 0..3 is done
    for (uint32_t c = threadIdx.x; c < width; c += blockDim.x) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        skv[(size_t)s * width + c] = skv[(size_t)(4 + s) * width + c];
        ssc[(size_t)s * width + c] = ssc[(size_t)(4 + s) * width + c];
      }
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) append_step_kernel(AppendArgs a) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const uint32_t b = blockIdx.x, p = seq_base(a.seq_pos, a.pos0, b), role = blockIdx.y + a.y0;
  if (role == 0) {
    const T *src = static_cast<const T *>(a.raw_in) + (size_t)b * a.head_dim;
    T *dst = static_cast<T *>(a.raw_dst) +
             ((size_t)b * a.cap_raw + p % a.cap_raw) * a.head_dim;
    raw_row(src, dst, a.head_dim, a.n_rot, p, a.cos, a.sin);
    return;
  }
  lane_step_block<T>(a, a.lane[role - 1], b, p, red);
}

// Decode step on clusters of kSplit CTAs, for compressed layers whose
// attention rows are 512 or 1024 wide: every (sequence, role) is one cluster.
// The raw row and the attention lane are split by channel: CTA c owns channels
// [c w / kSplit, (c + 1) w / kSplit) (64 of a 512-wide row: one FP8 block).
// The attention lane stores the token's candidate and score and, at a window
// boundary, pools its channels over the W slots (spread over the CTA's eight
// warps, W / 8 slots per thread with every load in flight at once; then the
// per-channel maxima, then the weighted sums combined in warp order), adds the
// squares of its pooled channels, and takes the row's RMS from the cluster's
// partial sums (read in rank order from each CTA's shared memory, so every
// CTA gets the same value) before it normalises, rotates, rounds and stores
// its channels; ratio 4 then moves its channels of slots 4..7 to 0..3. One CTA
// per sequence would read the whole window state alone (512 KiB on ratio 128).
// The indexer lane (ratio 4, a 128-wide row with its norm and the optional
// FP4 round trip over the whole row) runs in the cluster's first CTA.
constexpr uint32_t kSplit = 8;
constexpr uint32_t kSlotGroups = kThreads / 32;   // 8 warps x 32 channel pairs

template <typename T, uint32_t W>
__global__ void __launch_bounds__(kThreads) append_step_split_kernel(AppendArgs a) {
  constexpr uint32_t SPT = W / kSlotGroups;   // slots per thread
  __shared__ float sm_max[kSlotGroups][64], sm_den[kSlotGroups][64], sm_num[kSlotGroups][64];
  __shared__ float part;
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const uint32_t rank = blockIdx.x % kSplit, cl = blockIdx.x / kSplit;
  const uint32_t b = cl % a.batch, role = cl / a.batch + a.y0;
  const uint32_t p = seq_base(a.seq_pos, a.pos0, b);
  const uint32_t t = threadIdx.x, pr = t & 31, g = t >> 5;
  if (role == 0) {   // the raw row: this CTA's channels
    const uint32_t D = a.head_dim, n_nope = D - a.n_rot, c = rank * (D / kSplit) + 2 * t;
    if (2 * t < D / kSplit) {
      const T *src = static_cast<const T *>(a.raw_in) + (size_t)b * D;
      T *dst = static_cast<T *>(a.raw_dst) + ((size_t)b * a.cap_raw + p % a.cap_raw) * D;
      float x0 = ld_f32(src, c), x1 = ld_f32(src, c + 1);
      if (c >= n_nope) {
        const uint32_t fi = (c - n_nope) / 2;
        const float co = a.cos[(size_t)p * (a.n_rot / 2) + fi];
        const float si = a.sin[(size_t)p * (a.n_rot / 2) + fi];
        const float r0 = x0 * co - x1 * si, r1 = x0 * si + x1 * co;
        x0 = r0;
        x1 = r1;
      }
      st_elem(dst, c, x0);
      st_elem(dst, c + 1, x1);
    }
    return;
  }
  const LaneArgs &L = a.lane[role - 1];
  if (L.norm) {   // the indexer lane: whole rows in the first CTA
    if (rank == 0) lane_step_block<T>(a, L, b, p, red);
    return;
  }
  const uint32_t r = a.ratio, width = L.width, cpc = width / kSplit;   // channels per CTA
  const uint32_t slot = r == 4 ? 4 + p % 4 : p % r;
  float *skv = L.state_kv + (size_t)b * W * width;
  float *ssc = L.state_score + (size_t)b * W * width;
  const T *cand = static_cast<const T *>(L.cand) + (size_t)b * width;
  const T *score = static_cast<const T *>(L.score) + (size_t)b * width;
  const uint32_t cbase = rank * cpc;
  for (uint32_t c = cbase + t; c < cbase + cpc; c += kThreads) {
    skv[(size_t)slot * width + c] = ld_f32(cand, c);
    ssc[(size_t)slot * width + c] = ld_f32(score, c);
  }
  if ((p + 1) % r != 0) return;   // uniform over the cluster
  const uint32_t i = (p + 1) / r - 1;
  const T *ape = static_cast<const T *>(L.ape);
  const T *gamma = static_cast<const T *>(L.gamma);
  __syncthreads();   // the token's slot is written
  // channels cbase + 64 q + 2 pr, + 1 (q < cpc / 64); slots g, g + 8, ...
  const uint32_t nq = cpc / 64;
  float y[2][2];
  for (uint32_t q = 0; q < nq; ++q) {
    const uint32_t c = cbase + 64 * q + 2 * pr;
    float2 kv[SPT], sg[SPT];
#pragma unroll
    for (uint32_t j = 0; j < SPT; ++j) {
      const uint32_t sl = g + kSlotGroups * j;
      kv[j] = *reinterpret_cast<const float2 *>(skv + (size_t)sl * width + c);
      const float2 sc = *reinterpret_cast<const float2 *>(ssc + (size_t)sl * width + c);
      sg[j] = make_float2(sc.x + ld_f32(ape, (size_t)sl * width + c),
                          sc.y + ld_f32(ape, (size_t)sl * width + c + 1));
    }
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (uint32_t j = 0; j < SPT; ++j) {
      m0 = fmaxf(m0, sg[j].x);
      m1 = fmaxf(m1, sg[j].y);
    }
    sm_max[g][2 * pr] = m0;
    sm_max[g][2 * pr + 1] = m1;
    __syncthreads();
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (uint32_t gg = 0; gg < kSlotGroups; ++gg) {
      M0 = fmaxf(M0, sm_max[gg][2 * pr]);
      M1 = fmaxf(M1, sm_max[gg][2 * pr + 1]);
    }
    float d0 = 0.f, n0 = 0.f, d1 = 0.f, n1 = 0.f;
    if (M0 != -INFINITY) {
#pragma unroll
      for (uint32_t j = 0; j < SPT; ++j) {
        const float w = expf(sg[j].x - M0);
        if (w > 0.f) {
          d0 += w;
          n0 += w * kv[j].x;
        }
      }
    }
    if (M1 != -INFINITY) {
#pragma unroll
      for (uint32_t j = 0; j < SPT; ++j) {
        const float w = expf(sg[j].y - M1);
        if (w > 0.f) {
          d1 += w;
          n1 += w * kv[j].y;
        }
      }
    }
    sm_den[g][2 * pr] = d0;
    sm_den[g][2 * pr + 1] = d1;
    sm_num[g][2 * pr] = n0;
    sm_num[g][2 * pr + 1] = n1;
    __syncthreads();
    if (g == 0) {
      float D0 = 0.f, N0 = 0.f, D1 = 0.f, N1 = 0.f;
#pragma unroll
      for (uint32_t gg = 0; gg < kSlotGroups; ++gg) {
        D0 += sm_den[gg][2 * pr];
        N0 += sm_num[gg][2 * pr];
        D1 += sm_den[gg][2 * pr + 1];
        N1 += sm_num[gg][2 * pr + 1];
      }
      y[q][0] = D0 > 0.f ? N0 / D0 : 0.f;
      y[q][1] = D1 > 0.f ? N1 / D1 : 0.f;
    }
    __syncthreads();   // the shared partials are reused by the next 64 channels
  }
  if (r == 4) {   // every read of slots 0..3 is done: the frontier moves
    for (uint32_t c = cbase + t; c < cbase + cpc; c += kThreads) {
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        skv[(size_t)sl * width + c] = skv[(size_t)(4 + sl) * width + c];
        ssc[(size_t)sl * width + c] = ssc[(size_t)(4 + sl) * width + c];
      }
    }
  }
  // RMS over the whole row: this CTA's squares, then every rank's in order
  if (g == 0) {
    float ss = 0.f;
    for (uint32_t q = 0; q < nq; ++q) ss += y[q][0] * y[q][0] + y[q][1] * y[q][1];
    ss = warp_sum(ss);
    if (pr == 0) part = ss;
  }
  cluster_sync_all();
  float tot = 0.f;
  if (g == 0) {
    const uint32_t addr = smem_u32(&part);
    for (uint32_t rr = 0; rr < kSplit; ++rr) tot += ld_cluster_f32(mapa_shared(addr, rr));
  }
  cluster_sync_all();   // every rank's partial has been read
  if (g != 0) return;
  const float inv = 1.0f / sqrtf(tot / (float)width + kRmsEps);
  const uint32_t n_nope = width - L.n_rot;
  size_t prow;
  const bool mapped = L.map.phys(b, i, prow);
  T *row = static_cast<T *>(L.comp) + prow * width;
  for (uint32_t q = 0; q < nq; ++q) {
    const uint32_t c = cbase + 64 * q + 2 * pr;
    float v0 = ld_f32(gamma, c) * (y[q][0] * inv);
    float v1 = ld_f32(gamma, c + 1) * (y[q][1] * inv);
    if (c >= n_nope) {
      const uint32_t fi = (c - n_nope) / 2;
      const float co = L.cos[(size_t)(i * r) * (L.n_rot / 2) + fi];
      const float si = L.sin[(size_t)(i * r) * (L.n_rot / 2) + fi];
      const float r0 = v0 * co - v1 * si, r1 = v0 * si + v1 * co;
      v0 = r0;
      v1 = r1;
    }
    if (L.quant == 1) {   // FP8 on the non-RoPE dims: this warp's 64 channels are one block
      const bool in = c < n_nope;
      const float am = warp_max(in ? fmaxf(fabsf(v0), fabsf(v1)) : 0.f);
      const int ke = block_scale_exp(am, kE4M3);
      if (in) {
        v0 = quant_dequant(v0, ke, kE4M3);
        v1 = quant_dequant(v1, ke, kE4M3);
      }
    }
    if (mapped) {
      st_elem(row, c, v0);
      st_elem(row, c + 1, v1);
    }
  }
}

// Window slot s of compressed row i, for a chunk that starts at pos0: the
// token is i*r + s - (W - r); tokens before 0 are empty, tokens of the chunk
// come from the inputs, earlier ones from the state as it was before the chunk.
template <typename T>
struct ChunkSlot {
  const LaneArgs *L;
  uint32_t r, W, b, i, pos0, T_len;
  __device__ SlotVal operator()(uint32_t s, uint32_t c) const {
    const int64_t tok = (int64_t)i * r + s - (int64_t)(W - r);
    const uint32_t width = L->width;
    if (tok < 0) return SlotVal{0.f, -INFINITY};
    if (tok >= (int64_t)pos0) {
      const size_t off = ((size_t)b * T_len + (size_t)(tok - pos0)) * width + c;
      return SlotVal{ld_f32(static_cast<const T *>(L->cand), off),
                     ld_f32(static_cast<const T *>(L->score), off)};
    }
    uint32_t slot;
    if (r == 4)
      slot = tok >= (int64_t)(pos0 / 4) * 4 ? 4 + (uint32_t)(tok % 4) : (uint32_t)(tok % 4);
    else
      slot = (uint32_t)(tok % r);
    const size_t off = ((size_t)b * W + slot) * width + c;
    return SlotVal{L->state_kv[off], L->state_score[off]};
  }
};

// n_emit: compressed rows per lane the grid has room for (the most any
// sequence completes in the chunk); sequence b, whose chunk starts at p0 (its
// own position in a ragged batch), completes (p0 + T) / r - p0 / r of them.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    append_rows_kernel(AppendArgs a, uint32_t n_raw, uint32_t n_emit) {
  __shared__ float red[32];
  const uint32_t b = blockIdx.y;
  const uint32_t p0 = seq_base(a.seq_pos, a.pos0, b);
  uint32_t x = blockIdx.x;
  if (x < n_raw) {
    const uint32_t t = (a.direct ? a.T - n_raw : 0) + x;
    const uint32_t p = p0 + t;
    const T *src = static_cast<const T *>(a.raw_in) + ((size_t)b * a.T + t) * a.head_dim;
    T *dst = static_cast<T *>(a.raw_dst) +
             (a.direct ? ((size_t)b * a.cap_raw + p % a.cap_raw) * a.head_dim
                       : ((size_t)b * a.T + t) * a.head_dim);
    raw_row(src, dst, a.head_dim, a.n_rot, p, a.cos, a.sin);
    return;
  }
  x -= n_raw;
  const uint32_t l = x / n_emit, e = x % n_emit;
  const LaneArgs &L = a.lane[l];
  const uint32_t r = a.ratio, i = p0 / r + e;
  if (e >= (p0 + a.T) / r - p0 / r) return;   // (ragged: fewer rows in this sequence)
  ChunkSlot<T> get{&L, r, a.window, b, i, p0, a.T};
  pool_norm_rope_store<T>(L, a.window, b, i, i * r, get, red);
}

// State after the chunk, as the token-by-token process leaves it.
template <typename T>
__global__ void __launch_bounds__(kThreads) append_state_kernel(AppendArgs a) {
  const uint32_t b = blockIdx.x;
  const LaneArgs &L = a.lane[blockIdx.y];
  const uint32_t r = a.ratio, W = a.window, width = L.width;
  const uint32_t pos0 = seq_base(a.seq_pos, a.pos0, b), n = pos0 + a.T;
  float *skv = L.state_kv + (size_t)b * W * width;
  float *ssc = L.state_score + (size_t)b * W * width;
  const T *cand = static_cast<const T *>(L.cand) + (size_t)b * a.T * width;
  const T *score = static_cast<const T *>(L.score) + (size_t)b * a.T * width;
  for (uint32_t c = threadIdx.x; c < width; c += blockDim.x) {
    if (r == 4) {
      float nkv[8], nsc[8];
      bool wr[8];
#pragma unroll
      for (int s = 0; s < 8; ++s) wr[s] = false;
      // slots 4+j: the last chunk token with p % 4 == j
#pragma unroll
      for (uint32_t j = 0; j < 4; ++j) {
        const int64_t tl = (int64_t)n - 1 - (int64_t)((n - 1 + 4 - j) % 4);
        if (tl >= (int64_t)pos0) {
          nkv[4 + j] = ld_f32(cand, (size_t)(tl - pos0) * width + c);
          nsc[4 + j] = ld_f32(score, (size_t)(tl - pos0) * width + c);
          wr[4 + j] = true;
        }
      }
      // slots 0..3: the group moved there by the last boundary inside the chunk
      const int64_t pb = (int64_t)(n / 4) * 4 - 1;
      if (pb >= (int64_t)pos0) {
#pragma unroll
        for (uint32_t j = 0; j < 4; ++j) {
          const int64_t tok = pb - 3 + j;
          if (tok >= (int64_t)pos0) {
            nkv[j] = ld_f32(cand, (size_t)(tok - pos0) * width + c);
            nsc[j] = ld_f32(score, (size_t)(tok - pos0) * width + c);
          } else {
            nkv[j] = skv[(size_t)(4 + j) * width + c];
            nsc[j] = ssc[(size_t)(4 + j) * width + c];
          }
          wr[j] = true;
        }
      }
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (wr[s]) {
          skv[(size_t)s * width + c] = nkv[s];
          ssc[(size_t)s * width + c] = nsc[s];
        }
    } else {
      for (uint32_t s = 0; s < W; ++s) {
        const int64_t tl = (int64_t)n - 1 - (int64_t)((n - 1 + W - s % W) % W);
        if (tl >= (int64_t)pos0) {
          skv[(size_t)s * width + c] = ld_f32(cand, (size_t)(tl - pos0) * width + c);
          ssc[(size_t)s * width + c] = ld_f32(score, (size_t)(tl - pos0) * width + c);
        }
      }
    }
  }
}

__global__ void state_reset_kernel(float *kv, float *score, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    kv[i] = 0.f;
    score[i] = -INFINITY;
  }
}

template <typename T>
cudaError_t launch_append_t(const AppendArgs &a, cudaStream_t s) {
  // compressed-layer decode with 512- or 1024-wide rows: one cluster per
  // (sequence, role)
  if (a.T == 1 && a.direct && a.ratio != 0 && a.head_dim % (64 * kSplit) == 0 &&
      a.head_dim <= 128 * kSplit) {
    const uint32_t roles = (a.y0 ? 0u : 1u) + (uint32_t)a.n_lanes;
    if (!roles) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kSplit;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(roles * a.batch * kSplit);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    cudaError_t e = a.ratio == 4 ? cudaLaunchKernelEx(&cfg, append_step_split_kernel<T, 8>, a)
                                 : cudaLaunchKernelEx(&cfg, append_step_split_kernel<T, 128>, a);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
  }
  if (a.T == 1 && a.direct) {
    const uint32_t roles = (a.y0 ? 0u : 1u) + (uint32_t)a.n_lanes;
    if (!roles) return cudaSuccess;
    cudaError_t e = launch_pdl(append_step_kernel<T>, dim3(a.batch, roles), dim3(kThreads), 0,
                               s, a);
    if (e != cudaSuccess) return e;
    note_launches(1);
    return cudaGetLastError();
  }
  const uint32_t n_raw = a.y0 ? 0u : a.direct ? (a.T < a.cap_raw ? a.T : a.cap_raw) : a.T;
  // rows completed in the chunk; with per-sequence positions, the most any
  // sequence can complete
  const uint32_t n_emit = !a.ratio ? 0u
                          : a.seq_pos ? a.T / a.ratio + 1u
                                      : (a.pos0 + a.T) / a.ratio - a.pos0 / a.ratio;
  const uint32_t nblk = n_raw + n_emit * a.n_lanes;
  if (nblk) {
    append_rows_kernel<T><<<dim3(nblk, a.batch), kThreads, 0, s>>>(a, n_raw, n_emit ? n_emit : 1);
    note_launches(1);
  }
  if (a.n_lanes) {
    append_state_kernel<T><<<dim3(a.batch, a.n_lanes), kThreads, 0, s>>>(a);
    note_launches(1);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const AppendArgs &a, cudaStream_t s) {
  return a.dtype == DS4A_BF16 ? launch_append_t<__nv_bfloat16>(a, s) : launch_append_t<float>(a, s);
}

cudaError_t launch_state_reset(float *kv, float *score, size_t n, cudaStream_t s) {
  if (!n) return cudaSuccess;
  const int blocks = (int)((n + 255) / 256 < 1184 ? (n + 255) / 256 : 1184);
  state_reset_kernel<<<blocks, 256, 0, s>>>(kv, score, n);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_index_norms(int dtype, const void *rows, const RowMap &map, uint32_t dim,
                               uint32_t batch, uint32_t n_rows, float *norm, uint32_t *norm_max,
                               cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const dim3 grid((n_rows + 7) / 8, batch);
  if (dtype == DS4A_BF16)
    index_norms_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(rows), map, dim,
                                            n_rows, norm, norm_max);
  else
    index_norms_kernel<<<grid, 256, 0, s>>>(static_cast<const float *>(rows), map, dim, n_rows,
                                            norm, norm_max);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace ds4a
