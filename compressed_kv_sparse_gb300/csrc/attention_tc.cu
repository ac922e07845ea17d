// Sparse attention on the tensor cores (bf16 layers, 64 heads x 512 dims,
// 64-dim rotated tail): "【#3】ds4.c を読み解く" §7 mixed attention; vLLM
// DeepSeek V4 page: shared K = V, inverse RoPE on the output, 128-token window.
//
// A work item is one query (and, in decode, one 128-row split of its row
// list). Its rows — the raw window followed by the compressed rows of the
// top-k list (ratio 4) or of the visible range (ratio 128) — are gathered 128
// at a time into shared memory, in eight 64-dim blocks laid out with the
// 128-byte swizzle. Each tile is used twice by the tensor cores, which is
// where K = V pays:
//   S^T = K Q^T    M = 128 rows, N = 64 heads, K = 512   (tile read K-major)
//   O^T += V^T P^T M = 4 x 128 dims, N = 64 heads, K = 128 rows (tile read MN-major)
// S^T (64 columns) and O^T (256 columns) live in TMEM. The softmax thread of a
// row reads its 64 head scores from its TMEM lane and writes its probabilities
// as one 128-byte row of P. The running maximum of each head starts at the
// scores of the first valid row and is only raised (rescaling O and the sums)
// when a score exceeds it by 2^8, so the common path needs no reduction across
// rows; the per-head sums are reduced once per query.
//
// Warps 0-3: softmax and output epilogue (TMEM lanes = rows, then dims);
// warps 4-7: gather loaders (cp.async, zero fill for masked rows) and the query
// rotation; warp 8: MMA issue (one thread) and TMEM allocation. Every wait is
// bounded (tc.cuh); a timeout sets the error word and the CTA winds down.
#include <cuda_bf16.h>

#include "common.cuh"
#include "tc.cuh"

namespace ds4a {
namespace {

constexpr int kH = 64, kD = 512, kNope = 448, kRows = 128;
constexpr int kQBlk = kH * 128;        // one 64-dim block of Q: 64 heads x 128 B
constexpr int kKBlk = kRows * 128;     // one 64-dim block of the row tile
constexpr int kThreads = 288;
constexpr uint32_t kNoRow = 0x7fffffffu;
constexpr float kRaiseLog2 = 8.0f;     // raise the running max beyond 2^8

struct TcAttnParams {
  uint32_t ratio, batch, T, pos0, cap_raw, comp_cap, n_comp, top_k;
  uint32_t n_splits, tiles_per_split, n_items;
  float c2;  // softmax scale * log2(e)
  const __nv_bfloat16 *q, *ring, *chunk, *comp;
  const int32_t *topk;
  const float *cos, *sin;
  __nv_bfloat16 *out;
  float *part;
  int *err;
};

struct Smem {
  uint8_t q[8 * kQBlk];     // 64 KiB
  uint8_t kv[8 * kKBlk];    // 128 KiB
  uint8_t p[kRows * 128];   // 16 KiB
  uint64_t kv_full[8], kv_empty[8];
  uint64_t q_full, q_empty, s_full, p_full, p_empty, o_full, o_empty, sm_bar, ld_bar;
  float mref[kH], alpha[kH], lsh[kH], linv[kH];
  float tmax[4][kH], lpart[4][kH];
  uint32_t first_row, flagcnt[3], tmem;
};

// Query-level geometry shared by every role.
struct QueryGeo {
  uint32_t qi, split, b, p, n_w, n_list, N, t0, t1;
  const int32_t *tk;
};

__device__ __forceinline__ QueryGeo query_geo(const TcAttnParams &P, uint32_t item, uint32_t lane) {
  QueryGeo g;
  g.qi = item / P.n_splits;
  g.split = item % P.n_splits;
  g.b = g.qi / P.T;
  g.p = P.pos0 + g.qi % P.T;
  g.n_w = min(g.p + 1, P.cap_raw);
  g.tk = P.topk ? P.topk + (size_t)g.qi * P.top_k : nullptr;
  g.n_list = 0;
  if (P.ratio == 4) {
    const uint32_t vis = min((g.p + 1) / 4, P.n_comp);
    // the list ends at its first entry >= vis; 8 independent loads per round
    g.n_list = P.top_k;
    for (uint32_t base = 0; base < P.top_k; base += 256) {
      int32_t v[8];
#pragma unroll
      for (uint32_t i = 0; i < 8; ++i) {
        const uint32_t j = base + 32 * i + lane;
        v[i] = j < P.top_k ? g.tk[j] : -1;
      }
      uint32_t found = 0xffffffffu;
#pragma unroll
      for (uint32_t i = 0; i < 8; ++i) {
        const uint32_t bal = __ballot_sync(0xffffffffu, v[i] >= 0 && (uint32_t)v[i] >= vis);
        if (bal && found == 0xffffffffu) found = base + 32 * i + __ffs(bal) - 1;
      }
      if (found != 0xffffffffu) {
        g.n_list = found;
        break;
      }
    }
  } else if (P.ratio == 128) {
    g.n_list = min((g.p + 1) / 128, P.n_comp);
  }
  g.N = g.n_w + g.n_list;
  const uint32_t n_tiles = (g.N + kRows - 1) / kRows;
  g.t0 = g.split * P.tiles_per_split;
  g.t1 = min(n_tiles, g.t0 + P.tiles_per_split);
  return g;
}

// Source row of list entry r (nullptr: masked).
__device__ __forceinline__ const __nv_bfloat16 *row_src(const TcAttnParams &P, const QueryGeo &g,
                                                        uint32_t r) {
  if (r < g.n_w) {
    const uint32_t pos = g.p - g.n_w + 1 + r;
    if (P.chunk && pos >= P.pos0)
      return P.chunk + ((size_t)g.b * P.T + (pos - P.pos0)) * kD;
    return P.ring + ((size_t)g.b * P.cap_raw + pos % P.cap_raw) * kD;
  }
  if (r < g.N) {
    const uint32_t j = r - g.n_w;
    const int32_t idx = P.ratio == 4 ? g.tk[j] : (int32_t)j;
    if (idx >= 0) return P.comp + ((size_t)g.b * P.comp_cap + (uint32_t)idx) * kD;
  }
  return nullptr;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(TcAttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  Smem &S = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~(uintptr_t)1023);
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) {
      mbar_init(&S.kv_full[i], 128);
      mbar_init(&S.kv_empty[i], 1);
    }
    mbar_init(&S.q_full, 128);
    mbar_init(&S.q_empty, 1);
    mbar_init(&S.s_full, 1);
    mbar_init(&S.p_full, 128);
    mbar_init(&S.p_empty, 1);
    mbar_init(&S.o_full, 1);
    mbar_init(&S.o_empty, 4);
    mbar_init(&S.sm_bar, 128);
    mbar_init(&S.ld_bar, 128);
    S.flagcnt[0] = S.flagcnt[1] = S.flagcnt[2] = 0;
    fence_mbar_init();
  }
  if (warp == 8) tmem_alloc(&S.tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem;
  // TMEM columns: S^T 0..63, row sums L 64..127, an all-ones bf16 A operand
  // 128..159 (L = ones x P^T), O^T 256..511
  const uint32_t tmS = tmem, tmL = tmem + 64, tmOnes = tmem + 128, tmO = tmem + 256;
  if (warp < 4) {
    uint32_t ones[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) ones[i] = 0x3F803F80u;   // two bf16 1.0
    tmem_st32(tmOnes + ((warp * 32) << 16), ones);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ loaders
    const uint32_t lt = threadIdx.x - 128, lw = warp - 4;
    uint32_t n = 0, qn = 0, ld_phase = 0;
    // issue all eight 64-dim blocks of a tile (one cp.async group each) as
    // their slots free up; rows of this lane: lw*32 + lane/8 + 4i, chunk lane%8
    auto issue_tile = [&](const QueryGeo &g, uint32_t tile, uint32_t n) -> bool {
      const __nv_bfloat16 *src[8];
#pragma unroll
      for (uint32_t i = 0; i < 8; ++i)
        src[i] = row_src(P, g, tile * kRows + lw * 32 + (lane >> 3) + 4 * i);
      const uint32_t cc = lane & 7;
      for (uint32_t kb = 0; kb < 8; ++kb) {
        if (!mbar_wait_warp(&S.kv_empty[kb], (n & 1) ^ 1, P.err)) return false;
        uint8_t *slot = S.kv + kb * kKBlk;
#pragma unroll
        for (uint32_t i = 0; i < 8; ++i) {
          const uint32_t r = lw * 32 + (lane >> 3) + 4 * i;
          uint8_t *dst = slot + (r >> 3) * 1024 + (r & 7) * 128 + ((cc ^ (r & 7)) << 4);
          const __nv_bfloat16 *sp = src[i] ? src[i] + kb * 64 + cc * 8 : P.ring;
          cp_async16(dst, sp, src[i] ? 16u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      }
      return true;
    };
    for (uint32_t item = blockIdx.x; item < P.n_items; item += gridDim.x) {
      const QueryGeo g = query_geo(P, item, lane);
      if (g.t0 >= g.t1) continue;
      if (!mbar_wait_warp(&S.q_empty, (qn & 1) ^ 1, P.err)) goto done_loader;
      {
        // Q: warp lw loads heads 16 lw .. 16 lw + 15, two half rows per head
        const __nv_bfloat16 *q = P.q + (size_t)g.qi * kH * kD;
        for (uint32_t hh = 0; hh < 16; ++hh) {
          const uint32_t h = lw * 16 + hh;
#pragma unroll
          for (uint32_t half = 0; half < 2; ++half) {
            const uint32_t ch = lane + 32 * half;           // 16-byte chunk 0..63 of the row
            const uint32_t kb = ch >> 3, c = ch & 7;
            uint8_t *dst = S.q + kb * kQBlk + h * 128 + ((c ^ (h & 7)) << 4);
            cp_async16(dst, q + (size_t)h * kD + ch * 8, 16);
          }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        // the first tile's rows start loading before Q is rotated
        if (!issue_tile(g, g.t0, n)) goto done_loader;
        asm volatile("cp.async.wait_group 8;" ::: "memory");   // Q landed
        if (!group_sync(&S.ld_bar, ld_phase, P.err)) goto done_loader;
        // rotate the tail (dims 448..511 = block 7) at position p, in place
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i) {
          const uint32_t id = lt + 128 * i, h = id >> 3, pc = id & 7, lc = pc ^ (h & 7);
          uint4 *ptr = reinterpret_cast<uint4 *>(S.q + 7 * kQBlk + h * 128 + pc * 16);
          uint4 v = *ptr;
          uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (uint32_t e = 0; e < 4; ++e) {
            const uint32_t fi = 4 * lc + e;
            const float co = P.cos[(size_t)g.p * 32 + fi], si = P.sin[(size_t)g.p * 32 + fi];
            const float x0 = bf16lo(w4[e]), x1 = bf16hi(w4[e]);
            w4[e] = pack_bf16(x0 * co - x1 * si, x0 * si + x1 * co);
          }
          *ptr = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        fence_proxy_async();
        mbar_arrive(&S.q_full);
      }
      for (uint32_t tile = g.t0; tile < g.t1; ++tile, ++n) {
        if (tile != g.t0 && !issue_tile(g, tile, n)) goto done_loader;
#define DS4A_KV_LANDED(NPEND, KB)                                   \
  asm volatile("cp.async.wait_group " #NPEND ";" ::: "memory");     \
  fence_proxy_async();                                              \
  mbar_arrive(&S.kv_full[KB]);
        DS4A_KV_LANDED(7, 0)
        DS4A_KV_LANDED(6, 1)
        DS4A_KV_LANDED(5, 2)
        DS4A_KV_LANDED(4, 3)
        DS4A_KV_LANDED(3, 4)
        DS4A_KV_LANDED(2, 5)
        DS4A_KV_LANDED(1, 6)
        DS4A_KV_LANDED(0, 7)
#undef DS4A_KV_LANDED
      }
      ++qn;
    }
  done_loader:
    cp_async_wait_all();
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idS = idesc_bf16_f32(kRows, kH);
    constexpr uint32_t idPV = idesc_bf16_f32(kRows, kH) | kIdescMajorA_MN | kIdescMajorB_MN;
    const uint32_t q_base = smem_u32(S.q), kv_base = smem_u32(S.kv), p_base = smem_u32(S.p);
    uint32_t n = 0, qn = 0;
    bool ok = true;
    for (uint32_t item = blockIdx.x; item < P.n_items && ok; item += gridDim.x) {
      const QueryGeo g = query_geo(P, item, lane);
      if (g.t0 >= g.t1) continue;
      if (lane == 0) {
        ok = mbar_wait(&S.q_full, qn & 1, P.err);
        for (uint32_t tile = g.t0; ok && tile < g.t1; ++tile, ++n) {
          const bool first = tile == g.t0, last = tile + 1 == g.t1;
          for (uint32_t kb = 0; kb < 8 && ok; ++kb) {
            ok = mbar_wait(&S.kv_full[kb], n & 1, P.err);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (uint32_t kk = 0; kk < 4; ++kk)
              mma_bf16(tmS, sdesc_sw128(kv_base + kb * kKBlk + kk * 32),
                       sdesc_sw128(q_base + kb * kQBlk + kk * 32), idS, (kb | kk) ? 1u : 0u);
          }
          if (!ok) break;
          mma_commit(&S.s_full);
          if (last) mma_commit(&S.q_empty);
          ok = mbar_wait(&S.p_full, n & 1, P.err);
          if (ok && first) ok = mbar_wait(&S.o_empty, (qn & 1) ^ 1, P.err);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (uint32_t m = 0; m < 4; ++m) {
#pragma unroll
            for (uint32_t kk = 0; kk < 8; ++kk) {
              const uint64_t ad = sdesc_sw128_mn(kv_base + 2 * m * kKBlk + kk * 2048, kKBlk, 1024);
              const uint64_t bd = sdesc_sw128_mn(p_base + kk * 2048, 8192, 1024);
              mma_bf16(tmO + m * kH, ad, bd, idPV, (first && kk == 0) ? 0u : 1u);
            }
            mma_commit(&S.kv_empty[2 * m]);
            mma_commit(&S.kv_empty[2 * m + 1]);
          }
          // per-head row sums of P on the tensor core: every row of L = 1^T P^T
          constexpr uint32_t idL = idesc_bf16_f32(kRows, kH) | kIdescMajorB_MN;
#pragma unroll
          for (uint32_t kk = 0; kk < 8; ++kk)
            mma_bf16_ta(tmL, tmOnes, sdesc_sw128_mn(p_base + kk * 2048, 8192, 1024), idL,
                        (first && kk == 0) ? 0u : 1u);
          mma_commit(&S.p_empty);
          if (last) mma_commit(&S.o_full);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      n = __shfl_sync(0xffffffffu, n, 0);
      ++qn;
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const uint32_t r = threadIdx.x;          // tile row / TMEM lane, then dim within a block
    const uint32_t lane_base = (warp * 32) << 16;
    uint32_t n = 0, qn = 0, sm_phase = 0;
    // P row r from the scores in TMEM with the current running maxima;
    // returns whether a score exceeds its head's maximum by more than 2^8
    auto write_p = [&](bool valid) {
      bool flag = false;
      uint8_t *prow = S.p + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (uint32_t hf = 0; hf < 2; ++hf) {
        uint32_t a[32];
        tmem_ld32(tmS + lane_base + 32 * hf, a);
        tmem_ld_wait();
#pragma unroll
        for (uint32_t c4 = 0; c4 < 4; ++c4) {
          uint32_t w4[4];
#pragma unroll
          for (uint32_t e = 0; e < 4; ++e) {
            const uint32_t hl = 8 * c4 + 2 * e, h = 32 * hf + hl;
            const float t0 = fmaf(__uint_as_float(a[hl]), P.c2, -S.mref[h]);
            const float t1 = fmaf(__uint_as_float(a[hl + 1]), P.c2, -S.mref[h + 1]);
            flag |= valid && (t0 > kRaiseLog2 || t1 > kRaiseLog2);
            w4[e] = valid ? pack_bf16(ex2_approx(t0), ex2_approx(t1)) : 0u;
          }
          *reinterpret_cast<uint4 *>(prow + (((4 * hf + c4) ^ (r & 7)) << 4)) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      return flag;
    };
    for (uint32_t item = blockIdx.x; item < P.n_items; item += gridDim.x) {
      const QueryGeo g = query_geo(P, item, lane);
      const bool has_tiles = g.t0 < g.t1;
      bool any_valid = false;
      for (uint32_t tile = g.t0; tile < g.t1; ++tile, ++n) {
        const bool first = tile == g.t0;
        const uint32_t row = tile * kRows + r;
        bool valid = row < g.n_w;
        if (!valid && row < g.N) valid = P.ratio != 4 || g.tk[row - g.n_w] >= 0;
        if (!mbar_wait_warp(&S.s_full, n & 1, P.err)) goto done_softmax;
        tc_fence_after();
        if (first) {
          // running maxima start at the scores of the first valid row
          if (r == 0) S.first_row = kNoRow;
          if (!group_sync(&S.sm_bar, sm_phase, P.err)) goto done_softmax;
          if (valid) atomicMin(&S.first_row, r);
          if (!group_sync(&S.sm_bar, sm_phase, P.err)) goto done_softmax;
          const uint32_t fr = S.first_row;
          // (tcgen05.ld is warp-collective: every lane loads, one lane keeps)
#pragma unroll 1
          for (uint32_t hf = 0; hf < 2; ++hf) {
            uint32_t a[32];
            tmem_ld32(tmS + lane_base + 32 * hf, a);
            tmem_ld_wait();
            if (fr == r) {
#pragma unroll
              for (int h = 0; h < 32; ++h) S.mref[32 * hf + h] = __uint_as_float(a[h]) * P.c2;
            }
          }
          if (fr == kNoRow && r == 0) {
#pragma unroll
            for (int h = 0; h < kH; ++h) S.mref[h] = 0.f;
          }
          any_valid = fr != kNoRow;
          if (!group_sync(&S.sm_bar, sm_phase, P.err)) goto done_softmax;
        }
        // P of this tile (the previous PV must be done with the buffer)
        if (!mbar_wait_warp(&S.p_empty, (n & 1) ^ 1, P.err)) goto done_softmax;
        const bool flag = write_p(valid);
        const uint32_t fc = n % 3;
        if (r == 0) S.flagcnt[(n + 1) % 3] = 0;
        if (flag) atomicAdd(&S.flagcnt[fc], 1u);
        if (!group_sync(&S.sm_bar, sm_phase, P.err)) goto done_softmax;
        if (S.flagcnt[fc] != 0) {
          // rare path: exact tile max per head, raise the running max, rescale
          // O and L, rewrite P
#pragma unroll 1
          for (uint32_t hf = 0; hf < 2; ++hf) {
            uint32_t a[32];
            tmem_ld32(tmS + lane_base + 32 * hf, a);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; ++h) {
              const float v = warp_max(valid ? __uint_as_float(a[h]) * P.c2 : -INFINITY);
              if (lane == (uint32_t)h) S.tmax[warp][32 * hf + h] = v;
            }
          }
          if (!group_sync(&S.sm_bar, sm_phase, P.err)) goto done_softmax;
          if (r < kH) {
            const float M = fmaxf(fmaxf(S.tmax[0][r], S.tmax[1][r]), fmaxf(S.tmax[2][r], S.tmax[3][r]));
            const float mo = S.mref[r], mn = fmaxf(mo, M);
            S.alpha[r] = exp2f(mo - mn);
            S.mref[r] = mn;
          }
          if (!group_sync(&S.sm_bar, sm_phase, P.err)) goto done_softmax;
          if (!first) {
#pragma unroll 1
            for (uint32_t m = 0; m < 10; ++m) {   // O^T (8 x 32 columns) then L (2 x 32)
              uint32_t a[32];
              const uint32_t ta = (m < 8 ? tmO + m * 32 : tmL + (m - 8) * 32) + lane_base;
              tmem_ld32(ta, a);
              tmem_ld_wait();
#pragma unroll
              for (int h = 0; h < 32; ++h)
                a[h] = __float_as_uint(__uint_as_float(a[h]) * S.alpha[32 * (m & 1) + h]);
              tmem_st32(ta, a);
            }
            tmem_st_wait();
          }
          write_p(valid);
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&S.p_full);
      }
      // ---- item end: per-head sums (any lane of L), then the output
      {
        const bool final_out = P.n_splits == 1;
        if (has_tiles) {
          if (!mbar_wait_warp(&S.o_full, qn & 1, P.err)) goto done_softmax;
          tc_fence_after();
          if (warp == 0) {   // every row of L holds the sums; warp 0 loads, lane 0 keeps
#pragma unroll 1
            for (uint32_t hf = 0; hf < 2; ++hf) {
              uint32_t a[32];
              tmem_ld32(tmL + lane_base + 32 * hf, a);
              tmem_ld_wait();
              if (lane == 0) {
#pragma unroll
                for (int h = 0; h < 32; ++h) {
                  const float l = __uint_as_float(a[h]);
                  S.lsh[32 * hf + h] = l;
                  S.linv[32 * hf + h] = __frcp_rn(l);
                }
              }
            }
          }
        } else if (r < kH) {
          S.lsh[r] = 0.f;
          S.linv[r] = 0.f;
        }
        if (!group_sync(&S.sm_bar, sm_phase, P.err)) goto done_softmax;
        float co = 1.f, si = 0.f;
#pragma unroll 1
        for (uint32_t m = 0; m < 4; ++m) {
          const uint32_t d = m * 128 + r;
          const bool tail = final_out && d >= (uint32_t)kNope;
          if (tail) {
            const uint32_t fi = (d - kNope) >> 1;
            co = P.cos[(size_t)g.p * 32 + fi];
            si = P.sin[(size_t)g.p * 32 + fi];
          }
#pragma unroll 1
          for (uint32_t hf = 0; hf < 2; ++hf) {
            uint32_t a[32];
            if (has_tiles) {
              tmem_ld32(tmO + lane_base + m * kH + 32 * hf, a);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int h = 0; h < 32; ++h) a[h] = 0u;
            }
            if (final_out) {
              __nv_bfloat16 *o = P.out + (size_t)g.qi * kH * kD + (size_t)(32 * hf) * kD + d;
              if (m == 3 && r >= 64) {   // warp-uniform: the rotated tail dims
#pragma unroll
                for (int h = 0; h < 32; ++h) {
                  float v = __uint_as_float(a[h]) * S.linv[32 * hf + h];
                  const float other = __shfl_xor_sync(0xffffffffu, v, 1);
                  // rotate back by -p: (x0, x1) -> (x0 c + x1 s, -x0 s + x1 c)
                  v = (d & 1) ? (v * co - other * si) : (v * co + other * si);
                  o[(size_t)h * kD] = __float2bfloat16_rn(v);
                }
              } else {
#pragma unroll
                for (int h = 0; h < 32; ++h)
                  o[(size_t)h * kD] = __float2bfloat16_rn(__uint_as_float(a[h]) * S.linv[32 * hf + h]);
              }
            } else {
              float *po = P.part + ((size_t)g.qi * P.n_splits + g.split) * kH * kD +
                          (size_t)(32 * hf) * kD + d;
#pragma unroll
              for (int h = 0; h < 32; ++h) po[(size_t)h * kD] = __uint_as_float(a[h]);
            }
          }
        }
        if (!final_out && r < kH) {
          const size_t nq = (size_t)P.batch * P.T;
          float *pml = P.part + nq * P.n_splits * kH * kD +
                       (((size_t)g.qi * P.n_splits + g.split) * kH + r) * 2;
          pml[0] = any_valid ? S.mref[r] * 0.69314718055994531f : -INFINITY;
          pml[1] = S.lsh[r];
        }
        if (has_tiles) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.o_empty);
          ++qn;
        }
      }
      // keep the shared sums alive until every thread has read them
      if (!group_sync(&S.sm_bar, sm_phase, P.err)) goto done_softmax;
    }
  done_softmax:;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, 512);
}

}  // namespace

bool attn_tc_supported(int dtype, uint32_t H, uint32_t D, uint32_t n_rot) {
  return dtype == DS4A_BF16 && H == (uint32_t)kH && D == (uint32_t)kD && n_rot == 64;
}

uint32_t attn_tc_splits(uint32_t T, uint32_t rows_max) {
  return T == 1 ? (rows_max + kRows - 1) / kRows : 1;
}

cudaError_t launch_attention_tc(const AttnArgs &a, uint32_t rows_max, int *err, cudaStream_t s) {
  TcAttnParams P;
  P.ratio = a.ratio;
  P.batch = a.batch;
  P.T = a.T;
  P.pos0 = a.pos0;
  P.cap_raw = a.cap_raw;
  P.comp_cap = a.comp_cap;
  P.n_comp = a.n_comp;
  P.top_k = a.top_k;
  P.n_splits = attn_tc_splits(a.T, rows_max);
  P.tiles_per_split = a.T == 1 ? 1 : (rows_max + kRows - 1) / kRows;
  P.n_items = a.batch * a.T * P.n_splits;
  P.c2 = a.scale * 1.4426950408889634f;
  P.q = static_cast<const __nv_bfloat16 *>(a.q);
  P.ring = static_cast<const __nv_bfloat16 *>(a.ring);
  P.chunk = static_cast<const __nv_bfloat16 *>(a.chunk);
  P.comp = static_cast<const __nv_bfloat16 *>(a.comp);
  P.topk = a.topk;
  P.cos = a.cos;
  P.sin = a.sin;
  P.out = static_cast<__nv_bfloat16 *>(a.out);
  P.part = static_cast<float *>(a.ws);
  P.err = err;
  const size_t smem = sizeof(Smem) + 1024;
  static int smem_set = 0;
  cudaError_t e = ensure_smem(attn_tc_kernel, smem, &smem_set);
  if (e != cudaSuccess) return e;
  const uint32_t grid = min(P.n_items, (uint32_t)num_sms());
  attn_tc_kernel<<<grid, kThreads, smem, s>>>(P);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace ds4a
