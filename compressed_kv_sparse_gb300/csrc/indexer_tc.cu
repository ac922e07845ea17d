// Indexer scores on the tensor cores (bf16 layers): approximate fp32 scores
// whose error the certified top-k bounds with the row norms kept in the cache
// ("【#3】ds4.c を読み解く" §6 indexer; vLLM DeepSeek V4 page, DSA).
//
// For every visible compressed index row s of sequence b and every query t of
// a group of QG queries:  S~(t, s) = sum_h w_h(t) * max(0, q'_h(t) . k_s).
// The dot products are one tcgen05 MMA per 128-row tile: A = 128 key rows
// (M = 128, K = Di = 128, TMA-loaded with the 128-byte swizzle), B = the QG x 64
// rotated query heads (N = 64 QG); the fp32 accumulator sits in TMEM (two
// buffers so the epilogue of one tile overlaps the MMA of the next). Each
// epilogue thread owns one TMEM lane = one key row of its warp's queries: it
// reads their 64 head dots each and applies ReLU and the head weights; with
// QG = 1 (decode) it also counts the top 12 bits of each score key into a
// per-CTA histogram that the selection uses to place its threshold.
//
// Persistent kernel, one CTA per SM: warp 0 issues TMA, warp 1 issues MMAs
// (one thread each), warps 2.. run the epilogue (4 for one query per group,
// 16 for four: one query each, four per TMEM lane quarter). Work items are
// (sequence, query group, 128-row tile), split into contiguous ranges so the
// B operand (the query group's heads) is reloaded only when the group
// changes: an even share of one group's visible tiles per CTA (decode), or
// an even share of all visible tiles from a host-computed range table
// (chunks, whose later queries see more rows).
// Every wait is bounded (tc.cuh); on a timeout the kernel sets *err and winds
// down, still freeing its TMEM.
#include <cuda_bf16.h>

#include "common.cuh"
#include "split.h"
#include "tc.cuh"

namespace ds4a {
namespace {

constexpr int kRows = 128;         // key rows per tile (MMA M)
constexpr int kDim = 128;          // Di (MMA K)
constexpr int kHeads = 64;         // Hi
constexpr int kKBlockBytes = kRows * 128;          // one 64-column K block of A
constexpr int kABytes = 2 * kKBlockBytes;          // 32 KiB per A stage

template <int QG>
struct Cfg {
  static constexpr int N = kHeads * QG;
  // epilogue warps: 4 (one per TMEM lane quarter) for one query, 16 for four
  // (four per quarter, one query each)
  static constexpr int kEpiWarps = QG == 1 ? 4 : 16;
  static constexpr int kQPW = QG * 4 / kEpiWarps;   // queries per epilogue warp
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kStages = QG == 1 ? 5 : 4;
  static constexpr int kHistBytes = QG == 1 ? 4096 * 4 : 0;   // per-CTA key histogram
  static constexpr int kBBytes = N * kDim * 2;
  // two accumulators of N columns (the allocation is a power of two >= 32)
  static constexpr int kTmemCols = QG == 1 ? 128 : 512;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kABytes + kBBytes + 1024 +
                                  kEpiWarps * QG * kHeads * 4 + kHistBytes;
};

constexpr uint32_t kMaxSplit = 256;   // CTAs of a range table (more: the even item split)

struct ScoreParams {
  uint32_t batch, T, pos0, comp_cap, n_comp, n_groups, tiles_per, total_items;
  uint32_t cta_per_group;   // > 0: that many CTAs per (sequence, group), none crossing one
  // split > 0: CTA j takes the items it_start[j] .. it_start[j + 1] - 1, an even
  // share of the visible tiles (computed on the host when every sequence
  // starts at pos0)
  uint32_t split;
  uint32_t it_start[kMaxSplit + 1];
  RowMap map;               // paged keys (map.table != NULL): 64-row blocks of the pool
  const uint32_t *seq_pos;  // [B] per-sequence positions (ragged decode) or NULL
  const __nv_bfloat16 *w;   // [B][T][Hi]
  float *scores;            // [B][T][score_stride]
  uint32_t score_stride;
  uint32_t *hist;           // [B*T][4096] counts of the top 12 bits of the score keys
  int *err;
};

// Order-preserving unsigned key of an fp32 score (+0 and -0 share a key).
__device__ __forceinline__ uint32_t score_key_tc(float f) {
  if (f == 0.f) f = 0.f;
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t vis_of(const ScoreParams &P, uint32_t b, uint32_t t) {
  return min((seq_base(P.seq_pos, P.pos0, b) + t + 1) / 4, P.n_comp);
}

// Walk over the work items it .. end - 1, item = (b * n_groups + g) *
// tiles_per + tile, without a division per item. A tile is visited when some
// row of it is visible to the group's last query (n_vis: the group's visible
// tiles); the rest of a group is skipped in one step. Every role walks the
// same items in the same order.
struct Walk {
  uint32_t it, end, b, g, tile, n_vis;
};

template <int QG>
__device__ __forceinline__ uint32_t visible_tiles(const ScoreParams &P, uint32_t b, uint32_t g) {
  const uint32_t last = min(P.T, (g + 1) * QG) - 1;
  return min(P.tiles_per, (vis_of(P, b, last) + kRows - 1) / kRows);
}

template <int QG>
__device__ __forceinline__ Walk walk_start(const ScoreParams &P, uint32_t i0, uint32_t i1) {
  Walk w;
  w.it = i0;
  w.end = i1;
  w.tile = i0 % P.tiles_per;
  const uint32_t rest = i0 / P.tiles_per;
  w.g = rest % P.n_groups;
  w.b = rest / P.n_groups;
  w.n_vis = i0 < i1 ? visible_tiles<QG>(P, w.b, w.g) : 0u;
  return w;
}

// Moves to the first visible item at or after the current one; false when
// the range is done.
template <int QG>
__device__ __forceinline__ bool walk_valid(const ScoreParams &P, Walk &w) {
  while (w.it < w.end) {
    if (w.tile < w.n_vis) return true;
    w.it += P.tiles_per - w.tile;   // the group's first tile past its visible ones
    w.tile = 0;
    if (++w.g == P.n_groups) {
      w.g = 0;
      ++w.b;
    }
    if (w.it < w.end) w.n_vis = visible_tiles<QG>(P, w.b, w.g);
  }
  return false;
}

template <int QG>
__device__ __forceinline__ void walk_next(const ScoreParams &P, Walk &w) {
  ++w.it;
  if (++w.tile == P.tiles_per) {
    w.tile = 0;
    if (++w.g == P.n_groups) {
      w.g = 0;
      ++w.b;
    }
    if (w.it < w.end) w.n_vis = visible_tiles<QG>(P, w.b, w.g);
  }
}

// d0 += a0 * b0, d1 += a1 * b1 as one packed fp32 pair FMA (round to nearest
// each, as two fmaf)
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0,
                                      float b1) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

template <int QG>
__global__ void __launch_bounds__(Cfg<QG>::kThreads, 1)
    index_score_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_q, ScoreParams P) {
  using C = Cfg<QG>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned. Decode (QG = 1) takes an offset from the shared array
  // itself, so its accesses compile to shared-memory instructions (index
  // call 36.5 -> 35.8 us at 8 x 32,768 rows); the four-query form keeps the
  // integer round trip and generic accesses, which measured faster there
  // (prefill index 725 against 743 us)
  uint8_t *smem;
  if (QG == 1)
    smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  else
    smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~(uintptr_t)1023);
  uint8_t *sA = smem;                                   // [stages][32 KiB]
  uint8_t *sB = sA + (size_t)C::kStages * kABytes;       // [2 K blocks][N][64] bf16
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + C::kBBytes);
  uint64_t *a_full = bars, *a_empty = bars + C::kStages;
  uint64_t *acc_full = a_empty + C::kStages, *acc_empty = acc_full + 2;
  uint64_t *b_full = acc_empty + 2, *b_empty = b_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(b_empty + 1);
  float *sw_all = reinterpret_cast<float *>(sB + C::kBBytes + 1024);   // [epi warps][QG][64]
  uint32_t *shist = reinterpret_cast<uint32_t *>(sw_all + C::kEpiWarps * QG * kHeads);   // QG == 1
  uint64_t *epi_bar = reinterpret_cast<uint64_t *>(tmem_slot + 2);

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work range: contiguous items, or (cta_per_group > 0) an even share of one
  // (sequence, group)'s visible tiles, so that no CTA changes query mid-range
  uint32_t it0, it1;
  if (P.cta_per_group) {
    const uint32_t bg = blockIdx.x / P.cta_per_group, j = blockIdx.x % P.cta_per_group;
    const uint32_t last = min(P.T, (bg % P.n_groups + 1) * QG) - 1;
    const uint32_t nt =
        min(P.tiles_per, (vis_of(P, bg / P.n_groups, last) + kRows - 1) / kRows);
    it0 = bg * P.tiles_per + j * nt / P.cta_per_group;
    it1 = bg * P.tiles_per + (j + 1) * nt / P.cta_per_group;
  } else if (P.split) {
    it0 = P.it_start[blockIdx.x];
    it1 = P.it_start[blockIdx.x + 1];
  } else {
    const uint32_t per = (P.total_items + gridDim.x - 1) / gridDim.x;
    it0 = min(P.total_items, blockIdx.x * per);
    it1 = min(P.total_items, it0 + per);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], C::kEpiWarps);
    }
    mbar_init(b_full, 1);
    mbar_init(b_empty, 1);
    mbar_init(epi_bar, 128);
    fence_mbar_init();
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_q);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x != 0) {   // the TMA producer waits after its first key loads
    pdl_wait();
    pdl_trigger();
  }

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      uint32_t stage = 0, phase = 0, b_phase = 0;
      int32_t cur = -1;
      int issued[C::kStages];
      for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
      // one 128-row key tile: two 64-dim K blocks, each one box of 128 rows
      // (contiguous keys) or two boxes of 64 rows from the tile's two
      // physical blocks (paged)
      // one query per group (decode): the keys stream through once, so
      // evict-first keeps them from pushing the step's code and small reused
      // arrays out of L2; every group of a chunk rereads the same keys, which
      // stay at the default priority
      const uint64_t pol = QG == 1 ? l2_evict_first_policy() : l2_evict_normal_policy();
      auto issue_a = [&](uint32_t st, uint32_t b, uint32_t tile) {
        uint8_t *dst = sA + (size_t)st * kABytes;
        mbar_arrive_expect_tx(&a_full[st], kABytes);
        if (!P.map.table) {
          tma_load_3d_hint(dst, &tmap_k, &a_full[st], 0, (int)(tile * kRows), (int)b, pol);
          tma_load_3d_hint(dst + kKBlockBytes, &tmap_k, &a_full[st], 64, (int)(tile * kRows),
                           (int)b, pol);
        } else {
#pragma unroll
          for (uint32_t hb = 0; hb < 2; ++hb) {
            const int y = (int)P.map.row_of(b, tile * kRows + 64 * hb);
            tma_load_2d_hint(dst + hb * (kKBlockBytes / 2), &tmap_k, &a_full[st], 0, y, pol);
            tma_load_2d_hint(dst + kKBlockBytes + hb * (kKBlockBytes / 2), &tmap_k, &a_full[st],
                             64, y, pol);
          }
        }
      };
      // the key tiles of the first stages load before the wait for the
      // previous launch: the rows were written two or more launches back
      uint32_t pre = 0;
      for (Walk w = walk_start<QG>(P, it0, it1); pre < (uint32_t)C::kStages && walk_valid<QG>(P, w);
           walk_next<QG>(P, w)) {
        issue_a(pre, w.b, w.tile);
        issued[pre] = 0;
        ++pre;
      }
      pdl_wait();
      pdl_trigger();
      uint32_t n_vis = 0;
      for (Walk w = walk_start<QG>(P, it0, it1); walk_valid<QG>(P, w); walk_next<QG>(P, w)) {
        const uint32_t b = w.b, g = w.g, tile = w.tile;
        const int32_t bg = (int32_t)(b * P.n_groups + g);
        if (bg != cur) {
          if (cur >= 0) {
            if (!mbar_wait(b_empty, b_phase, P.err)) break;
            b_phase ^= 1;
          }
          mbar_arrive_expect_tx(b_full, C::kBBytes);
          const int row0 = (int)((b * P.T + g * QG) * kHeads);
          tma_load_2d(sB, &tmap_q, b_full, 0, row0);
          tma_load_2d(sB + C::kBBytes / 2, &tmap_q, b_full, 64, row0);
          cur = bg;
        }
        if (n_vis++ >= pre) {   // (the first `pre` are in flight already)
          if (!mbar_wait(&a_empty[stage], phase ^ 1, P.err)) break;
          issue_a(stage, b, tile);
          issued[stage] = (int)phase;
        }
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      // let every load this CTA issued land before the CTA can exit
      for (int s = 0; s < C::kStages; ++s) {
        if (issued[s] < 0) continue;
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(&a_full[s], (uint32_t)issued[s]) &&
               global_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kRows, C::N);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, bf_phase = 0;
      int32_t cur = -1;
      const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
      for (Walk w = walk_start<QG>(P, it0, it1); walk_valid<QG>(P, w); walk_next<QG>(P, w)) {
        const int32_t bg = (int32_t)(w.b * P.n_groups + w.g);
        if (bg != cur) {
          if (cur >= 0) mma_commit(b_empty);
          if (!mbar_wait(b_full, bf_phase, P.err)) break;
          bf_phase ^= 1;
          cur = bg;
        }
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, P.err)) break;
        if (!mbar_wait(&a_full[stage], phase, P.err)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * C::N;
        const uint32_t a0 = a_base + stage * kABytes;
#pragma unroll
        for (uint32_t kk = 0; kk < kDim / 16; ++kk) {
          const uint32_t koff = (kk % 4) * 32;   // 16 bf16 = 32 B inside a swizzle row
          const uint64_t ad = sdesc_sw128(a0 + (kk / 4) * kKBlockBytes + koff);
          const uint64_t bd = sdesc_sw128(b_base + (kk / 4) * (C::kBBytes / 2) + koff);
          mma_bf16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&a_empty[stage]);
        mma_commit(&acc_full[acc]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else {
    // ---------------- epilogue: warps 2.., TMEM lanes 32 * (warp % 4) ..,
    // queries kQPW * ((warp - 2) / 4) .. + kQPW - 1
    const uint32_t lg = warp & 3, q0 = C::kQPW * ((warp - 2) >> 2);
    const uint32_t row = lg * 32 + lane;
    float *sw = sw_all + (warp - 2) * QG * kHeads;   // this warp's copy of the weights
    const uint32_t et = threadIdx.x - 64;             // 0..127
    uint32_t acc = 0, acc_phase = 0, epi_phase = 0;
    int32_t cur = -1;
    bool ok = true;
    // one query per group when QG == 1: its key histogram is gathered here and
    // added to the global one when the query changes
    auto flush_hist = [&](int32_t q) {
      if (!group_sync(epi_bar, epi_phase, P.err)) return false;
      // eight 16-byte loads per thread in flight at once, then the adds
      uint4 *h4 = reinterpret_cast<uint4 *>(shist);
      uint4 v[8];
#pragma unroll
      for (uint32_t j = 0; j < 8; ++j) v[j] = h4[et + 128 * j];
#pragma unroll
      for (uint32_t j = 0; j < 8; ++j) {
        const uint32_t c[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        if ((c[0] | c[1] | c[2] | c[3]) == 0u) continue;
        const uint32_t i0 = 4 * (et + 128 * j);
#pragma unroll
        for (uint32_t e = 0; e < 4; ++e)
          if (c[e] && q >= 0 && P.hist) atomicAdd(&P.hist[(size_t)q * 4096 + i0 + e], c[e]);
        h4[et + 128 * j] = make_uint4(0u, 0u, 0u, 0u);
      }
      return group_sync(epi_bar, epi_phase, P.err);
    };
    if (QG == 1) {
      for (uint32_t i = et; i < 4096; i += 128) shist[i] = 0;
    }
    uint32_t vis_q = 0;   // rows visible to this warp's query of the current group
    for (Walk w = walk_start<QG>(P, it0, it1); ok && walk_valid<QG>(P, w); walk_next<QG>(P, w)) {
      const uint32_t b = w.b, g = w.g, tile = w.tile;
      const int32_t bg = (int32_t)(b * P.n_groups + g);
      if (bg != cur) {
        if (QG == 1 && !flush_hist(cur)) {
          ok = false;
          break;
        }
        __syncwarp();
        for (uint32_t i = lane; i < QG * kHeads; i += 32) {
          const uint32_t t = g * QG + i / kHeads;
          sw[i] = t < P.T ? __bfloat162float(P.w[((size_t)b * P.T + t) * kHeads + i % kHeads])
                          : 0.f;
        }
        __syncwarp();
        const uint32_t tq = g * QG + q0;
        vis_q = tq < P.T ? vis_of(P, b, tq) : 0u;
        cur = bg;
      }
      if (!mbar_wait_warp(&acc_full[acc], acc_phase, P.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t grow = tile * kRows + row;
      static_assert(C::kQPW == 1, "one query per epilogue warp");
      {
        const int q = (int)q0;
        uint32_t r0[32], r1[32];
        const uint32_t taddr = tmem + ((lg * 32) << 16) + acc * C::N + q * kHeads;
        tmem_ld32(taddr, r0);
        tmem_ld32(taddr + 32, r1);
        tmem_ld_wait();
        // the accumulator is free once its columns are in registers: the
        // MMA two items on may start while this warp finishes the scores
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        // approximate score: any summation order is covered by the error
        // bound, so eight independent chains (as four packed pairs) and
        // vector loads of the weights
        const uint32_t wq_s = smem_u32(sw + q * kHeads);   // (explicit shared loads)
        float acc8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc8[j] = 0.f;
#pragma unroll
        for (int h4 = 0; h4 < 16; ++h4) {
          float4 w4;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(w4.x), "=f"(w4.y), "=f"(w4.z), "=f"(w4.w)
                       : "r"(wq_s + 16u * h4));
          const uint32_t *rr = h4 < 8 ? r0 : r1;
          const int hb = (h4 & 7) * 4, c = (2 * h4) & 7;
          ffma2(acc8[c], acc8[c + 1], w4.x, w4.y, fmaxf(__uint_as_float(rr[hb + 0]), 0.f),
                fmaxf(__uint_as_float(rr[hb + 1]), 0.f));
          ffma2(acc8[c], acc8[c + 1], w4.z, w4.w, fmaxf(__uint_as_float(rr[hb + 2]), 0.f),
                fmaxf(__uint_as_float(rr[hb + 3]), 0.f));
        }
        const float s = ((acc8[0] + acc8[1]) + (acc8[2] + acc8[3])) +
                        ((acc8[4] + acc8[5]) + (acc8[6] + acc8[7]));
        const uint32_t t = g * QG + q;
        const bool valid = grow < vis_q;
        if (valid) P.scores[((size_t)b * P.T + t) * P.score_stride + grow] = s;
        // histogram of the keys' top 12 bits (lanes in one bin add once), per
        // CTA in shared memory, added to the query's when the query changes
        if (QG == 1) {   // (the selection samples its threshold otherwise)
          const uint32_t bin = valid ? score_key_tc(s) >> 20 : 4096u;
          const uint32_t peers = __match_any_sync(0xffffffffu, bin);
          if (bin < 4096u && lane == (uint32_t)(__ffs(peers) - 1))
            atomicAdd(&shist[bin], (uint32_t)__popc(peers));
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (QG == 1 && ok && cur >= 0) flush_hist(cur);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <int QG>
cudaError_t launch_qg(const IndexTcArgs &a, cudaStream_t s) {
  using C = Cfg<QG>;
  CUtensorMap tk, tq;
  cudaError_t e;
  if (!a.map.table) {
    const uint64_t kd[3] = {kDim, a.comp_cap, a.batch};
    const uint64_t ks[2] = {(uint64_t)kDim * 2, (uint64_t)a.comp_cap * kDim * 2};
    const uint32_t kb[3] = {64, kRows, 1};
    e = make_tmap_bf16(&tk, a.keys, 3, kd, ks, kb);
  } else {   // the pool as [n_blocks * 64][128], boxes of 64 rows
    const uint64_t kd[2] = {kDim, (uint64_t)a.map.n_blocks * a.map.rpb};
    const uint64_t ks[1] = {(uint64_t)kDim * 2};
    const uint32_t kb[2] = {64, 64};
    e = make_tmap_bf16(&tk, a.keys, 2, kd, ks, kb);
  }
  if (e != cudaSuccess) return e;
  const uint64_t qd[2] = {kDim, (uint64_t)a.batch * a.T * kHeads};
  const uint64_t qs[1] = {(uint64_t)kDim * 2};
  const uint32_t qb[2] = {64, (uint32_t)C::N};
  e = make_tmap_bf16(&tq, a.qbf, 2, qd, qs, qb);
  if (e != cudaSuccess) return e;
  ScoreParams P;
  P.batch = a.batch;
  P.T = a.T;
  P.pos0 = a.pos0;
  P.comp_cap = a.comp_cap;
  P.n_comp = a.n_comp;
  P.n_groups = (a.T + QG - 1) / QG;
  const uint32_t vis_max = min((a.pos0 + a.T) / 4, a.n_comp);
  P.tiles_per = (vis_max + kRows - 1) / kRows;
  P.total_items = a.batch * P.n_groups * P.tiles_per;
  P.w = static_cast<const __nv_bfloat16 *>(a.w);
  P.scores = a.scores;
  P.score_stride = a.score_stride;
  P.hist = a.hist;
  P.err = a.err;
  P.map = a.map;
  P.seq_pos = a.seq_pos;
  if (P.total_items == 0) return cudaSuccess;
  static int smem_set = 0;
  e = ensure_smem(index_score_tc_kernel<QG>, C::kSmem, &smem_set);
  if (e != cudaSuccess) return e;
  // one group per CTA range when that costs no more tiles per CTA than the
  // contiguous split (a CTA that changes query reloads its heads and flushes
  // its histogram in between)
  const uint32_t sms = (uint32_t)num_sms(), n_bg = a.batch * P.n_groups;
  uint32_t grid = min(P.total_items, sms);
  P.cta_per_group = 0;
  P.split = 0;
  if (n_bg <= sms) {
    const uint32_t cpg = sms / n_bg;
    const uint32_t max_contig = (P.total_items + grid - 1) / grid;
    if ((P.tiles_per + cpg - 1) / cpg <= max_contig) {
      P.cta_per_group = cpg;
      grid = n_bg * cpg;
    }
  }
  if (!P.cta_per_group && !a.seq_pos && grid <= kMaxSplit) {
    // a chunk's later queries see more rows: split the visible tiles, not
    // the items, evenly (every sequence has the same visible tiles per group)
    split_visible_tiles(a.batch, a.T, QG, a.pos0, a.n_comp, kRows, P.n_groups, P.tiles_per, grid,
                        P.it_start);
    P.split = 1;
  }
  e = launch_pdl(index_score_tc_kernel<QG>, dim3(grid), dim3(C::kThreads), C::kSmem, s, tk, tq, P);
  if (e != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

bool index_tc_supported(uint32_t n_heads, uint32_t dim) {
  return n_heads == kHeads && dim == kDim;
}

cudaError_t launch_index_score_tc(const IndexTcArgs &a, cudaStream_t s) {
  return a.T >= 4 ? launch_qg<4>(a, s) : launch_qg<1>(a, s);
}

}  // namespace ds4a
