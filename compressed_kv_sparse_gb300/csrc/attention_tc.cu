// Sparse attention on the tensor cores (bf16 layers, 64 heads x 512 dims,
// 64-dim rotated tail): "【#3】ds4.c を読み解く" §7 mixed attention; vLLM
// DeepSeek V4 page: shared K = V, inverse RoPE on the output, 128-token window.
//
// A query's rows — the raw window followed by the compressed rows of the
// top-k list (ratio 4) or of the visible range (ratio 128) — are gathered 128
// at a time into shared memory, in eight 64-dim blocks laid out with the
// 128-byte swizzle. Each tile is used twice by the tensor cores, which is
// where K = V pays:
//   S^T = K Q^T    M = 128 rows, N = 64 heads, K = 512   (tile read K-major)
//   O^T += V^T P^T M = 4 x 128 dims, N = 64 heads, K = 128 rows (tile read MN-major)
// S^T (64 columns) and O^T (256 columns) live in TMEM. The softmax thread of a
// row reads its 64 head scores from its TMEM lane and writes its probabilities
// as one 128-byte row of P. The running maximum of each head starts at the
// exact per-head maximum of the query's first tile and is only raised
// (rescaling O and the sums) when a later score exceeds it by 2^8, so later
// tiles need no reduction across rows; the per-head sums come from the tensor
// core (ones x P^T).
//
// Decode: a query's 64 heads are split into two groups of 32, each its own
// set of CTAs over the same rows (S^T then has N = 32; P keeps the 64-column
// layout with the other group's columns zero, so PV and the sums are the
// 64-head MMAs). The tiles of a (query, head group) are spread over a
// thread-block cluster (rank c takes tiles c, c + C, ...). Each CTA writes its
// normalised O and per-head (max, sum) to the workspace straight from TMEM;
// after one cluster barrier, rank c pulls heads [32c/C, 32(c+1)/C) of the
// group from every rank into its freed tile buffer (bulk copies from L2),
// combines them in rank order, rotates the tail back and writes bf16 rows.
// (On this part the L2 round trip moves these bytes faster than distributed
// shared memory does.) Splitting the heads halves each CTA's softmax and
// exchange and doubles the CTAs a small batch puts to work. A (query, head
// group) that fits one CTA (C = 1) and prefill write the output directly from
// registers: lane pairs (dims d, d + 1) swap one value per pair of heads, so
// each thread rotates and stores one head's bf16 pair.
//
// In decode on ratios 0 and 128 the rows of a tile are contiguous (the
// window is the whole 128-slot ring once p >= 127, a compressed tile is 128
// consecutive rows): such a tile is eight TMA boxes issued by one thread
// instead of 8192 16-byte gathers.
//
// Warps 0-3: softmax and output epilogue (TMEM lanes = rows, then dims);
// warps 4-7: gather loaders (cp.async, zero fill for masked rows) and the query
// rotation; warp 8: MMA issue (one thread) and TMEM allocation. Every wait is
// bounded (tc.cuh); a timeout sets the error word and the CTA winds down.
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "tc.cuh"

namespace ds4a {
namespace {

constexpr int kH = 64, kD = 512, kNope = 448, kRows = 128;
constexpr int kQBlk = kH * 128;        // one 64-dim block of Q: 64 heads x 128 B
// Heads per CTA: decode splits a query's 64 heads over two clusters (every
// rank reads the same rows for half the heads); prefill keeps all 64.
template <bool DEC>
struct Heads {
  static constexpr int NH = DEC ? 32 : 64;   // heads of this CTA
  static constexpr int HG = kH / NH;         // head groups per query
  static constexpr int NHF = NH / 32;        // 32-column halves of the S accumulator
  static constexpr int QBLK = NH * 128;      // one 64-dim block of this CTA's Q
};
constexpr int kKBlk = kRows * 128;     // one 64-dim block of the row tile
constexpr int kThreads = 288;
constexpr uint32_t kMaxCluster = 16;   // cluster size; beyond 8 (the portable limit) when the
                                       // device allows non-portable sizes
constexpr float kRaiseLog2 = 8.0f;     // raise the running max beyond 2^8

struct TcAttnParams {
  uint32_t ratio, batch, T, pos0, cap_raw, comp_cap, n_comp, top_k;
  RowMap map;         // rows of comp
  const uint32_t *seq_pos;   // [B] per-sequence positions (ragged decode) or NULL
  uint32_t cluster;   // decode: CTAs per query (one cluster); 0: prefill, persistent CTAs
  // decode tiles of contiguous rows by TMA instead of row gathers (ratios 0
  // and 128): bit 0 the window tile as the whole 128-slot ring, bit 1 (ratio
  // 128) the compressed tiles (the visible rows, the same count for every
  // sequence)
  uint32_t tma_rows;
  uint32_t n_q;       // queries = batch * T
  float c2;           // softmax scale * log2(e)
  const __nv_bfloat16 *q, *ring, *chunk, *comp;
  const int32_t *topk;
  const float *cos, *sin;
  __nv_bfloat16 *out;
  // decode, C > 1: each rank's O / L as [n_q][C][64][512] bf16, and its
  // (max, sum) per head as [n_q][C][64][2] fp32
  __nv_bfloat16 *part;
  float *ml;
  int *err;
};

struct Smem {
  uint8_t q[8 * kQBlk];     // 64 KiB
  uint8_t kv[8 * kKBlk];    // 128 KiB; decode merge: afterwards the pulled slices (with p)
  uint8_t p[kRows * 128];   // 16 KiB; direct output: afterwards staging, [64 heads][128] bf16
  uint64_t kv_full, kv_empty[4];   // kv_full: the whole tile landed; kv_empty[m]: blocks 2m, 2m+1 free
  uint64_t q_full, q_empty, s_full, p_full, p_empty, o_full, o_empty, sm_bar;
  uint64_t q_tma;   // the query's eight Q blocks landed (TMA transaction count)
  uint64_t kv_tma;  // a tile loaded by TMA landed
  uint64_t mg_bar;  // decode merge: the peers' partial O slices landed
  float mref[kH], alpha[kH], lsh[kH], linv[kH];
  float tmax[4][kH];
  float mw[kH][kMaxCluster];        // decode merge: weight of each rank, per owned head
  uint32_t flagcnt[3], tmem, has_tiles;
};
// the merge pulls at most C * ceil(64 / C) rows of 1 KiB (75 at C = 15)
constexpr uint32_t max_pulled_rows(uint32_t C = 1) {
  return C > kMaxCluster ? 0u
                         : (C * ((kH + C - 1) / C) > max_pulled_rows(C + 1) ? C * ((kH + C - 1) / C)
                                                                             : max_pulled_rows(C + 1));
}
static_assert(8 * kKBlk >= max_pulled_rows() * kD * 2, "pulled slices fit the row buffer");
static_assert(2 * kH * 128 == kRows * 128, "output staging fills the P buffer");

// Rows that a query can have at most, without reading its top-k list.
__device__ __forceinline__ uint32_t rows_bound(const TcAttnParams &P, uint32_t qi) {
  const uint32_t p = seq_base(P.seq_pos, P.pos0, qi / P.T) + qi % P.T;
  uint32_t n = min(p + 1, P.cap_raw);
  if (P.ratio == 4) n += min(P.top_k, min((p + 1) / 4, P.n_comp));
  else if (P.ratio == 128) n += min((p + 1) / 128, P.n_comp);
  return n;
}

// Query-level geometry shared by every role: tiles t0, t0 + ts, ... < t1.
struct QueryGeo {
  uint32_t qi, b, p0, p, n_w, n_list, N, t0, t1, ts;   // p0: the sequence's first chunk position
  const int32_t *tk;
};

// SCAN: read the list for its end (prefill: a chunk query's list may hold
// rows past its visible ones). A decode list holds visible rows, then -1, so
// decode takes the bound min(top_k, visible) and masks the -1 entries row by
// row, with no dependent list read before the first gather.
template <bool SCAN>
__device__ __forceinline__ QueryGeo query_geo(const TcAttnParams &P, uint32_t qi, uint32_t t0,
                                              uint32_t ts, uint32_t lane) {
  QueryGeo g;
  g.qi = qi;
  g.b = qi / P.T;
  g.p0 = seq_base(P.seq_pos, P.pos0, g.b);
  g.p = g.p0 + qi % P.T;
  g.n_w = min(g.p + 1, P.cap_raw);
  g.tk = P.topk ? P.topk + (size_t)qi * P.top_k : nullptr;
  g.n_list = 0;
  if (P.ratio == 4 && !SCAN) {
    g.n_list = min(P.top_k, min((g.p + 1) / 4, P.n_comp));
  } else if (P.ratio == 4) {
    const uint32_t vis = min((g.p + 1) / 4, P.n_comp);
    // the list ends at its first entry >= vis; 16 independent loads per round
    g.n_list = P.top_k;
    for (uint32_t base = 0; base < P.top_k; base += 512) {
      int32_t v[16];
#pragma unroll
      for (uint32_t i = 0; i < 16; ++i) {
        const uint32_t j = base + 32 * i + lane;
        v[i] = j < P.top_k ? g.tk[j] : -1;
      }
      uint32_t found = 0xffffffffu;
#pragma unroll
      for (uint32_t i = 0; i < 16; ++i) {
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
  g.t0 = t0;
  g.t1 = (g.N + kRows - 1) / kRows;
  g.ts = ts;
  return g;
}

// How tile `tile` of a decode query loads: 0 row gathers, 1 the whole ring
// by TMA (the window of 128 rows, in slot order: the softmax does not depend
// on the order of the rows), 2 compressed rows 128 (tile - 1) .. by TMA.
template <bool DEC, bool PAGED>
__device__ __forceinline__ uint32_t tile_kind(const TcAttnParams &P, const QueryGeo &g,
                                              uint32_t tile) {
  if (!DEC || g.n_w != (uint32_t)kRows) return 0;
  if (tile == 0) return (P.tma_rows & 1u) ? 1u : 0u;
  return (!PAGED && (P.tma_rows & 2u) && P.ratio == 128) ? 2u : 0u;
}

// Source row of list entry r (nullptr: masked).
template <bool PAGED>
__device__ __forceinline__ const __nv_bfloat16 *row_src(const TcAttnParams &P, const QueryGeo &g,
                                                        uint32_t r) {
  if (r < g.n_w) {
    const uint32_t pos = g.p - g.n_w + 1 + r;
    if (P.chunk && pos >= g.p0)
      return P.chunk + ((size_t)g.b * P.T + (pos - g.p0)) * kD;
    return P.ring + ((size_t)g.b * P.cap_raw + pos % P.cap_raw) * kD;
  }
  if (r < g.N) {
    const uint32_t j = r - g.n_w;
    const int32_t idx = P.ratio == 4 ? g.tk[j] : (int32_t)j;
    if (idx >= 0) {
      if (PAGED) return P.comp + P.map.row_of(g.b, (uint32_t)idx) * kD;
      return P.comp + ((size_t)g.b * P.comp_cap + (uint32_t)idx) * kD;
    }
  }
  return nullptr;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Decode merge of rank `rank` of a C-CTA cluster (C > 1; threads 0..255):
// heads [64 rank / C, 64 (rank + 1) / C) of every rank's partial O land in the
// row-tile buffer as [j][i][512] fp32 and are combined in rank order with
// weights 2^(m_j - M) / sum_j 2^(m_j - M) l_j. A rank without rows left
// m = -inf and zeros; one with only masked rows left m = -inf and O = 0.
// CM: compile-time bound on the cluster size C (the loops over ranks unroll)
template <uint32_t CM, int NH>
__device__ __forceinline__ bool merge_heads(const TcAttnParams &P, Smem &S, uint32_t vq,
                                            uint32_t rank, uint32_t C, ErrWord ew) {
  const uint32_t t = threadIdx.x, qi = vq / (kH / NH), hq0 = (vq % (kH / NH)) * NH;
  const uint32_t h0 = rank * NH / C, h1 = (rank + 1) * NH / C, nh = h1 - h0;
  const __nv_bfloat16 *part = P.part + (size_t)vq * C * NH * kD;
  const float *ml = P.ml + (size_t)vq * C * NH * 2;
  __nv_bfloat16 *recv = reinterpret_cast<__nv_bfloat16 *>(S.kv);
  // rank j's rows h0 .. h1 - 1 are contiguous: one bulk copy per rank
  if (t == 0) {
    fence_proxy_async_global();
    mbar_arrive_expect_tx(&S.mg_bar, C * nh * kD * 2);
    for (uint32_t j = 0; j < C; ++j)
      bulk_load(recv + (size_t)j * nh * kD, part + ((size_t)j * NH + h0) * kD, nh * kD * 2,
                &S.mg_bar);
  }
  if (t < nh) {
    const uint32_t h = h0 + t;
    float m[CM], l[CM], M = -INFINITY;
#pragma unroll
    for (uint32_t j = 0; j < CM; ++j) {
      m[j] = j < C ? __ldcg(ml + ((size_t)j * NH + h) * 2) : -INFINITY;   // written by peers
      l[j] = j < C ? __ldcg(ml + ((size_t)j * NH + h) * 2 + 1) : 0.f;
    }
#pragma unroll
    for (uint32_t j = 0; j < CM; ++j) M = fmaxf(M, m[j]);
    // O = sum_j f_j (O_j / L_j) with f_j = 2^(m_j - M) L_j / sum_i 2^(m_i - M) L_i
    float f[CM], L = 0.f;
#pragma unroll
    for (uint32_t j = 0; j < CM; ++j) {
      f[j] = m[j] == -INFINITY ? 0.f : exp2f(m[j] - M) * l[j];
      L += f[j];
    }
    const float li = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (uint32_t j = 0; j < CM; ++j) S.mw[t][j] = f[j] * li;
  }
  // rotation coefficients load while the slices land
  const uint32_t p = seq_base(P.seq_pos, P.pos0, qi / P.T) + qi % P.T, c = t & 127, d = 4 * c;
  float co0 = 1.f, si0 = 0.f, co1 = 1.f, si1 = 0.f;
  if (d >= (uint32_t)kNope) {
    const uint32_t fi = (d - kNope) >> 1;
    co0 = P.cos[(size_t)p * 32 + fi];
    si0 = P.sin[(size_t)p * 32 + fi];
    co1 = P.cos[(size_t)p * 32 + fi + 1];
    si1 = P.sin[(size_t)p * 32 + fi + 1];
  }
  const bool ok = mbar_wait(&S.mg_bar, 0, ew);
  named_bar_sync(1, 256);
  if (!ok) return false;
#pragma unroll 1
  for (uint32_t i = t >> 7; i < nh; i += 2) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (uint32_t j = 0; j < CM; ++j) {
      const float f = S.mw[i][j];
      if (j < C && f != 0.f) {
        const uint2 v = *reinterpret_cast<const uint2 *>(recv + (j * nh + i) * kD + d);
        a0 = fmaf(f, bf16lo(v.x), a0);
        a1 = fmaf(f, bf16hi(v.x), a1);
        a2 = fmaf(f, bf16lo(v.y), a2);
        a3 = fmaf(f, bf16hi(v.y), a3);
      }
    }
    // rotate back by -p: (x0, x1) -> (x0 c + x1 s, -x0 s + x1 c)
    const float r0 = a0 * co0 + a1 * si0, r1 = -a0 * si0 + a1 * co0;
    const float r2 = a2 * co1 + a3 * si1, r3 = -a2 * si1 + a3 * co1;
    *reinterpret_cast<uint2 *>(P.out + ((size_t)qi * kH + hq0 + h0 + i) * kD + d) =
        make_uint2(pack_bf16(r0, r1), pack_bf16(r2, r3));
  }
  return true;
}

// DEC: decode (clusters of P.cluster CTAs per query) or prefill (persistent
// CTAs); two instantiations keep each path's code to itself
template <bool DEC, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_ring,
                   const __grid_constant__ CUtensorMap tmap_comp, TcAttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned. Prefill takes an offset from the shared array itself,
  // so its accesses to S compile to shared-memory instructions (chunk
  // attention 795 -> 750 us); decode keeps the integer round trip and generic
  // accesses, which measured faster for its c4a and c128a calls (14.5 / 16.7
  // against 14.8 / 17.0 us)
  uint8_t *sbase;
  if (DEC)
    sbase = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~(uintptr_t)1023);
  else
    sbase = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem &S = *reinterpret_cast<Smem *>(sbase);
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // decode: cluster of C CTAs per (query, head group), rank c takes tiles
  // c, c + C, ...; prefill: one whole query at a time per CTA
  constexpr bool dec = DEC;
  using HS = Heads<DEC>;
  constexpr int NH = HS::NH, NHF = HS::NHF, QBLK = HS::QBLK;
  const uint32_t C = dec ? P.cluster : 1u;
  const uint32_t rank = dec ? cluster_ctarank() : 0u;
  const uint32_t vq = dec ? blockIdx.x / C : 0u;          // decode: (query, head group)
  const uint32_t hq0 = dec ? (vq % HS::HG) * NH : 0u;     // first head of this CTA
  const uint32_t q_first = dec ? vq / HS::HG : blockIdx.x;
  const uint32_t q_step = dec ? P.n_q : gridDim.x;
  const int err_base = *(volatile int *)P.err;
  if (NH < kH) {
    // heads NH .. 63 of every P row stay zero: the PV and sum MMAs read all
    // 64 columns, and those of the other group contribute nothing
    uint4 *pz = reinterpret_cast<uint4 *>(S.p);
    for (uint32_t i = threadIdx.x; i < kRows * 128 / 16; i += blockDim.x)
      pz[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
  }

  if (threadIdx.x == 0) {
    mbar_init(&S.kv_full, 128);
    for (int i = 0; i < 4; ++i) mbar_init(&S.kv_empty[i], 1);
    mbar_init(&S.q_full, 128);
    mbar_init(&S.q_empty, 1);
    mbar_init(&S.s_full, 1);
    mbar_init(&S.p_full, 128);
    mbar_init(&S.p_empty, 1);
    mbar_init(&S.o_full, 1);
    mbar_init(&S.o_empty, 4);
    mbar_init(&S.sm_bar, 128);
    mbar_init(&S.q_tma, 1);
    mbar_init(&S.kv_tma, 1);
    mbar_init(&S.mg_bar, 1);
    S.flagcnt[0] = S.flagcnt[1] = S.flagcnt[2] = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_q);
    if (P.tma_rows) {
      prefetch_tmap(&tmap_ring);
      prefetch_tmap(&tmap_comp);
    }
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
  // the loaders wait for the previous launch themselves, after they have
  // started the first query's Q load
  const bool loader = warp >= 4 && warp < 8;
  if (!loader) {
    pdl_wait();
    pdl_trigger();
  }
  // this launch's view of the error word (see ErrWord), read before the wait
  // so that its latency overlaps the previous launch
  const ErrWord ew{P.err, err_base};

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ loaders
    const uint32_t lt = threadIdx.x - 128, lw = warp - 4;
    uint32_t n = 0, qn = 0, qt = 0, nk = 0;   // qt: Q loads issued, nk: TMA tiles issued
    // issue all eight 64-dim blocks of a tile (one cp.async group each) as
    // their slots free up; rows of this lane: lw*32 + lane/8 + 4i, chunk lane%8.
    // A tile of contiguous rows is eight TMA boxes of 128 rows x 64 dims
    // (one thread), in the same swizzled layout.
    auto issue_tile = [&](const QueryGeo &g, uint32_t tile, uint32_t n) -> bool {
      if (const uint32_t kind = tile_kind<DEC, PAGED>(P, g, tile)) {
        for (uint32_t kb = 0; kb < 8; ++kb) {
          if ((kb & 1) == 0 && !mbar_wait_warp(&S.kv_empty[kb >> 1], (n & 1) ^ 1, ew)) return false;
          if (lt == 0) {
            if (kb == 0) mbar_arrive_expect_tx(&S.kv_tma, 8 * kKBlk);
            if (kind == 1)
              tma_load_3d(S.kv + kb * kKBlk, &tmap_ring, &S.kv_tma, (int)(64 * kb), 0, (int)g.b);
            else
              tma_load_3d(S.kv + kb * kKBlk, &tmap_comp, &S.kv_tma, (int)(64 * kb),
                          (int)(kRows * (tile - 1)), (int)g.b);
          }
        }
        return true;
      }
      const __nv_bfloat16 *src[8];
#pragma unroll
      for (uint32_t i = 0; i < 8; ++i)
        src[i] = row_src<PAGED>(P, g, tile * kRows + lw * 32 + (lane >> 3) + 4 * i);
      const uint32_t cc = lane & 7;
      for (uint32_t kb = 0; kb < 8; ++kb) {
        if ((kb & 1) == 0 && !mbar_wait_warp(&S.kv_empty[kb >> 1], (n & 1) ^ 1, ew)) return false;
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
    // Q (it needs no list): eight TMA boxes of 64 heads x 64 dims, in the
    // 128-byte swizzled K-major layout the S MMAs read. The first query's
    // is issued before the wait for the previous launch: the queries are the
    // caller's input, written before that launch began (as are the rotation
    // tables), while the top-k lists and the new raw row are not.
    auto issue_q = [&](uint32_t qi) {
      if (lt == 0) {
        mbar_arrive_expect_tx(&S.q_tma, 8 * QBLK);
#pragma unroll
        for (uint32_t kb = 0; kb < 8; ++kb)
          tma_load_2d(S.q + kb * QBLK, &tmap_q, &S.q_tma, (int)(64 * kb), (int)(qi * kH + hq0));
      }
    };
    const bool q_early = q_first < P.n_q && rank * kRows < rows_bound(P, q_first);
    if (q_early) issue_q(q_first);
    // The loaders' own wait for the previous launch. Decode reads nothing of
    // it before the first rows (the rotation coefficients are inputs and a
    // decode list is not scanned), so its first query's coefficients and
    // geometry are prepared before the wait; prefill scans its lists, so it
    // waits here.
    bool waited = false;
    auto wait_prev = [&]() {
      if (!waited) {
        pdl_wait();
        pdl_trigger();
        waited = true;
      }
    };
    if (!DEC) wait_prev();
    for (uint32_t qi = q_first; qi < P.n_q; qi += q_step) {
      if (rank * kRows >= rows_bound(P, qi)) continue;   // no rows for this rank
      if (!mbar_wait_warp(&S.q_empty, (qn & 1) ^ 1, ew)) goto done_loader;
      if (!(q_early && qi == q_first)) issue_q(qi);
      {
        // this thread's 16-byte chunks of the tail: chunk lt (+ 128 i) of
        // block 7 hold pairs 4 lc .. 4 lc + 3 of head id / 8; their
        // coefficients load while the list is read
        const uint32_t pq = seq_base(P.seq_pos, P.pos0, qi / P.T) + qi % P.T;
        constexpr uint32_t kQC = NH / 16;   // tail chunks per loader thread
        float co[4 * kQC], si[4 * kQC];
#pragma unroll
        for (uint32_t i = 0; i < kQC; ++i) {
          const uint32_t id = lt + 128 * i, h = id >> 3, lc = (id & 7) ^ (h & 7);
#pragma unroll
          for (uint32_t e = 0; e < 4; ++e) {
            co[4 * i + e] = P.cos[(size_t)pq * 32 + 4 * lc + e];
            si[4 * i + e] = P.sin[(size_t)pq * 32 + 4 * lc + e];
          }
        }
        const QueryGeo g = query_geo<!DEC>(P, qi, rank, C, lane);
        if (g.t0 >= g.t1) {          // the list is shorter than the bound: nothing to do
          // (Q still lands: wait for it so the buffer is never written twice at once)
          if (!mbar_wait_warp(&S.q_tma, qt & 1, ew)) goto done_loader;
          ++qt;
          continue;
        }
        // the first tile's rows start loading before Q is rotated
        wait_prev();
        if (!issue_tile(g, g.t0, n)) goto done_loader;
        if (!mbar_wait_warp(&S.q_tma, qt & 1, ew)) goto done_loader;   // Q landed
        ++qt;
        // rotate the tail (dims 448..511 = block 7) at position p, in place
#pragma unroll
        for (uint32_t i = 0; i < kQC; ++i) {
          const uint32_t id = lt + 128 * i, h = id >> 3, pc = id & 7;
          uint4 *ptr = reinterpret_cast<uint4 *>(S.q + 7 * QBLK + h * 128 + pc * 16);
          uint4 v = *ptr;
          uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (uint32_t e = 0; e < 4; ++e) {
            const float c = co[4 * i + e], sn = si[4 * i + e];
            const float x0 = bf16lo(w4[e]), x1 = bf16hi(w4[e]);
            w4[e] = pack_bf16(x0 * c - x1 * sn, x0 * sn + x1 * c);
          }
          *ptr = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        fence_proxy_async();
        mbar_arrive(&S.q_full);
        for (uint32_t tile = g.t0; tile < g.t1; tile += g.ts, ++n) {
          if (tile != g.t0 && !issue_tile(g, tile, n)) goto done_loader;
          // one arrival per thread once all its rows of the tile landed: the
          // MMA issuer takes the tile whole (waits between the MMAs of one
          // accumulation halve their rate; issuing S pair by pair as the
          // blocks land measured slower)
          cp_async_wait_all();
          fence_proxy_async();
          if (tile_kind<DEC, PAGED>(P, g, tile)) {   // (one thread watches the TMA tile)
            if (lt == 0 && !mbar_wait(&S.kv_tma, nk & 1, ew)) goto done_loader;
            ++nk;
          }
          mbar_arrive(&S.kv_full);
        }
      }
      ++qn;
    }
  done_loader:
    cp_async_wait_all();
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idS = idesc_bf16_f32(kRows, NH);
    constexpr uint32_t idPV = idesc_bf16_f32(kRows, kH) | kIdescMajorA_MN | kIdescMajorB_MN;
    const uint32_t q_base = smem_u32(S.q), kv_base = smem_u32(S.kv), p_base = smem_u32(S.p);
    uint32_t n = 0, qn = 0, nk = 0;
    bool ok = true;
    for (uint32_t qi = q_first; qi < P.n_q && ok; qi += q_step) {
      if (rank * kRows >= rows_bound(P, qi)) continue;
      const QueryGeo g = query_geo<!DEC>(P, qi, rank, C, lane);
      if (g.t0 >= g.t1) continue;
      if (lane == 0) {
        ok = mbar_wait(&S.q_full, qn & 1, ew);
        for (uint32_t tile = g.t0; ok && tile < g.t1; tile += g.ts, ++n) {
          const bool first = tile == g.t0, last = tile + g.ts >= g.t1;
          ok = mbar_wait(&S.kv_full, n & 1, ew);
          if (ok && tile_kind<DEC, PAGED>(P, g, tile)) ok = mbar_wait(&S.kv_tma, nk++ & 1, ew);
          if (!ok) break;
          tc_fence_after();
          for (uint32_t kb = 0; kb < 8; ++kb)
#pragma unroll
            for (uint32_t kk = 0; kk < 4; ++kk)
              mma_bf16(tmS, sdesc_sw128(kv_base + kb * kKBlk + kk * 32),
                       sdesc_sw128(q_base + kb * QBLK + kk * 32), idS, (kb | kk) ? 1u : 0u);
          mma_commit(&S.s_full);
          if (last) mma_commit(&S.q_empty);
          ok = mbar_wait(&S.p_full, n & 1, ew);
          if (ok && first) ok = mbar_wait(&S.o_empty, (qn & 1) ^ 1, ew);
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
            mma_commit(&S.kv_empty[m]);
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
    // P of heads 32 hf .. + 31 of row r from their scores `a` with the current
    // running maxima; flags a score above its head's maximum by more than 2^8
    auto p_half = [&](bool valid, const uint32_t (&a)[32], uint32_t hf, bool &flag) {
      uint8_t *prow = S.p + (r >> 3) * 1024 + (r & 7) * 128;
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
    };
    // P row r from the scores in TMEM; returns whether a score exceeds its
    // head's running maximum by more than 2^8
    auto write_p = [&](bool valid) {
      bool flag = false;
#pragma unroll
      for (uint32_t hf = 0; hf < (uint32_t)NHF; ++hf) {
        uint32_t a[32];
        tmem_ld32(tmS + lane_base + 32 * hf, a);
        tmem_ld_wait();
        p_half(valid, a, hf, flag);
      }
      return flag;
    };
    for (uint32_t qi = q_first; qi < P.n_q; qi += q_step) {
      const bool maybe = rank * kRows < rows_bound(P, qi);
      QueryGeo g = {};
      if (maybe) g = query_geo<!DEC>(P, qi, rank, C, lane);
      const bool has_tiles = maybe && g.t0 < g.t1;
      bool any_valid = false;
      // the rotation coefficients of this thread's tail dim in the direct
      // output (dim 384 + r of the last chunk), loaded while the tiles run
      float ep_co = 1.f, ep_si = 0.f;
      if (!(dec && C > 1) && has_tiles && 384 + r >= (uint32_t)kNope) {
        const uint32_t fi = (384 + r - kNope) >> 1;
        ep_co = P.cos[(size_t)g.p * 32 + fi];
        ep_si = P.sin[(size_t)g.p * 32 + fi];
      }
      for (uint32_t tile = g.t0; has_tiles && tile < g.t1; tile += g.ts, ++n) {
        const bool first = tile == g.t0;
        const uint32_t row = tile * kRows + r;
        bool valid = row < g.n_w;
        if (!valid && row < g.N) valid = P.ratio != 4 || g.tk[row - g.n_w] >= 0;
        if (!mbar_wait_warp(&S.s_full, n & 1, ew)) goto done_softmax;
        tc_fence_after();
        if (first) {
          // running maxima start at the exact per-head maxima of the first
          // tile's scaled scores: warp maxima of order-keyed values, then the
          // largest of the four warps. P of this tile then has no score above
          // its maximum (no raise to check).
          uint32_t *tkey = reinterpret_cast<uint32_t *>(&S.tmax[0][0]);   // [4][kH]
          // eight heads per step of a short loop: this runs once per query,
          // its code is fetched cold, and an unrolled form measured ~2 us of
          // instruction fetch
#pragma unroll 1
          for (uint32_t c = 0; c < (uint32_t)NH; c += 8) {
            uint32_t a8[8];
            tmem_ld8(tmS + lane_base + c, a8);
            tmem_ld_wait();
#pragma unroll
            for (uint32_t j = 0; j < 8; ++j) {
              const uint32_t u = __float_as_uint(__uint_as_float(a8[j]) * P.c2);
              const uint32_t key = valid ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
              const uint32_t mk = redux_max_u32(key);
              if (lane == ((c + j) & 31)) tkey[warp * kH + c + j] = mk;
            }
          }
          if (r == 0) S.flagcnt[(n + 1) % 3] = 0;   // the next tile's raise count
          if (!group_sync(&S.sm_bar, sm_phase, ew)) goto done_softmax;
          const uint32_t k0 = max(max(tkey[0 * kH], tkey[1 * kH]), max(tkey[2 * kH], tkey[3 * kH]));
          any_valid = k0 != 0u;   // a valid row has a key above 0 for every head
          if (r < (uint32_t)NH) {
            const uint32_t mk = max(max(tkey[0 * kH + r], tkey[1 * kH + r]),
                                    max(tkey[2 * kH + r], tkey[3 * kH + r]));
            const float mx = __uint_as_float((mk & 0x80000000u) ? (mk & 0x7fffffffu) : ~mk);
            S.mref[r] = any_valid ? mx : 0.f;
          }
          if (!group_sync(&S.sm_bar, sm_phase, ew)) goto done_softmax;
          if (!mbar_wait_warp(&S.p_empty, (n & 1) ^ 1, ew)) goto done_softmax;
          // the scores (S stays until this tile's P is done)
          bool unused = false;
          if (NHF == 2) {
            uint32_t a0[32], a1[32];
            tmem_ld32(tmS + lane_base, a0);
            tmem_ld32(tmS + lane_base + 32, a1);
            tmem_ld_wait();
            p_half(valid, a0, 0, unused);
            p_half(valid, a1, 1, unused);
          } else {
            uint32_t a0[32];
            tmem_ld32(tmS + lane_base, a0);
            tmem_ld_wait();
            p_half(valid, a0, 0, unused);
          }
          fence_proxy_async();
          tc_fence_before();
          mbar_arrive(&S.p_full);
          continue;
        }
        // P of this tile (the previous PV must be done with the buffer)
        if (!mbar_wait_warp(&S.p_empty, (n & 1) ^ 1, ew)) goto done_softmax;
        const bool flag = write_p(valid);
        const uint32_t fc = n % 3;
        if (r == 0) S.flagcnt[(n + 1) % 3] = 0;
        if (flag) atomicAdd(&S.flagcnt[fc], 1u);
        if (!group_sync(&S.sm_bar, sm_phase, ew)) goto done_softmax;
        if (S.flagcnt[fc] != 0) {
          // rare path: exact tile max per head, raise the running max, rescale
          // O and L, rewrite P
#pragma unroll 1
          for (uint32_t hf = 0; hf < (uint32_t)NHF; ++hf) {
            uint32_t a[32];
            tmem_ld32(tmS + lane_base + 32 * hf, a);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; ++h) {
              const float v = warp_max(valid ? __uint_as_float(a[h]) * P.c2 : -INFINITY);
              if (lane == (uint32_t)h) S.tmax[warp][32 * hf + h] = v;
            }
          }
          if (!group_sync(&S.sm_bar, sm_phase, ew)) goto done_softmax;
          if (r < (uint32_t)NH) {
            const float M = fmaxf(fmaxf(S.tmax[0][r], S.tmax[1][r]), fmaxf(S.tmax[2][r], S.tmax[3][r]));
            const float mo = S.mref[r], mn = fmaxf(mo, M);
            S.alpha[r] = exp2f(mo - mn);
            S.mref[r] = mn;
          }
          if (!group_sync(&S.sm_bar, sm_phase, ew)) goto done_softmax;
          if (!first) {
#pragma unroll 1
            for (uint32_t m = 0; m < 5 * (uint32_t)NHF; ++m) {   // O^T (4 dim blocks) then L
              uint32_t a[32];
              const uint32_t blk = m / NHF, hf = m % NHF;
              const uint32_t ta = (blk < 4 ? tmO + blk * kH : tmL) + 32 * hf + lane_base;
              tmem_ld32(ta, a);
              tmem_ld_wait();
#pragma unroll
              for (int h = 0; h < 32; ++h)
                a[h] = __float_as_uint(__uint_as_float(a[h]) * S.alpha[32 * hf + h]);
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
      // ---- query end: per-head sums (any lane of L), then the output
      if (has_tiles) {
        if (!mbar_wait_warp(&S.o_full, qn & 1, ew)) goto done_softmax;
        tc_fence_after();
        if (warp < (uint32_t)NHF) {   // every row of L holds the sums: warp w keeps heads 32w + lane
          uint32_t a[32];
          tmem_ld32(tmL + lane_base + 32 * warp, a);
          tmem_ld_wait();
          float l = 0.f;
#pragma unroll
          for (uint32_t i = 0; i < 32; ++i)
            if (lane == i) l = __uint_as_float(a[i]);
          S.lsh[32 * warp + lane] = l;
          S.linv[32 * warp + lane] = l > 0.f ? 1.f / l : 0.f;
        }
      }
      if (!group_sync(&S.sm_bar, sm_phase, ew)) goto done_softmax;
      if (dec && C > 1) {
        // (max, sum) of this rank for the cluster merge; O follows from TMEM
        if (r < (uint32_t)NH) {
          float *ml = P.ml + ((size_t)(vq * C + rank) * NH + r) * 2;
          ml[0] = (has_tiles && any_valid) ? S.mref[r] : -INFINITY;
          ml[1] = has_tiles ? S.lsh[r] : 0.f;
        }
        if (r == 0) S.has_tiles = has_tiles ? 1u : 0u;
      } else {
        // normalise, rotate the tail back by -p and store bf16 pairs straight
        // from registers, four 128-dim chunks (no staging, no barrier)
        float li[NH];   // 1 / L per head, for the four chunks
#pragma unroll
        for (int h = 0; h < NH; ++h) li[h] = S.linv[h];
        const bool odd = lane & 1;
#pragma unroll 1
        for (uint32_t m = 0; m < 4; ++m) {
          const bool rot = m == 3 && r >= 64;   // warp-uniform: the rotated tail dims
          const float co = ep_co, si = ep_si;   // (the pair's coefficients: both lanes)
          __nv_bfloat16 *o = P.out + ((size_t)qi * kH + hq0) * kD + m * 128;
          uint32_t ab[NHF][32];
#pragma unroll
          for (uint32_t hf = 0; hf < (uint32_t)NHF; ++hf)
            tmem_ld32(tmO + lane_base + m * kH + 32 * hf, ab[hf]);
          tmem_ld_wait();
#pragma unroll
          for (uint32_t hf = 0; hf < (uint32_t)NHF; ++hf) {
#pragma unroll
            for (int h = 0; h < 32; h += 2) {
              const float v0 = __uint_as_float(ab[hf][h]) * li[32 * hf + h];
              const float v1 = __uint_as_float(ab[hf][h + 1]) * li[32 * hf + h + 1];
              // lanes 2i, 2i + 1 hold dims d, d + 1 of heads h, h + 1: one
              // swap gives the even lane head h's pair and the odd lane head
              // h + 1's, rotated in place and stored as one bf16 pair
              const float recv = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
              float x0 = odd ? recv : v0, x1 = odd ? v1 : recv;
              if (rot) {   // (x0, x1) -> (x0 c + x1 s, -x0 s + x1 c)
                const float y0 = x0 * co + x1 * si, y1 = -x0 * si + x1 * co;
                x0 = y0;
                x1 = y1;
              }
              const uint32_t row = 32 * hf + h + (odd ? 1u : 0u);
              *reinterpret_cast<uint32_t *>(o + (size_t)row * kD + (r & ~1u)) = pack_bf16(x0, x1);
            }
          }
        }
      }
      if (has_tiles) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.o_empty);
        ++qn;
      }
      // keep the shared sums alive until every thread has read them
      if (!group_sync(&S.sm_bar, sm_phase, ew)) goto done_softmax;
    }
  done_softmax:;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (dec && C > 1) {
    // this rank's O / L as [NH heads][512] bf16 straight to the workspace.
    // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (dims) for heads 32 hf ..
    // + 31 of dim blocks m0 .. m1 - 1 (64 heads: hf = w / 4, every block; 32
    // heads: hf = 0, two blocks per warp); lanes 2i, 2i + 1 hold dims d, d + 1:
    // the even lane stores the bf16 pair of head h, the odd lane that of head
    // h + 1 (one swap each)
    if (warp < 8) {
      __nv_bfloat16 *dst = P.part + ((size_t)vq * C + rank) * NH * kD;
      const uint32_t qw = warp & 3, hf = NHF == 2 ? warp >> 2 : 0u, dl = 32 * qw + lane;
      const uint32_t m0 = NHF == 2 ? 0u : 2 * (warp >> 2), m1 = NHF == 2 ? 4u : m0 + 2;
      const bool had = S.has_tiles != 0, odd = lane & 1;
      float li[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) li[h] = had ? S.linv[32 * hf + h] : 0.f;
#pragma unroll 1
      for (uint32_t m = m0; m < m1; ++m) {
        uint32_t a[32];
        if (had) {
          tmem_ld32(tmO + ((32 * qw) << 16) + m * kH + 32 * hf, a);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) a[h] = 0u;
        }
#pragma unroll
        for (int h = 0; h < 32; h += 2) {
          const float v0 = __uint_as_float(a[h]) * li[h], v1 = __uint_as_float(a[h + 1]) * li[h + 1];
          const float other = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
          const uint32_t row = 32 * hf + h + (odd ? 1 : 0);
          const uint32_t w = odd ? pack_bf16(other, v1) : pack_bf16(v0, other);
          *reinterpret_cast<uint32_t *>(dst + (size_t)row * kD + m * 128 + (dl & ~1u)) = w;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) tmem_dealloc(tmem, 512);
  if (dec && C > 1) {
    cluster_sync_all();   // every rank's O and (max, sum) are in the workspace
    if (warp < 8) {
      if (C <= 8)
        merge_heads<8, NH>(P, S, vq, rank, C, ew);
      else
        merge_heads<kMaxCluster, NH>(P, S, vq, rank, C, ew);
    }
  }
}

// Largest number of clusters of each size (1..16) that fit on the device at
// once, per device; 0 = not yet asked, -1 = the size cannot be launched.
std::atomic<int> g_max_clusters[64][kMaxCluster + 1];
// Per device: 1 = cluster sizes above 8 allowed for the kernel, -1 = refused.
std::atomic<int> g_nonportable[64];

int max_active_clusters(uint32_t C, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int v = g_max_clusters[dev][C].load(std::memory_order_relaxed);
  if (v != 0) return v;
  if (C > 8) {
    int np = g_nonportable[dev].load(std::memory_order_relaxed);
    if (np == 0) {
      np = cudaFuncSetAttribute(attn_tc_kernel<true, false>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
                   cudaFuncSetAttribute(attn_tc_kernel<true, true>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess
               ? 1
               : -1;
      (void)cudaGetLastError();
      g_nonportable[dev].store(np, std::memory_order_relaxed);
    }
    if (np < 0) {
      g_max_clusters[dev][C].store(-1, std::memory_order_relaxed);
      return -1;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(C * 64);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&v, attn_tc_kernel<true, false>, &cfg) != cudaSuccess || v <= 0) {
    (void)cudaGetLastError();
    // beyond the portable size an unanswered query means the size is not used
    v = C > 8 ? -1 : num_sms() / (int)C;
  }
  if (v == 0) v = 1;
  g_max_clusters[dev][C].store(v, std::memory_order_relaxed);
  return v;
}

// Cluster size for a decode batch: fewest rounds of tiles, counting a whole
// extra round for every wave of clusters beyond the first (a wave also pays
// the query load and the merge, modelled as two tiles). Ties: fewer CTAs.
uint32_t pick_cluster(uint32_t n_tiles, uint32_t n_q, size_t smem) {
  uint32_t best = 1, best_cost = 0xffffffffu;
  const uint32_t cmax = n_tiles < kMaxCluster ? (n_tiles ? n_tiles : 1u) : kMaxCluster;
  for (uint32_t C = 1; C <= cmax; ++C) {
    const int actv = max_active_clusters(C, smem);
    if (actv < 1) continue;
    const uint32_t act = (uint32_t)actv;
    const uint32_t waves = (n_q + act - 1) / act, tiles = (n_tiles + C - 1) / C;
    const uint32_t cost = waves * (tiles + 2);
    if (cost < best_cost) {
      best = C;
      best_cost = cost;
    }
  }
  return best;
}

// Process-wide cluster size forced by ds4a_set_decode_cluster (0: automatic).
std::atomic<uint32_t> g_force_cluster{0};

// The cluster size a decode launch uses: the forced size (clamped to the
// query's tile count and 16) when the device can launch it, else pick_cluster.
uint32_t decode_cluster(uint32_t rows_max, uint32_t n_q, size_t smem) {
  const uint32_t n_tiles = (rows_max + kRows - 1) / kRows;
  const uint32_t cmax = n_tiles < kMaxCluster ? (n_tiles ? n_tiles : 1u) : kMaxCluster;
  uint32_t f = g_force_cluster.load(std::memory_order_relaxed);
  if (f) {
    if (f > cmax) f = cmax;
    if (max_active_clusters(f, smem) >= 1) return f;
  }
  return pick_cluster(n_tiles, n_q, smem);
}

}  // namespace

void attn_tc_force_cluster(uint32_t C) {
  g_force_cluster.store(C > kMaxCluster ? kMaxCluster : C, std::memory_order_relaxed);
}

uint32_t attn_tc_decode_cluster(uint32_t rows_max, uint32_t n_q) {
  return decode_cluster(rows_max, n_q * Heads<true>::HG, sizeof(Smem) + 1024);
}

bool attn_tc_supported(int dtype, uint32_t H, uint32_t D, uint32_t n_rot) {
  return dtype == DS4A_BF16 && H == (uint32_t)kH && D == (uint32_t)kD && n_rot == 64;
}

// Error word, then (decode) room for the partials of the largest cluster.
size_t attn_tc_ws_bytes(uint32_t batch, uint32_t T, uint32_t rows_max) {
  if (T != 1) return 256;
  const uint32_t n_tiles = (rows_max + kRows - 1) / kRows;
  const uint32_t cmax = n_tiles < kMaxCluster ? (n_tiles ? n_tiles : 1u) : kMaxCluster;
  if (cmax < 2) return 256;
  return 256 + (size_t)batch * cmax * kH * (kD * sizeof(__nv_bfloat16) + 2 * sizeof(float));
}

cudaError_t launch_attention_tc(const AttnArgs &a, uint32_t rows_max, int *err, cudaStream_t s) {
  TcAttnParams P;
  P.ratio = a.ratio;
  P.batch = a.batch;
  P.T = a.T;
  P.pos0 = a.pos0;
  P.cap_raw = a.cap_raw;
  P.comp_cap = a.comp_cap;
  P.map = a.map;
  P.seq_pos = a.seq_pos;
  P.n_comp = a.n_comp;
  P.top_k = a.top_k;
  P.n_q = a.batch * a.T;
  P.c2 = a.scale * 1.4426950408889634f;
  P.q = static_cast<const __nv_bfloat16 *>(a.q);
  P.ring = static_cast<const __nv_bfloat16 *>(a.ring);
  P.chunk = static_cast<const __nv_bfloat16 *>(a.chunk);
  P.comp = static_cast<const __nv_bfloat16 *>(a.comp);
  P.topk = a.topk;
  P.cos = a.cos;
  P.sin = a.sin;
  P.out = static_cast<__nv_bfloat16 *>(a.out);
  P.part = reinterpret_cast<__nv_bfloat16 *>(static_cast<uint8_t *>(a.ws) + 256);
  P.ml = nullptr;
  P.err = err;
  const size_t smem = sizeof(Smem) + 1024;
  // paged rows: an instantiation of its own, so the contiguous gathers carry
  // no table code
  const bool paged = a.map.table != nullptr;
  auto *k_dec = paged ? attn_tc_kernel<true, true> : attn_tc_kernel<true, false>;
  auto *k_pf = paged ? attn_tc_kernel<false, true> : attn_tc_kernel<false, false>;
  static int smem_set[2][2] = {{0, 0}, {0, 0}};
  cudaError_t e = a.T == 1 ? ensure_smem(k_dec, smem, &smem_set[1][paged])
                           : ensure_smem(k_pf, smem, &smem_set[0][paged]);
  if (e != cudaSuccess) return e;
  // Q as [n_q * 64 heads][512] bf16 rows; boxes of one CTA's heads x 64 dims
  CUtensorMap tq;
  const uint64_t qd[2] = {(uint64_t)kD, (uint64_t)P.n_q * kH};
  const uint64_t qs[1] = {(uint64_t)kD * 2};
  const uint32_t qb[2] = {64, (uint32_t)(a.T == 1 ? Heads<true>::NH : Heads<false>::NH)};
  e = make_tmap_bf16(&tq, a.q, 2, qd, qs, qb);
  if (e != cudaSuccess) return e;
  // decode tiles of contiguous rows: the ring [B][128][512] (one box of its
  // 128 slots per 64 dims) and, on ratio 128 with one position for every
  // sequence, the visible compressed rows [B][n_list][512] (rows past n_list
  // read as zeros); a map that cannot be built leaves the gathers
  CUtensorMap tr = tq, tcmp = tq;
  P.tma_rows = 0;
  // (ratio 4 keeps its window on the gathers: its first rank runs the window
  // tile beside the list tiles, and by TMA it measured slower)
  if (a.T == 1 && a.cap_raw == (uint32_t)kRows && a.ratio != 4) {
    const uint64_t rd[3] = {(uint64_t)kD, (uint64_t)a.cap_raw, (uint64_t)a.batch};
    const uint64_t rs[2] = {(uint64_t)kD * 2, (uint64_t)a.cap_raw * kD * 2};
    const uint32_t rb[3] = {64, (uint32_t)kRows, 1};
    if (make_tmap_bf16(&tr, a.ring, 3, rd, rs, rb) == cudaSuccess) P.tma_rows |= 1u;
    const uint32_t n_list = a.ratio == 128 ? min((a.pos0 + 1) / 128, a.n_comp) : 0u;
    if (a.ratio == 128 && !paged && !a.seq_pos && n_list >= (uint32_t)kRows) {
      const uint64_t cd[3] = {(uint64_t)kD, (uint64_t)n_list, (uint64_t)a.batch};
      const uint64_t cs[2] = {(uint64_t)kD * 2, (uint64_t)a.comp_cap * kD * 2};
      if (make_tmap_bf16(&tcmp, a.comp, 3, cd, cs, rb) == cudaSuccess) P.tma_rows |= 2u;
    }
  }
  if (a.T == 1) {
    // one cluster of P.cluster CTAs per (query, head group)
    const uint32_t n_vq = P.n_q * Heads<true>::HG;
    P.cluster = decode_cluster(rows_max, n_vq, smem);
    P.ml = reinterpret_cast<float *>(P.part + (size_t)P.n_q * P.cluster * kH * kD);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = P.cluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(n_vq * P.cluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, k_dec, tq, tr, tcmp, P);
    note_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  P.cluster = 0;
  const uint32_t grid = min(P.n_q, (uint32_t)num_sms());
  e = launch_pdl(k_pf, dim3(grid), dim3(kThreads), smem, s, tq, tr, tcmp, P);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ds4a
