// C ABI of libds4a: argument checks, position bookkeeping and kernel dispatch.
// Every check happens on the host before the first launch of a call; a failed
// check launches nothing.
#include <atomic>
#include <cmath>
#include <cstring>

#include "internal.h"

using namespace ds4a;

namespace ds4a {
static std::atomic<uint64_t> g_launches{0};
static std::atomic<int> g_last_error{0};
void note_launches(uint32_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
cudaError_t note_error(cudaError_t e) {
  if (e != cudaSuccess) g_last_error.store((int)e, std::memory_order_relaxed);
  return e;
}
}  // namespace ds4a

namespace {

uint32_t window_of(uint32_t ratio) { return ratio == 4 ? 8u : ratio == 128 ? 128u : 0u; }

ds4a_status check_cache(const ds4a_layer_cache *c) {
  if (!c) return DS4A_ERR_ARG;
  if (c->dtype != DS4A_F32 && c->dtype != DS4A_BF16) return DS4A_ERR_DTYPE;
  if (c->ratio != 0 && c->ratio != 4 && c->ratio != 128) return DS4A_ERR_ARG;
  if (c->batch == 0 || c->head_dim == 0 || c->head_dim > 1024 || c->head_dim % 4) return DS4A_ERR_SHAPE;
  if (c->n_rot > c->head_dim || c->n_rot % 2) return DS4A_ERR_SHAPE;
  if (c->cap_raw == 0 || c->cap_raw > 1024) return DS4A_ERR_SHAPE;
  if (!c->raw_kv || !c->rope_cos || !c->rope_sin || c->rope_max_pos == 0) return DS4A_ERR_ARG;
  if (c->ratio) {
    if (!c->attn_comp_kv || !c->attn_state_kv || !c->attn_state_score) return DS4A_ERR_ARG;
    if (c->comp_cap == 0) return DS4A_ERR_CAPACITY;
  }
  if (c->ratio == 4) {
    if (c->index_dim == 0 || c->index_dim > 256 || c->index_dim % 4) return DS4A_ERR_SHAPE;
    if (c->index_rot > c->index_dim || c->index_rot % 2) return DS4A_ERR_SHAPE;
    if (!c->index_comp_kv || !c->index_state_kv || !c->index_state_score) return DS4A_ERR_ARG;
    if (!c->index_norm || !c->index_norm_max) return DS4A_ERR_ARG;
    if (!c->index_rope_cos || !c->index_rope_sin) return DS4A_ERR_ARG;
  }
  if (c->block_table) {
    if (c->ratio == 0 || c->max_blocks == 0 || c->n_blocks == 0) return DS4A_ERR_ARG;
    if ((uint64_t)c->max_blocks * (256u / c->ratio) != c->comp_cap) return DS4A_ERR_SHAPE;
  }
  if (c->qat & ~(DS4A_QAT_FP8_ATTN | DS4A_QAT_FP4_INDEX)) return DS4A_ERR_ARG;
  if ((c->qat & DS4A_QAT_FP8_ATTN) && c->ratio == 0) return DS4A_ERR_ARG;
  if (c->qat & DS4A_QAT_FP4_INDEX) {
    if (c->ratio != 4) return DS4A_ERR_ARG;
    if (c->index_dim < 32 || (c->index_dim & (c->index_dim - 1))) return DS4A_ERR_SHAPE;
  }
  return DS4A_OK;
}

ds4a_status cuda_status(cudaError_t e) {
  return note_error(e) == cudaSuccess ? DS4A_OK : DS4A_ERR_CUDA;
}

// Row maps of the attention lane (256/ratio rows per block) and the indexer
// lane (64 rows per block).
RowMap attn_map(const ds4a_layer_cache *c) {
  const uint32_t rpb = c->ratio ? 256u / c->ratio : 1u;
  return RowMap{c->block_table, c->comp_cap, c->max_blocks, rpb, c->n_blocks};
}
RowMap index_map(const ds4a_layer_cache *c) {
  return RowMap{c->block_table, c->comp_cap, c->max_blocks, 64u, c->n_blocks};
}

// c = 1/sqrt(n) rounded to fp32, the Hadamard normalisation of the FP4 round trip.
float hadamard_scale(uint32_t n) { return (float)(1.0 / std::sqrt((double)n)); }

uint32_t comp_rows(const ds4a_layer_cache *c, uint32_t n_tokens) {
  return c->ratio ? n_tokens / c->ratio : 0;
}

}  // namespace

extern "C" {

const char *ds4a_status_string(ds4a_status s) {
  switch (s) {
    case DS4A_OK: return "ok";
    case DS4A_ERR_ARG: return "invalid argument";
    case DS4A_ERR_SHAPE: return "unsupported or inconsistent shape";
    case DS4A_ERR_CAPACITY: return "capacity exceeded";
    case DS4A_ERR_POSITION: return "position does not match the cache";
    case DS4A_ERR_DTYPE: return "unknown dtype";
    case DS4A_ERR_CUDA: return "CUDA error";
    case DS4A_ERR_TIMEOUT: return "device wait timed out";
    case DS4A_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

uint32_t ds4a_layer_compress_ratio(int variant, uint32_t il) {
  if (il < 2) return variant == 0 ? 0u : 128u;
  return (il % 2 == 0) ? 4u : 128u;
}

const char *ds4a_last_error(void) {
  const int e = g_last_error.load(std::memory_order_relaxed);
  return e ? cudaGetErrorString((cudaError_t)e) : "no error";
}

uint64_t ds4a_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

uint32_t ds4a_prefill_chunk_cap(uint32_t prompt_len) { return prompt_len > 4096 ? 4096u : 0u; }

uint64_t ds4a_cache_bytes(uint32_t ratio, uint32_t head_dim, uint32_t index_dim, uint64_t ctx,
                          uint32_t batch, uint32_t elem_bytes) {
  const uint64_t raw = (ctx < 128 ? ctx : 128) * (uint64_t)head_dim;
  uint64_t comp = 0;
  if (ratio) comp = (ctx / ratio) * (uint64_t)(head_dim + (ratio == 4 ? index_dim : 0));
  return (uint64_t)batch * (raw + comp) * elem_bytes;
}

ds4a_status ds4a_rope_table(double base, uint32_t n_rot, uint32_t n_pos, float *cos_out,
                            float *sin_out) {
  if (!cos_out || !sin_out || n_rot == 0 || n_rot % 2 || !(base > 0.0)) return DS4A_ERR_ARG;
  const uint32_t half = n_rot / 2;
  double *theta = new double[half];
  for (uint32_t i = 0; i < half; ++i) theta[i] = std::pow(base, -2.0 * (double)i / (double)n_rot);
  for (uint32_t p = 0; p < n_pos; ++p)
    for (uint32_t i = 0; i < half; ++i) {
      const double ang = (double)p * theta[i];
      cos_out[(size_t)p * half + i] = (float)std::cos(ang);
      sin_out[(size_t)p * half + i] = (float)std::sin(ang);
    }
  delete[] theta;
  return DS4A_OK;
}

ds4a_status ds4a_cache_reset(ds4a_layer_cache *c, ds4a_stream_t stream) {
  ds4a_status st = check_cache(c);
  if (st) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint32_t W = window_of(c->ratio);
  if (c->ratio) {
    st = cuda_status(launch_state_reset(c->attn_state_kv, c->attn_state_score,
                                        (size_t)c->batch * W * c->head_dim, s));
    if (st) return st;
  }
  if (c->ratio == 4) {
    st = cuda_status(launch_state_reset(c->index_state_kv, c->index_state_score,
                                        (size_t)c->batch * 8 * c->index_dim, s));
    if (st) return st;
    st = cuda_status(cudaMemsetAsync(c->index_norm_max, 0, sizeof(uint32_t) * c->batch, s));
    if (st) return st;
  }
  c->n_tokens = 0;
  return DS4A_OK;
}

ds4a_status ds4a_index_norms(ds4a_layer_cache *c, ds4a_stream_t stream) {
  ds4a_status st = check_cache(c);
  if (st) return st;
  if (c->ratio != 4) return DS4A_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = cuda_status(cudaMemsetAsync(c->index_norm_max, 0, sizeof(uint32_t) * c->batch, s));
  if (st) return st;
  return cuda_status(launch_index_norms(c->dtype, c->index_comp_kv, index_map(c), c->index_dim,
                                        c->batch, comp_rows(c, c->n_tokens), c->index_norm,
                                        c->index_norm_max, s));
}

}  // extern "C"

namespace {

// The append of the parts in `lanes` (DS4A_LANE_*); `advance`: set n_tokens.
ds4a_status append_parts(ds4a_layer_cache *c, uint32_t pos0, uint32_t T, uint32_t lanes,
                         bool advance, const void *raw_kv_in, const void *attn_cand,
                         const void *attn_score, const void *ape_attn, const void *gamma_attn,
                         const void *idx_cand, const void *idx_score, const void *ape_idx,
                         const void *gamma_idx, void *raw_chunk_out, ds4a_stream_t stream) {
  ds4a_status st = check_cache(c);
  if (st) return st;
  if (T == 0) return DS4A_ERR_SHAPE;
  if (!lanes || (lanes & ~(DS4A_LANE_RAW | DS4A_LANE_ATTN | DS4A_LANE_INDEX))) return DS4A_ERR_ARG;
  const bool raw = lanes & DS4A_LANE_RAW;
  const bool la = lanes & DS4A_LANE_ATTN, li = lanes & DS4A_LANE_INDEX;
  if ((la && c->ratio == 0) || (li && c->ratio != 4)) return DS4A_ERR_ARG;
  if (raw && !raw_kv_in) return DS4A_ERR_ARG;
  if (pos0 != c->n_tokens) return DS4A_ERR_POSITION;
  if ((uint64_t)pos0 + T > c->rope_max_pos) return DS4A_ERR_CAPACITY;
  if (c->ratio && comp_rows(c, pos0 + T) > c->comp_cap) return DS4A_ERR_CAPACITY;
  if (la && (!attn_cand || !attn_score || !ape_attn || !gamma_attn)) return DS4A_ERR_ARG;
  if (li && (!idx_cand || !idx_score || !ape_idx || !gamma_idx)) return DS4A_ERR_ARG;

  AppendArgs a;
  std::memset(&a, 0, sizeof(a));
  a.ratio = c->ratio;
  a.window = window_of(c->ratio);
  a.batch = c->batch;
  a.cap_raw = c->cap_raw;
  a.comp_cap = c->comp_cap;
  a.head_dim = c->head_dim;
  a.n_rot = c->n_rot;
  a.pos0 = pos0;
  a.T = T;
  a.dtype = c->dtype;
  a.raw_in = raw_kv_in;
  a.direct = raw_chunk_out == nullptr;
  a.raw_dst = a.direct ? c->raw_kv : raw_chunk_out;
  a.cos = c->rope_cos;
  a.sin = c->rope_sin;
  a.y0 = raw ? 0u : 1u;
  a.seq_pos = c->seq_pos;
  a.n_lanes = 0;
  if (la) {
    a.lane[a.n_lanes++] =
        LaneArgs{c->head_dim, c->n_rot, c->attn_comp_kv, c->attn_state_kv, c->attn_state_score,
                 c->rope_cos, c->rope_sin, attn_cand, attn_score, ape_attn, gamma_attn,
                 nullptr, nullptr, (c->qat & DS4A_QAT_FP8_ATTN) ? 1u : 0u, 0.f, attn_map(c)};
  }
  if (li) {
    a.lane[a.n_lanes++] =
        LaneArgs{c->index_dim, c->index_rot, c->index_comp_kv, c->index_state_kv,
                 c->index_state_score, c->index_rope_cos, c->index_rope_sin, idx_cand,
                 idx_score, ape_idx, gamma_idx, c->index_norm, c->index_norm_max,
                 (c->qat & DS4A_QAT_FP4_INDEX) ? 2u : 0u, hadamard_scale(c->index_dim),
                 index_map(c)};
  }
  st = cuda_status(launch_append(a, reinterpret_cast<cudaStream_t>(stream)));
  if (st) return st;
  if (advance) c->n_tokens = pos0 + T;
  return DS4A_OK;
}

}  // namespace

extern "C" {

ds4a_status ds4a_compress_append(ds4a_layer_cache *c, uint32_t pos0, uint32_t T,
                                 const void *raw_kv_in, const void *attn_cand,
                                 const void *attn_score, const void *ape_attn,
                                 const void *gamma_attn, const void *idx_cand,
                                 const void *idx_score, const void *ape_idx,
                                 const void *gamma_idx, void *raw_chunk_out,
                                 ds4a_stream_t stream) {
  if (!c) return DS4A_ERR_ARG;
  const uint32_t lanes = DS4A_LANE_RAW | (c->ratio ? DS4A_LANE_ATTN : 0u) |
                         (c->ratio == 4 ? DS4A_LANE_INDEX : 0u);
  return append_parts(c, pos0, T, lanes, true, raw_kv_in, attn_cand, attn_score, ape_attn,
                      gamma_attn, idx_cand, idx_score, ape_idx, gamma_idx, raw_chunk_out, stream);
}

ds4a_status ds4a_compress_append_lanes(ds4a_layer_cache *c, uint32_t pos0, uint32_t T,
                                       uint32_t lanes, const void *raw_kv_in,
                                       const void *attn_cand, const void *attn_score,
                                       const void *ape_attn, const void *gamma_attn,
                                       const void *idx_cand, const void *idx_score,
                                       const void *ape_idx, const void *gamma_idx,
                                       void *raw_chunk_out, ds4a_stream_t stream) {
  return append_parts(c, pos0, T, lanes, false, raw_kv_in, attn_cand, attn_score, ape_attn,
                      gamma_attn, idx_cand, idx_score, ape_idx, gamma_idx, raw_chunk_out, stream);
}

size_t ds4a_workspace_bytes(int call, const ds4a_layer_cache *c, uint32_t T, uint32_t n_heads,
                            uint32_t top_k) {
  if (!c) return 0;
  switch (call) {
    case DS4A_CALL_INDEX_TOPK:
      return index_ws_bytes(c->dtype, c->batch, T, n_heads, c->index_dim, c->comp_cap);
    case DS4A_CALL_ATTN_DECODE:
      return attn_ws_bytes(c->dtype, c->ratio, c->batch, 1, n_heads, c->head_dim, c->n_rot,
                           c->cap_raw, c->comp_cap, c->ratio == 4 ? top_k : 0);
    case DS4A_CALL_ATTN_PREFILL:
      return attn_ws_bytes(c->dtype, c->ratio, c->batch, T, n_heads, c->head_dim, c->n_rot,
                           c->cap_raw, c->comp_cap, c->ratio == 4 ? top_k : 0);
    default:
      return 0;
  }
}

}  // extern "C"

namespace ds4a {
// Every check of ds4a_index_topk except the workspace's (shared with the
// no-allocation variant, which checks its scratch size after these).
ds4a_status index_topk_check(const ds4a_layer_cache *c, uint32_t pos0, uint32_t T,
                             const void *q_idx, const void *w, uint32_t n_heads, uint32_t top_k,
                             const int32_t *topk) {
  ds4a_status st = check_cache(c);
  if (st) return st;
  if (c->ratio != 4) return DS4A_ERR_ARG;
  if (T == 0 || n_heads == 0 || n_heads > 128 || top_k == 0 || top_k > 2048) return DS4A_ERR_SHAPE;
  if (!q_idx || !w || !topk) return DS4A_ERR_ARG;
  if ((uint64_t)pos0 + T > c->n_tokens) return DS4A_ERR_POSITION;
  const uint32_t Hp = (n_heads + 7u) & ~7u;
  if (((size_t)c->index_dim * Hp + Hp + 128 * (size_t)(c->index_dim + 1)) * 4 > 227 * 1024)
    return DS4A_ERR_SHAPE;
  return DS4A_OK;
}
}  // namespace ds4a

extern "C" {

ds4a_status ds4a_index_topk(const ds4a_layer_cache *c, uint32_t pos0, uint32_t T,
                            const void *q_idx, const void *w, uint32_t n_heads, uint32_t top_k,
                            int32_t *topk, void *ws, size_t ws_bytes, ds4a_stream_t stream) {
  const ds4a_status st = index_topk_check(c, pos0, T, q_idx, w, n_heads, top_k, topk);
  if (st) return st;
  const size_t need = index_ws_bytes(c->dtype, c->batch, T, n_heads, c->index_dim, c->comp_cap);
  if (!ws || ws_bytes < need) return DS4A_ERR_WORKSPACE;
  IndexArgs a;
  a.batch = c->batch;
  a.T = T;
  a.pos0 = pos0;
  a.n_heads = n_heads;
  a.dim = c->index_dim;
  a.rot = c->index_rot;
  a.top_k = top_k;
  a.comp_cap = c->comp_cap;
  a.n_comp = comp_rows(c, c->n_tokens);
  a.dtype = c->dtype;
  a.q_idx = q_idx;
  a.w = w;
  a.keys = c->index_comp_kv;
  a.norms = c->index_norm;
  a.norm_max = c->index_norm_max;
  a.cos = c->index_rope_cos;
  a.sin = c->index_rope_sin;
  a.topk = topk;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.qat = (c->qat & DS4A_QAT_FP4_INDEX) != 0;
  a.had_c = hadamard_scale(c->index_dim);
  a.map = index_map(c);
  a.seq_pos = c->seq_pos;
  return cuda_status(launch_index_topk(a, reinterpret_cast<cudaStream_t>(stream)));
}

static ds4a_status attn_common(const ds4a_layer_cache *c, uint32_t pos0, uint32_t T,
                               const void *q, uint32_t n_heads, const void *raw_chunk,
                               const int32_t *topk, uint32_t top_k, float scale, void *out,
                               void *ws, size_t ws_bytes, cudaStream_t s) {
  if (T == 0 || n_heads == 0 || n_heads > 128) return DS4A_ERR_SHAPE;
  if (!q || !out) return DS4A_ERR_ARG;
  if (!std::isfinite(scale)) return DS4A_ERR_ARG;
  if (c->ratio == 4 && (!topk || top_k == 0 || top_k > 2048)) return DS4A_ERR_ARG;
  const size_t need = attn_ws_bytes(c->dtype, c->ratio, c->batch, T, n_heads, c->head_dim,
                                    c->n_rot, c->cap_raw, c->comp_cap, c->ratio == 4 ? top_k : 0);
  if (need && (!ws || ws_bytes < need)) return DS4A_ERR_WORKSPACE;
  AttnArgs a;
  a.ratio = c->ratio;
  a.batch = c->batch;
  a.T = T;
  a.pos0 = pos0;
  a.n_heads = n_heads;
  a.head_dim = c->head_dim;
  a.n_rot = c->n_rot;
  a.cap_raw = c->cap_raw;
  a.comp_cap = c->comp_cap;
  a.n_comp = comp_rows(c, c->n_tokens);
  a.top_k = c->ratio == 4 ? top_k : 0;
  a.dtype = c->dtype;
  a.scale = scale;
  a.q = q;
  a.ring = c->raw_kv;
  a.chunk = raw_chunk;
  a.comp = c->attn_comp_kv;
  a.topk = c->ratio == 4 ? topk : nullptr;
  a.cos = c->rope_cos;
  a.sin = c->rope_sin;
  a.out = out;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.map = attn_map(c);
  a.seq_pos = c->seq_pos;
  return cuda_status(launch_attention(a, s));
}

ds4a_status ds4a_sparse_attn_decode(const ds4a_layer_cache *c, uint32_t pos, const void *q,
                                    uint32_t n_heads, const int32_t *topk, uint32_t top_k,
                                    float scale, void *out, void *ws, size_t ws_bytes,
                                    ds4a_stream_t stream) {
  ds4a_status st = check_cache(c);
  if (st) return st;
  if ((uint64_t)pos + 1 != c->n_tokens) return DS4A_ERR_POSITION;
  return attn_common(c, pos, 1, q, n_heads, nullptr, topk, top_k, scale, out, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

ds4a_status ds4a_set_decode_cluster(uint32_t C) {
  if (C > 16) return DS4A_ERR_ARG;
  attn_tc_force_cluster(C);
  return DS4A_OK;
}

uint32_t ds4a_decode_cluster_size(const ds4a_layer_cache *c, uint32_t n_heads, uint32_t top_k) {
  if (check_cache(c) != DS4A_OK) return 0;
  // (a decode call's token is at n_tokens - 1)
  return attn_decode_cluster(c->dtype, c->ratio, c->batch, n_heads, c->head_dim, c->n_rot,
                             c->cap_raw, c->comp_cap, c->ratio == 4 ? top_k : 0,
                             comp_rows(c, c->n_tokens), c->n_tokens);
}

ds4a_status ds4a_sparse_attn_prefill_chunk(ds4a_layer_cache *c, uint32_t pos0, uint32_t T,
                                           const void *q, uint32_t n_heads,
                                           const void *raw_chunk, const int32_t *topk,
                                           uint32_t top_k, float scale, void *out, void *ws,
                                           size_t ws_bytes, ds4a_stream_t stream) {
  ds4a_status st = check_cache(c);
  if (st) return st;
  if (!raw_chunk) return DS4A_ERR_ARG;
  if (T == 0) return DS4A_ERR_SHAPE;
  if ((uint64_t)pos0 + T != c->n_tokens) return DS4A_ERR_POSITION;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = attn_common(c, pos0, T, q, n_heads, raw_chunk, topk, top_k, scale, out, ws, ws_bytes, s);
  if (st) return st;
  return cuda_status(launch_ring_commit(c->dtype, c->batch, T, pos0, c->seq_pos, c->cap_raw,
                                        c->head_dim, raw_chunk, c->raw_kv, s));
}

}  // extern "C"
