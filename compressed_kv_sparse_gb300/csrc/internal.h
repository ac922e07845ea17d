// Internal launcher interface between the C ABI layer (api.cu) and the kernel
// translation units. Arguments have been validated by the caller.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ds4a.h"

namespace ds4a {

// Counts kernel launches (ds4a_launch_count); call once per launch.
void note_launches(uint32_t n);

// Records a CUDA error for ds4a_last_error and passes it through.
cudaError_t note_error(cudaError_t e);

// Raise a kernel's dynamic shared memory limit to `bytes` (no-op below 48 KiB
// or when already raised that far).
template <typename F>
cudaError_t ensure_smem(F *func, size_t bytes, int *done) {
  if (bytes <= 48 * 1024 || (size_t)*done >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) *done = (int)bytes;
  return e;
}

// Launch with programmatic stream serialization (see pdl_wait in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Where row i of sequence b of a compressed lane lives. Contiguous (table
// NULL): row b * cap + i. Paged: the logical block i / rpb of sequence b is
// physical block table[b * max_blocks + i / rpb] and the row is that block's
// row i % rpb. An entry outside [0, n_blocks) is a caller error: its rows
// are not written, and reads of them return rows of block 0 (every access
// stays inside the pools). phys() returns false for such rows and for rows
// past the table's max_blocks logical blocks.
struct RowMap {
  const int32_t *table;
  uint32_t cap, max_blocks, rpb, n_blocks;
#ifdef __CUDACC__
  __device__ __forceinline__ bool phys(uint32_t b, uint32_t i, size_t &row) const {
    if (!table) {
      row = (size_t)b * cap + i;
      return true;
    }
    const uint32_t lb = i / rpb;   // (rows past the last logical block: block 0, not ok)
    const uint32_t blk = lb < max_blocks ? (uint32_t)__ldg(table + (size_t)b * max_blocks + lb)
                                         : 0xffffffffu;
    const bool ok = blk < n_blocks;
    row = (size_t)(ok ? blk : 0u) * rpb + i % rpb;
    return ok;
  }
  __device__ __forceinline__ size_t row_of(uint32_t b, uint32_t i) const {
    size_t r;
    phys(b, i, r);
    return r;
  }
#endif
};

// The argument checks of ds4a_index_topk other than the workspace's (api.cu).
ds4a_status index_topk_check(const ds4a_layer_cache *c, uint32_t pos0, uint32_t T,
                             const void *q_idx, const void *w, uint32_t n_heads, uint32_t top_k,
                             const int32_t *topk);

// TMA tensor map over bf16 data with 128-byte swizzle (tmap.cu).
cudaError_t make_tmap_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                           const uint64_t *strides_bytes, const uint32_t *box);
int num_sms();

// One compressor lane (attention or indexer) of a layer.
struct LaneArgs {
  uint32_t width, n_rot;
  void *comp;             // [B][comp_cap][width]
  float *state_kv, *state_score;  // [B][W][width]
  const float *cos, *sin; // [max_pos][n_rot/2]
  const void *cand, *score;       // [B][T][width]
  const void *ape, *gamma;        // [W][width], [width]
  float *norm;                    // [B][comp_cap] row norms (indexer lane) or NULL
  uint32_t *norm_max;             // [B] float bits of the largest norm
  uint32_t quant;                 // step 8: 0 none, 1 FP8 non-RoPE dims, 2 FP4 QAT
  float had_c;                    // 1/sqrt(width) in fp32 (quant 2)
  RowMap map;                     // rows of comp (and norm)
};

struct AppendArgs {
  uint32_t ratio, window, batch, cap_raw, comp_cap, head_dim, n_rot, pos0, T;
  int dtype;
  const void *raw_in;     // [B][T][D]
  void *raw_dst;          // ring [B][cap][D] (direct) or chunk [B][T][D]
  bool direct;            // raw rows go to the ring
  const float *cos, *sin; // attention-lane / raw-row table
  int n_lanes;             // lanes to append (lane[0 .. n_lanes-1])
  LaneArgs lane[2];
  uint32_t y0;             // 1: the raw rows are not part of this append
  const uint32_t *seq_pos; // [B] per-sequence first positions (ragged batches) or NULL
};
cudaError_t launch_append(const AppendArgs &a, cudaStream_t s);

struct IndexArgs {
  uint32_t batch, T, pos0, n_heads, dim, rot, top_k, comp_cap, n_comp;
  int dtype;
  const void *q_idx, *w, *keys;   // [B][T][Hi][Di], [B][T][Hi], [B][comp_cap][Di]
  const float *norms;             // [B][comp_cap] row norms
  const uint32_t *norm_max;       // [B] float bits of the largest row norm
  const float *cos, *sin;
  int32_t *topk;
  void *ws;
  size_t ws_bytes;
  bool qat;                       // FP4 QAT round trip of the rotated query
  float had_c;                    // 1/sqrt(dim) in fp32
  RowMap map;                     // rows of keys and norms
  const uint32_t *seq_pos;        // [B] per-sequence positions (ragged decode) or NULL
};
size_t index_ws_bytes(int dtype, uint32_t batch, uint32_t T, uint32_t n_heads, uint32_t dim,
                      uint32_t comp_cap);

// Tensor-core scorer of bf16 layers (indexer_tc.cu).
struct IndexTcArgs {
  uint32_t batch, T, pos0, comp_cap, n_comp;
  const void *keys;   // [B][comp_cap][128] bf16
  const void *qbf;    // [B][T][64][128] bf16, rotated queries
  const void *w;      // [B][T][64] bf16
  float *scores;      // [B][T][score_stride]
  uint32_t score_stride;
  uint32_t *hist;     // [B*T][4096], zeroed before the call
  int *err;
  RowMap map;         // rows of keys
  const uint32_t *seq_pos;   // [B] per-sequence positions (ragged decode) or NULL
};
bool index_tc_supported(uint32_t n_heads, uint32_t dim);
cudaError_t launch_index_score_tc(const IndexTcArgs &a, cudaStream_t s);
cudaError_t launch_index_topk(const IndexArgs &a, cudaStream_t s);

struct AttnArgs {
  uint32_t ratio, batch, T, pos0, n_heads, head_dim, n_rot, cap_raw, comp_cap, n_comp, top_k;
  int dtype;
  float scale;
  const void *q;          // [B][T][H][D]
  const void *ring;       // [B][cap][D]
  const void *chunk;      // [B][T][D] or NULL
  const void *comp;       // [B][comp_cap][D]
  const int32_t *topk;    // [B][T][k] or NULL
  const float *cos, *sin;
  void *out;              // [B][T][H][D]
  void *ws;
  size_t ws_bytes;
  RowMap map;             // rows of comp
  const uint32_t *seq_pos;  // [B] per-sequence positions (ragged decode) or NULL
};
size_t attn_ws_bytes(int dtype, uint32_t ratio, uint32_t batch, uint32_t T, uint32_t n_heads,
                     uint32_t head_dim, uint32_t n_rot, uint32_t cap_raw, uint32_t comp_cap,
                     uint32_t top_k);
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s);

// Tensor-core attention (attention_tc.cu): bf16, 64 heads x 512 dims, 64-dim tail.
bool attn_tc_supported(int dtype, uint32_t H, uint32_t D, uint32_t n_rot);
size_t attn_tc_ws_bytes(uint32_t batch, uint32_t T, uint32_t rows_max);
cudaError_t launch_attention_tc(const AttnArgs &a, uint32_t rows_max, int *err, cudaStream_t s);
// Decode cluster size: forced process-wide (0 = automatic), and the size a
// decode launch of `n_q` queries with at most `rows_max` rows each uses.
void attn_tc_force_cluster(uint32_t C);
uint32_t attn_tc_decode_cluster(uint32_t rows_max, uint32_t n_q);
// The same for the arguments of a decode call whose token is at position
// pos_end - 1: 0 when it does not run on the tensor-core kernel.
uint32_t attn_decode_cluster(int dtype, uint32_t ratio, uint32_t batch, uint32_t n_heads,
                             uint32_t head_dim, uint32_t n_rot, uint32_t cap_raw,
                             uint32_t comp_cap, uint32_t top_k, uint32_t n_comp,
                             uint64_t pos_end);
cudaError_t launch_ring_commit(int dtype, uint32_t batch, uint32_t T, uint32_t pos0,
                               const uint32_t *seq_pos, uint32_t cap_raw, uint32_t head_dim,
                               const void *chunk, void *ring, cudaStream_t s);
cudaError_t launch_state_reset(float *kv, float *score, size_t n, cudaStream_t s);
cudaError_t launch_index_norms(int dtype, const void *rows, const RowMap &map, uint32_t dim,
                               uint32_t batch, uint32_t n_rows, float *norm, uint32_t *norm_max,
                               cudaStream_t s);

}  // namespace ds4a
