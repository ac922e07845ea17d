/*
 * ds4a — compressed-KV sparse attention layer for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libds4a.so. One call per step of the per-layer path an inference
 * engine runs for every token of a DeepSeek-V4-style model:
 *
 *   ds4a_compress_append          raw-window insert + KV compressor
 *                                 (ds4a_compress_append_lanes: a part of it)
 *   ds4a_index_topk               ratio-4 indexer scores + exact top-k
 *   ds4a_sparse_attn_decode       attention of one new token per sequence
 *   ds4a_sparse_attn_prefill_chunk attention of a chunk of T tokens
 *
 * Sources ("page §n" below): "【#3】ds4.c を読み解く" (qiita, DwarfStar series
 * part 3) and "vLLM DeepSeek V4 サポート: 効率的な長文コンテキスト注意機構"
 * (section "DeepSeek V4 アテンションアーキテクチャ").
 *
 * Conventions for every call:
 *  - All tensor pointers are caller-owned DEVICE memory unless stated
 *    otherwise; the library never allocates, frees or synchronises. Calls are
 *    asynchronous on the given stream (0 = legacy default stream).
 *  - Arguments are checked on the host before any launch; a failed check
 *    returns a negative status and launches nothing. A launch error returns
 *    DS4A_ERR_CUDA (the CUDA error is left for the caller to read).
 *  - All sequences of a batch are at the same position. ds4a_layer_cache.n_tokens
 *    is the host-side count of tokens appended so far; ds4a_compress_append
 *    requires pos0 == n_tokens and advances it, the other calls require the
 *    tokens they read to have been appended (DS4A_ERR_POSITION otherwise).
 *  - Row-major layouts, innermost dimension last. Element type of rows,
 *    inputs and outputs is ds4a_layer_cache.dtype (fp32 or bf16); the
 *    compressor state is always fp32.
 *  - Order within a step: append -> index_topk (ratio 4) -> attention.
 */
#ifndef DS4A_H
#define DS4A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ds4a_stream_t; /* same as cudaStream_t */

typedef enum {
  DS4A_OK = 0,
  DS4A_ERR_ARG = -1,       /* NULL pointer or unsupported parameter value */
  DS4A_ERR_SHAPE = -2,     /* inconsistent or unsupported sizes */
  DS4A_ERR_CAPACITY = -3,  /* comp_cap or a table too small for the request */
  DS4A_ERR_POSITION = -4,  /* pos0 does not match the cache's token count */
  DS4A_ERR_DTYPE = -5,     /* unknown dtype */
  DS4A_ERR_CUDA = -6,      /* a CUDA launch or API call failed */
  DS4A_ERR_TIMEOUT = -7,   /* a bounded device-side wait gave up */
  DS4A_ERR_WORKSPACE = -8  /* workspace missing or smaller than required */
} ds4a_status;

typedef enum { DS4A_F32 = 0, DS4A_BF16 = 1 } ds4a_dtype;

/*
 * One layer's cache for `batch` sequences (page §2, ds4_layer_cache).
 *
 *  ratio        0 (raw window only), 4 (c4a) or 128 (c128a) — page §1.
 *  head_dim     D, the shared K = V head dimension; even, <= 1024.
 *  n_rot        rotated tail dims of attention rows and queries (page §8: 64);
 *               even, <= head_dim.
 *  index_dim    Di, indexer head dim (ratio 4 only; page §6: 128); even, <= 256.
 *  index_rot    rotated tail dims of indexer rows and queries (min(64, Di)).
 *  batch        B.
 *  cap_raw      raw window rows (page §2: 128); row of position p is at slot
 *               p % cap_raw. 1 <= cap_raw <= 1024.
 *  comp_cap     compressed rows held per sequence (ratio != 0).
 *  dtype        ds4a_dtype of rows, inputs and outputs.
 *  n_tokens     HOST field: tokens appended so far (same for every sequence).
 *
 *  raw_kv            [B][cap_raw][D]      rotated raw rows (K = V)
 *  attn_comp_kv      [B][comp_cap][D]     compressed attention rows
 *  attn_state_kv     [B][W][D] fp32       W = 8 (ratio 4) or 128 (ratio 128)
 *  attn_state_score  [B][W][D] fp32       scores WITHOUT the APE bias; -inf = empty
 *  index_comp_kv     [B][comp_cap][Di]    compressed indexer rows (ratio 4, else NULL)
 *  index_state_kv    [B][8][Di] fp32
 *  index_state_score [B][8][Di] fp32
 *  index_norm        [B][comp_cap] fp32 (ratio 4): Euclidean norm of each stored
 *                    indexer row, widened by 1e-4; the certified top-k bounds
 *                    the error of its tensor-core scores with it. Written by
 *                    ds4a_compress_append; after writing rows any other way,
 *                    call ds4a_index_norms. Not part of the pages' cache.
 *  index_norm_max    [B] uint32 (ratio 4): float bits of the largest
 *                    index_norm written to each sequence since the last
 *                    ds4a_cache_reset.
 *  rope_cos/rope_sin [rope_max_pos][n_rot/2] fp32: this layer's rotation
 *                    coefficients (ds4a_rope_table), base = compression base on
 *                    layers with ratio != 0, normal base otherwise (page §8).
 *  index_rope_cos/sin [rope_max_pos][index_rot/2] fp32 (same base), ratio 4.
 *  rope_max_pos      rows of the tables; every position used must be below it.
 *  qat               step 8 of the compressor (page §4 step 8, §9), a bit set:
 *                    DS4A_QAT_FP8_ATTN (ratio != 0): every compressed attention
 *                    row is quantised to FP8 E4M3 and back on its leading
 *                    head_dim - n_rot dims before it is stored;
 *                    DS4A_QAT_FP4_INDEX (ratio 4, Di a power of two >= 32):
 *                    compressed indexer rows, and in ds4a_index_topk the
 *                    rotated queries, take the FP4 QAT round trip. 0 = off.
 *                    Scales and arithmetic: see DS4A_QAT_FP8_ATTN below.
 *  block_table       NULL: compressed rows are contiguous per sequence as laid
 *                    out above. Non-NULL (ratio != 0): a paged cache (vLLM's
 *                    page: one logical block = 256 token positions on every
 *                    compressed layer, i.e. 64 rows on c4a, 2 on c128a).
 *                    [B][max_blocks] int32 DEVICE array: entry (b, j) is the
 *                    physical block holding rows 256/ratio * j .. of sequence
 *                    b. Then attn_comp_kv is a pool [n_blocks][256/ratio][D],
 *                    index_comp_kv [n_blocks][64][Di] and index_norm
 *                    [n_blocks][64], and comp_cap must equal
 *                    max_blocks * 256/ratio. Sequences may share blocks (a
 *                    common prefix) when nothing appends into them. Entries
 *                    must lie in [0, n_blocks); an entry outside is not
 *                    written to, and reads of its rows return rows of block 0.
 *  max_blocks, n_blocks  see block_table (ignored when it is NULL).
 *  seq_pos           NULL: every sequence is at the call's position. Non-NULL
 *                    (ragged batches): [B] uint32 DEVICE array, the position
 *                    of sequence b's first token in this call: a decode step
 *                    (T = 1) places and reads sequence b's token at seq_pos[b]
 *                    instead of pos, and a prefill chunk (T > 1) covers
 *                    positions seq_pos[b] .. seq_pos[b] + T - 1 of sequence b
 *                    instead of pos0 .. pos0 + T - 1 (each sequence's raw
 *                    window, compressor boundaries, visible rows and window
 *                    commit follow its own positions). The host checks use the
 *                    call's pos0 and n_tokens: the caller keeps every
 *                    seq_pos[b] <= pos0 (the capacity and rope-table checks
 *                    then cover every sequence) and updates the array between
 *                    calls.
 *
 * State layout: ratio 4 keeps the last complete group of 4 tokens in slots
 * 0..3 and token p of the current group in slot 4 + p % 4 (page §5's 8-row
 * frontier); ratio 128 keeps token p in slot p % 128. A fresh cache must have
 * every state score at -inf (ds4a_cache_reset).
 */
typedef struct {
  uint32_t ratio, head_dim, n_rot, index_dim, index_rot, batch, cap_raw, comp_cap;
  int32_t dtype;
  uint32_t n_tokens;
  void *raw_kv;
  void *attn_comp_kv;
  float *attn_state_kv, *attn_state_score;
  void *index_comp_kv;
  float *index_state_kv, *index_state_score;
  float *index_norm;
  uint32_t *index_norm_max;
  const float *rope_cos, *rope_sin;
  const float *index_rope_cos, *index_rope_sin;
  uint32_t rope_max_pos;
  uint32_t qat;
  const int32_t *block_table;
  uint32_t max_blocks, n_blocks;
  const uint32_t *seq_pos;
} ds4a_layer_cache;

/*
 * Step-8 round trips (page §9: E4M3 FP8 on the non-RoPE part of attention
 * rows; Hadamard-128 plus FP4 activation quantisation on indexer rows and the
 * indexer query). The pages give no granularity; this library fixes it:
 *  FP8: blocks of 64 consecutive non-RoPE dims (the last may be shorter), each
 *       with the scale 2^k, k the smallest integer >= -127 such that
 *       amax <= 448 * 2^k; each dim becomes the E4M3 value nearest x / 2^k
 *       (ties to the even code) times 2^k. RoPE dims are unchanged.
 *  FP4: z = c * H x, with H the Sylvester Hadamard matrix of order Di,
 *       applied as radix-2 butterflies over stages h = 1, 2, ..., Di/2 in fp32,
 *       and c = 1/sqrt(Di) rounded to fp32. z is cut into blocks of 32, each
 *       with the scale 2^k (amax <= 6 * 2^k, k >= -127) and the nearest E2M1
 *       value. The result is x' = c * H z'.
 * The input is the fp32 row (after RMSNorm and tail RoPE) or query (after its
 * tail rotation). The output is rounded once to dtype; FP8 values are exact in
 * both dtypes. The cache keeps the dequantised values in dtype.
 */
#define DS4A_QAT_FP8_ATTN 1u
#define DS4A_QAT_FP4_INDEX 2u

/* Workspace selectors for ds4a_workspace_bytes. */
enum { DS4A_CALL_APPEND = 0, DS4A_CALL_INDEX_TOPK = 1, DS4A_CALL_ATTN_DECODE = 2,
       DS4A_CALL_ATTN_PREFILL = 3 };

/*
 * Empty the compressor state (kv 0, score -inf), zero index_norm_max and set
 * n_tokens = 0. Rows are left as they are. Asynchronous on `stream`.
 */
ds4a_status ds4a_cache_reset(ds4a_layer_cache *cache, ds4a_stream_t stream);

/*
 * Recompute index_norm for rows 0 .. n_comp - 1 of every sequence (n_comp =
 * compressed rows of n_tokens tokens) and index_norm_max from them, for a
 * ratio-4 cache whose indexer rows were written by the caller (a restored or
 * imported cache). The pages have no counterpart: the norms serve the
 * certified top-k only. Asynchronous on `stream`.
 * Errors: DS4A_ERR_ARG (not ratio 4, or a cache field missing),
 * DS4A_ERR_CUDA.
 */
ds4a_status ds4a_index_norms(ds4a_layer_cache *cache, ds4a_stream_t stream);

/*
 * Append tokens pos0 .. pos0+T-1 of every sequence (page §4 compressor steps
 * 1-7, §5 frontier, §8 tail RoPE; vLLM c4a / c128a window geometry).
 *
 *  raw_kv_in    [B][T][D]   projected raw KV row of each token (before RoPE)
 *  attn_cand    [B][T][D]   compressor KV candidate (wkv output)   } ratio != 0,
 *  attn_score   [B][T][D]   compressor score (wgate output)        } else NULL
 *  ape_attn     [W][D]      APE bias, row = slot within the window (0 = oldest)
 *  gamma_attn   [D]         RMSNorm gain of compressed attention rows
 *  idx_cand, idx_score [B][T][Di], ape_idx [8][Di], gamma_idx [Di]: the indexer
 *               lane (ratio 4, else NULL).
 *  raw_chunk_out NULL: each token's rotated raw row goes into raw_kv at slot
 *               p % cap_raw (decode). Non-NULL: [B][T][D] receives the rotated
 *               raw rows and raw_kv is NOT touched; ds4a_sparse_attn_prefill_chunk
 *               then attends them and writes the last min(T, cap_raw) of them
 *               into raw_kv (prefill).
 *
 * Per token p: raw row = tail-RoPE(raw_kv_in, p). For each lane, the candidate
 * and score go into the state slot of p; when (p + 1) % ratio == 0 the window
 * is pooled per channel with weights exp(score + APE - max) (empty slots weigh
 * 0, an all-empty channel gives 0), RMS-normalised (eps 1e-6) with the gain,
 * rotated at position i * ratio and stored as compressed row i = (p+1)/ratio - 1;
 * ratio 4 then moves slots 4..7 to 0..3. Requires pos0 == n_tokens and
 * (pos0 + T) / ratio <= comp_cap; sets n_tokens = pos0 + T.
 */
ds4a_status ds4a_compress_append(ds4a_layer_cache *cache, uint32_t pos0, uint32_t T,
                                 const void *raw_kv_in, const void *attn_cand,
                                 const void *attn_score, const void *ape_attn,
                                 const void *gamma_attn, const void *idx_cand,
                                 const void *idx_score, const void *ape_idx,
                                 const void *gamma_idx, void *raw_chunk_out,
                                 ds4a_stream_t stream);

/* Parts of an append, for ds4a_compress_append_lanes. */
#define DS4A_LANE_RAW 1u    /* the raw-window rows (raw_kv or raw_chunk_out) */
#define DS4A_LANE_ATTN 2u   /* the attention lane: state and compressed rows */
#define DS4A_LANE_INDEX 4u  /* the indexer lane (ratio 4): state, rows, row norms */

/*
 * ds4a_compress_append restricted to the parts in `lanes` (a nonzero set of
 * DS4A_LANE_*; lanes the layer does not have are an error). The parts touch
 * disjoint memory, so they may run on different streams at once. vLLM's page
 * runs the indexer pipeline of a c4a layer on its own stream, beside the main
 * KV compression and the SWA insert ("Multi-stream Partitioning"). Inputs of
 * parts not selected may be NULL. Requires pos0 == n_tokens and leaves n_tokens
 * unchanged: once every part the caller needs is appended, it sets
 * cache->n_tokens = pos0 + T itself. Errors as for ds4a_compress_append, plus
 * DS4A_ERR_ARG for an empty or invalid lane set.
 */
ds4a_status ds4a_compress_append_lanes(ds4a_layer_cache *cache, uint32_t pos0, uint32_t T,
                                       uint32_t lanes, const void *raw_kv_in,
                                       const void *attn_cand, const void *attn_score,
                                       const void *ape_attn, const void *gamma_attn,
                                       const void *idx_cand, const void *idx_score,
                                       const void *ape_idx, const void *gamma_idx,
                                       void *raw_chunk_out, ds4a_stream_t stream);

/*
 * Indexer top-k for queries at positions pos0 .. pos0+T-1 (ratio 4 only;
 * page §6 indexer, §7 visible rows; vLLM DSA).
 *
 *  q_idx   [B][T][Hi][Di]  indexer queries before RoPE (dtype)
 *  w       [B][T][Hi]      per-head weights (dtype)
 *  n_heads Hi (1..128), top_k k (1..2048)
 *  topk    [B][T][k] int32 out: for the query at p, the k rows s < floor((p+1)/4)
 *          with the largest score I = sum_h w_h * ReLU(q'_h . k_s), ties to the
 *          lower index, in ascending order, padded with -1 when fewer are visible.
 *  ws      workspace of ds4a_workspace_bytes(DS4A_CALL_INDEX_TOPK, ...) bytes;
 *          its first 4 bytes are the call's wait status (ds4a_workspace_status).
 *
 * q' = tail rotation of q_idx at p, computed in fp32 (one rounding per
 * operation), then the FP4 QAT round trip when cache->qat has
 * DS4A_QAT_FP4_INDEX, and rounded to dtype. The selection is exact with respect to the
 * fp32 score defined by: dot_h accumulated in ascending d with separately
 * rounded products and sums, ReLU to +0, then w_h * relu_h summed in ascending
 * h from +0. Requires pos0 + T <= n_tokens.
 */
ds4a_status ds4a_index_topk(const ds4a_layer_cache *cache, uint32_t pos0, uint32_t T,
                            const void *q_idx, const void *w, uint32_t n_heads,
                            uint32_t top_k, int32_t *topk, void *ws, size_t ws_bytes,
                            ds4a_stream_t stream);

/*
 * Attention of the token at position pos of every sequence (page §7 mixed
 * attention; vLLM shared K = V, inverse RoPE, 128-token window).
 *
 *  q       [B][H][D]  queries before RoPE (dtype); n_heads = H (1..128)
 *  topk    [B][top_k] int32 compressed rows to attend (ratio 4): entries < 0 are
 *          skipped and the list ends at the first entry >= floor((pos+1)/4).
 *          Ignored (may be NULL) on ratio 0 and 128 layers: ratio 128 attends
 *          every visible row s < floor((pos+1)/128), ratio 0 none.
 *  scale   softmax scale (1/sqrt(D) is the usual choice)
 *  out     [B][H][D] (dtype): softmax over the raw rows of positions
 *          max(0, pos-cap_raw+1)..pos plus the compressed rows, V = K, with the
 *          output tail rotated back by -pos.
 *  ws      ds4a_workspace_bytes(DS4A_CALL_ATTN_DECODE, ...) bytes (may be NULL when
 *          that is 0); its first 4 bytes count timed-out device waits
 *          (ds4a_workspace_status).
 * Requires pos + 1 == n_tokens (the token has been appended).
 */
ds4a_status ds4a_sparse_attn_decode(const ds4a_layer_cache *cache, uint32_t pos,
                                    const void *q, uint32_t n_heads, const int32_t *topk,
                                    uint32_t top_k, float scale, void *out, void *ws,
                                    size_t ws_bytes, ds4a_stream_t stream);

/*
 * Attention of a prefill chunk, queries at pos0 .. pos0+T-1, then the raw
 * window commit (page §3: chunked prefill keeps absolute positions).
 *
 *  q         [B][T][H][D] queries before RoPE
 *  raw_chunk [B][T][D] the rotated raw rows ds4a_compress_append wrote to its
 *            raw_chunk_out for the same tokens
 *  topk      [B][T][top_k] (ratio 4) as for decode, per query
 *  out       [B][T][H][D]
 * The raw window of query p spans positions max(0, p-cap_raw+1)..p: rows before
 * pos0 come from raw_kv (still as it was before the chunk), the rest from
 * raw_chunk. Compressed rows visible to p are s < floor((p+1)/ratio). After the
 * attention, the last min(T, cap_raw) chunk rows are written to raw_kv.
 * Requires pos0 + T == n_tokens.
 */
ds4a_status ds4a_sparse_attn_prefill_chunk(ds4a_layer_cache *cache, uint32_t pos0, uint32_t T,
                                           const void *q, uint32_t n_heads,
                                           const void *raw_chunk, const int32_t *topk,
                                           uint32_t top_k, float scale, void *out, void *ws,
                                           size_t ws_bytes, ds4a_stream_t stream);

/*
 * ds4a_index_topk for callers that cannot allocate device memory (the pages
 * describe no such entry point; it has no counterpart in the method).
 *
 * Some callers of this library cannot call cudaMalloc: a host program that
 * links the C ABI without any device allocator of its own, code running
 * inside another runtime that owns all device memory through a fixed pool, or
 * a serving loop that must not take cudaMalloc's implicit device-wide
 * synchronisation in the middle of a step. This call takes the same
 * arguments as ds4a_index_topk minus the workspace and uses a scratch area of
 * DS4A_STATIC_SCRATCH_BYTES that lives inside the library as a static device
 * array. Every GPU that loads the library holds that array until the process
 * exits.
 *
 *  - The caller still passes (and owns) every input and output.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress); make that first call
 *    before any stream capture.
 *  - Requests whose ds4a_workspace_bytes(DS4A_CALL_INDEX_TOPK, ...) exceeds
 *    DS4A_STATIC_SCRATCH_BYTES return DS4A_ERR_WORKSPACE and launch nothing.
 *  - The call allocates nothing and frees nothing.
 *  - All calls share the one array, which keeps the previous call's contents
 *    (everything the call reads back is written first within the call). Calls
 *    that overlap on the GPU (different streams without ordering between
 *    them) race on it: order them.
 */
#define DS4A_STATIC_SCRATCH_BYTES (8u << 20)
ds4a_status ds4a_index_topk_noalloc(const ds4a_layer_cache *cache, uint32_t pos0, uint32_t T,
                                    const void *q_idx, const void *w, uint32_t n_heads,
                                    uint32_t top_k, int32_t *topk, ds4a_stream_t stream);

/*
 * No-allocation variant's wait status: ds4a_workspace_status (below) applied
 * to the static scratch of ds4a_index_topk_noalloc on the current device.
 */
ds4a_status ds4a_noalloc_status(uint32_t *count);

/*
 * Device wait status. Every wait inside the tensor-core kernels (on an
 * mbarrier: TMA and cp.async arrivals, MMA completion, barriers between warps)
 * gives up after 2 s, adds 1 to an error word and lets its thread block wind
 * down, so a stuck call ends instead of hanging the device; the call's outputs
 * are then invalid while the call itself has returned DS4A_OK (launches are
 * asynchronous). The error word is the int32 at byte offset 0 of the workspace
 * of ds4a_index_topk and of the attention calls (every workspace those calls
 * need is at least 256 bytes; calls that need none have no device waits):
 *  - ds4a_index_topk zeroes it at the start of every call, so after a call it
 *    counts that call's timed-out waits;
 *  - the attention calls never zero it (each launch compares it with its value
 *    at the start): it counts the timed-out waits of every call since it was
 *    last zeroed. Zero a new attention workspace once (ds4a_workspace_clear_status
 *    or a memset of the first 4 bytes) before relying on it.
 *
 * ds4a_workspace_status: call after synchronising the stream of the calls
 * that used `ws`. Copies the word to the host (a synchronous 4-byte
 * cudaMemcpy; host memory, such as a mapped workspace or a host copy of the
 * word, is read in place) and returns DS4A_OK when it is zero,
 * DS4A_ERR_TIMEOUT otherwise;
 * *count (may be NULL) receives its value. NULL ws or ws_bytes < 4:
 * DS4A_ERR_WORKSPACE; a failed copy: DS4A_ERR_CUDA.
 * ds4a_workspace_clear_status: zeroes the word, asynchronously on `stream`.
 */
ds4a_status ds4a_workspace_status(const void *ws, size_t ws_bytes, uint32_t *count);
ds4a_status ds4a_workspace_clear_status(void *ws, size_t ws_bytes, ds4a_stream_t stream);

/*
 * Self-test of the bounded waits (the pages have no counterpart): one block of
 * 128 threads waits, through the same bounded-wait code as the kernels but
 * with a limit of limit_us microseconds (1 .. 1,000,000), on a barrier phase
 * that nothing completes. No copy or MMA is in flight. Each waiting thread gives
 * up when the limit has passed (or once another has recorded the timeout),
 * the error word at byte offset 0 of ws grows by at least 1, and the block
 * returns; ds4a_workspace_status then reports DS4A_ERR_TIMEOUT. Asynchronous
 * on `stream`. Errors: DS4A_ERR_WORKSPACE (NULL ws, ws_bytes < 4),
 * DS4A_ERR_ARG (limit out of range), DS4A_ERR_CUDA.
 */
ds4a_status ds4a_wait_selftest(void *ws, size_t ws_bytes, uint32_t limit_us,
                               ds4a_stream_t stream);

/*
 * Cluster size of the tensor-core decode attention (bf16 layers, 64 heads x
 * 512 dims, 64 rotated dims). That kernel spreads each query's 128-row tiles
 * over a thread-block cluster of C CTAs and merges their partial outputs. C
 * is chosen from the tile count (a bound on a query's rows at the call's
 * position: min(pos + 1, cap_raw) window rows plus min(top_k, (pos + 1) / 4)
 * on ratio 4, (pos + 1) / 128 on ratio 128, each at most the compressed rows
 * held) and the device's cluster occupancy, so that the batch runs in one
 * wave; sizes above 8 are used only where the device allows them.
 *
 * ds4a_set_decode_cluster(C): 0 (the default) keeps the automatic choice;
 * 1 .. 16 forces C for every later decode launch of this process (a tuning
 * and test hook), reduced to the call's tile count, and ignored where the
 * device cannot launch that size. DS4A_ERR_ARG for C > 16.
 * ds4a_decode_cluster_size: the C that ds4a_sparse_attn_decode uses for this
 * cache and these arguments at pos = n_tokens - 1 (the token appended last),
 * with the current device current; 0 when the call does not run on that
 * kernel (fp32 layers, other head shapes) or the cache fails its checks.
 */
ds4a_status ds4a_set_decode_cluster(uint32_t C);
uint32_t ds4a_decode_cluster_size(const ds4a_layer_cache *cache, uint32_t n_heads,
                                  uint32_t top_k);

/* Workspace bytes a call needs for these sizes (0: none). */
size_t ds4a_workspace_bytes(int call, const ds4a_layer_cache *cache, uint32_t T,
                            uint32_t n_heads, uint32_t top_k);

/*
 * Host helper: rotation coefficients for positions 0..n_pos-1 into HOST arrays
 * cos_out/sin_out [n_pos][n_rot/2]: theta_i = base^(-2i/n_rot), angle p*theta_i,
 * all in fp64, cos and sin then rounded to fp32 (page §8 tail-only RoPE; the
 * fp64 angle keeps positions up to 1M exact to fp32 resolution).
 */
ds4a_status ds4a_rope_table(double base, uint32_t n_rot, uint32_t n_pos, float *cos_out,
                            float *sin_out);

/*
 * KV-cache bytes of one layer holding ctx tokens for `batch` sequences: the raw
 * window min(128, ctx) rows plus floor(ctx / ratio) compressed rows (c4a rows
 * also carry the indexer row), elem_bytes per element. Summed over the Pro
 * schedule (61 layers, D 512, Di 128, bf16) at 1M tokens this is the vLLM
 * page's 9.62 GiB. The compressor state is not included.
 */
uint64_t ds4a_cache_bytes(uint32_t ratio, uint32_t head_dim, uint32_t index_dim, uint64_t ctx,
                          uint32_t batch, uint32_t elem_bytes);

/* Page §1 schedule: variant 0 = Flash (layers 0-1 ratio 0), 1 = Pro (layers
 * 0-1 ratio 128); then even layers 4, odd layers 128. */
uint32_t ds4a_layer_compress_ratio(int variant, uint32_t il);

/* Page §3: largest prefill chunk for a prompt (4096 beyond 4096 tokens, else 0
 * = the whole prompt at once). */
uint32_t ds4a_prefill_chunk_cap(uint32_t prompt_len);

const char *ds4a_status_string(ds4a_status status);

/* Diagnostic: kernel launches this library has enqueued in this process so
 * far (all threads, all streams; a launch captured into a CUDA graph counts
 * once, at capture). */
uint64_t ds4a_launch_count(void);

/* Diagnostic: text of the last CUDA error a call of this library returned
 * DS4A_ERR_CUDA for ("no error" if none). */
const char *ds4a_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DS4A_H */
