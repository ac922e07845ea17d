"""Per-layer compression schedule and KV-cache sizes.

* ``layer_compress_ratio`` — "【#3】ds4.c を読み解く" §1 (per-layer ratio table):
  Flash: layers 0-1 uncompressed, then even layers ratio 4, odd layers ratio 128;
  Pro: layers 0-1 ratio 128, then the same alternation.
* ``raw_capacity`` — same page §2: the raw sliding window holds DS4_N_SWA = 128
  rows, capped by the context size.
* ``prefill_chunk_cap`` — same page §3: prompts longer than 4096 tokens are
  prefilled in 4096-token chunks.
* ``kv_cache_bytes`` — bytes of the per-layer KV cache: raw window rows plus
  compressed rows (c4a layers also hold the indexer rows). vLLM's page
  ("DeepSeek V4 アテンションアーキテクチャ") gives 9.62 GiB per 1M-token
  sequence in bf16 for the Pro model; the compressor's recurrent state is not
  part of that figure and is not counted here.
"""

FLASH, PRO = 0, 1
N_SWA = 128


def layer_compress_ratio(variant: int, il: int) -> int:
    if il < 2:
        return 0 if variant == FLASH else 128
    return 4 if il % 2 == 0 else 128


def raw_capacity(ctx: int) -> int:
    return min(N_SWA, ctx)


def prefill_chunk_cap(prompt_len: int) -> int:
    """Largest chunk the prefill graph takes (0: the whole prompt in one go)."""
    return 4096 if prompt_len > 4096 else 0


def n_comp_rows(ratio: int, n_tokens: int) -> int:
    """Compressed rows held after n_tokens tokens: one per completed window."""
    return 0 if ratio == 0 else n_tokens // ratio


def kv_cache_bytes(ratio: int, head_dim: int, index_dim: int, ctx: int, batch: int,
                   elem_bytes: int) -> int:
    raw = raw_capacity(ctx) * head_dim
    comp = n_comp_rows(ratio, ctx) * (head_dim + (index_dim if ratio == 4 else 0))
    return batch * (raw + comp) * elem_bytes


def stack_kv_bytes(variant: int, n_layers: int, head_dim: int, index_dim: int, ctx: int,
                   batch: int, elem_bytes: int) -> int:
    return sum(kv_cache_bytes(layer_compress_ratio(variant, il), head_dim, index_dim, ctx,
                              batch, elem_bytes) for il in range(n_layers))
