"""Every cluster size of the tensor-core decode attention against the oracle.

The decode kernel spreads a query's 128-row tiles over a thread-block cluster
of C CTAs (C up to 16; above 8 the sizes are non-portable) and merges the
partial outputs. These cases make the automatic choice run over c128a decode
batches whose queries have 2, 6, 9, 12 and 16 tiles at 1, 8 and 32 sequences,
and force each C from 1 to 16 on a 16-tile batch; each output is compared
with the oracle ("【#3】ds4.c を読み解く" §7; vLLM page: c128a layers attend
every visible compressed row)."""
import numpy as np
import pytest
import torch

import synth
from helpers import TOL, gpu_cache, np_, oracle_cache, rel_l2
from oracle import layer as olayer

pytestmark = pytest.mark.gpu
DEV = "cuda"


def c128a_decode(tiles: int, B: int, seed: int, force: int = 0, check=None):
    """One c128a decode step whose query has `tiles` tiles of 128 rows (the
    window plus 128 (tiles - 1) - 10 compressed rows). Returns the cluster
    size the call used."""
    from compressed_kv_sparse_gb300 import lib
    shape = synth.LayerShape(ratio=128)
    n_comp = 128 * (tiles - 1) - 10
    p = 128 * n_comp + 3                      # (p + 1) // 128 == n_comp, no emission
    wl = synth.Workload("clu", seed, B, (shape,), p, "decode")
    hist = synth.cache_history(wl, 0, p + 1, comp_cap=n_comp)
    q = synth.normal((B, shape.n_heads, shape.head_dim), seed, "q", dtype="bf16")
    gc = gpu_cache(shape, B, n_comp, p + 2, hist, p + 1)
    out = torch.empty((B, shape.n_heads, shape.head_dim), dtype=torch.bfloat16, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_DECODE, 1, shape.n_heads, 0))
    lib.ds4a_set_decode_cluster(force)
    try:
        C = lib.ds4a_decode_cluster_size(gc, shape.n_heads, 0)
        lib.ds4a_sparse_attn_decode(gc, p, q.to(DEV), shape.n_heads, None, 0,
                                    1 / np.sqrt(shape.head_dim), out, ws)
        torch.cuda.synchronize()
    finally:
        lib.ds4a_set_decode_cluster(0)
    assert lib.ds4a_workspace_status(ws) == 0
    oc = oracle_cache(shape, hist, p + 1)
    seqs = check if check is not None else range(B)
    qs = [(b, 0) for b in seqs]
    ref = olayer.attention(oc, p, np_(q)[:, None], None, None, queries=qs)
    got = np.stack([np_(out[b]) for b in seqs])
    want = np.stack([ref[b, 0] for b in seqs])
    e = rel_l2(got, want)
    assert e <= TOL["bf16"], (tiles, B, C, e)
    return C


@pytest.mark.parametrize("tiles", [2, 6, 9, 12, 16])
@pytest.mark.parametrize("B", [1, 8, 32])
def test_decode_cluster_automatic(tiles, B):
    C = c128a_decode(tiles, B, seed=70 + tiles, check=(0, 13, 31) if B == 32 else None)
    print(f"tiles {tiles} batch {B}: cluster {C}")
    assert 1 <= C <= min(tiles, 16)
    if B == 1:
        assert C == tiles          # one query: every tile gets its own CTA


@pytest.mark.parametrize("C", list(range(1, 17)))
def test_decode_cluster_forced(C):
    used = c128a_decode(16, 2, seed=90 + C, force=C)
    assert used == C
