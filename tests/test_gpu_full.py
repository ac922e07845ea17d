"""GPU parity at the full workload sizes, in the launch configuration the
benchmark uses, on outputs the oracle can compute one by one (sampled
sequences / queries), plus the tensor-core indexer path on ragged and tied
inputs."""
import numpy as np
import pytest
import torch

import synth
from helpers import TOL, gpu_cache, np_, oracle_cache, rel_l2
from test_gpu_parity import compare_cache
from oracle import layer as olayer
from test_gpu_parity import lib_, run_attn, run_index

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_index_tc_prefill_ragged():
    """Flash indexer shape, 37 queries (not a multiple of the 4-query MMA
    group), visible counts above k, two sequences."""
    run_index(lib_(), synth.LayerShape(ratio=4), 2, 3001, 37, seed=31)


def test_index_tc_grid_ties():
    """Flash indexer shape on 1/8-grid inputs: many exact ties at the cut."""
    run_index(lib_(), synth.LayerShape(ratio=4), 2, 4000, 6, seed=32, grid=True)


def test_index_tc_all_rows_tied_fallback():
    """Every key row identical: all 16,384 scores tie, the candidate set
    overflows and the selection falls back to the full pass; the kept rows
    must be the 512 lowest indices."""
    lib = lib_()
    shape = synth.LayerShape(ratio=4)
    B, p = 2, 65536
    wl = synth.Workload("ties", 34, B, (shape,), p + 1, "decode")
    cap = (p + 1) // 4 + 1
    hist = synth.cache_history(wl, 0, p + 1, comp_cap=cap)
    hist["index_comp_kv"][:] = hist["index_comp_kv"][:, :1]
    q_idx = synth.normal((B, 1, 64, 128), 34, "q", dtype="bf16")
    w = synth.normal((B, 1, 64), 34, "w", dtype="bf16")
    gc = gpu_cache(shape, B, cap, p + 2, hist, p + 1)
    topk = torch.empty((B, 1, shape.top_k), dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, 1, 64, shape.top_k))
    lib.ds4a_index_topk(gc, p, 1, q_idx.to(DEV), w.to(DEV), 64, shape.top_k, topk, ws)
    torch.cuda.synchronize()
    oc = oracle_cache(shape, hist, p + 1)
    ref = olayer.index_topk(oc, p, np_(q_idx), np_(w), shape.top_k)
    assert np.array_equal(topk.cpu().numpy(), ref)
    assert np.array_equal(ref[0, 0], np.arange(shape.top_k))


def test_index_tc_prefill_visibility_edges():
    """Chunk starting below 4 k (some queries see <= k rows, the rest more)."""
    run_index(lib_(), synth.LayerShape(ratio=4), 1, 2030, 40, seed=33)


def test_c4a_decode_full_size_sampled():
    """32 sequences at 65,536 tokens (16,384 rows each): exact top-k and
    attention for sampled sequences."""
    lib = lib_()
    wl = synth.C4A_DECODE
    s = wl.layers[0]
    B, p = wl.batch, wl.context
    cap = (p + 1) // 4 + 1
    hist = synth.cache_history(wl, 0, p, comp_cap=cap, device=DEV)
    inp = {k: v.contiguous() for k, v in synth.step_inputs(wl, 0, p, 1, device=DEV).items()}
    gc = gpu_cache(s, B, cap, p + 2, hist, p)
    lib.ds4a_compress_append(gc, p, 1, inp)
    k = s.top_k
    topk = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, 1, s.index_heads, k))
    lib.ds4a_index_topk(gc, p, 1, inp["q_idx"], inp["w"], s.index_heads, k, topk, ws)
    out = torch.empty((B, s.n_heads, s.head_dim), dtype=torch.bfloat16, device=DEV)
    wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_DECODE, 1, s.n_heads, k))
    lib.ds4a_sparse_attn_decode(gc, p, inp["q"][:, 0].contiguous(), s.n_heads, topk, k,
                                1 / np.sqrt(s.head_dim), out, wa)
    torch.cuda.synchronize()
    for b in (0, 13, 31):
        one = {n: t[b:b + 1].cpu() for n, t in hist.items()}
        oc = oracle_cache(s, one, p)
        o_ref, tk_ref = olayer.decode_step(oc, p, {n: np_(t[b:b + 1]) if t.dim() > 2 else np_(t)
                                                   for n, t in inp.items()}, k)
        assert np.array_equal(topk[b].cpu().numpy(), tk_ref[0]), b
        assert rel_l2(np_(out[b]), o_ref[0]) <= TOL["bf16"], b


def prefill_samples(T: int):
    """Queries checked in a full chunk: every 16th, plus the four positions of
    each residue mod 4 at both ends of the chunk."""
    return sorted(set(range(0, T, 16)) | set(range(4)) | set(range(T - 4, T)))


def test_c4a_prefill_full_size_sampled():
    """The 4096-token chunk at 28,672 over a cache built from the 28,672
    earlier seeded tokens: on the GPU by seven 4096-token chunks of the real
    prefill path (append, top-k, chunk attention with the window commit), in
    the oracle by its own compressor from an empty cache. The caches must
    agree before the chunk (state bit-identical, rows within the bf16 bound)
    and the chunk's top-k lists and outputs must match on sampled queries
    ("【#3】ds4.c を読み解く" §3: chunks keep absolute positions)."""
    lib = lib_()
    wl = synth.C4A_PREFILL
    s = wl.layers[0]
    p0, T = wl.context, wl.chunk
    cap = (p0 + T) // 4 + 1
    k, scale = s.top_k, 1 / np.sqrt(s.head_dim)
    gc = gpu_cache(s, 1, cap, p0 + T + 1, synth.empty_history(wl, 0, cap, device=DEV), 0)
    lib.ds4a_cache_reset(gc)
    oc = oracle_cache(s, synth.empty_history(wl, 0, cap), 0)
    comp_keys = ("raw_kv_in", "attn_cand", "attn_score", "idx_cand", "idx_score", "ape_attn",
                 "gamma_attn", "ape_idx", "gamma_idx")
    chunk = torch.empty((1, T, s.head_dim), dtype=torch.bfloat16, device=DEV)
    topk = torch.empty((1, T, k), dtype=torch.int32, device=DEV)
    out = torch.empty((1, T, s.n_heads, s.head_dim), dtype=torch.bfloat16, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, T, s.index_heads, k))
    wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_PREFILL, T, s.n_heads, k))
    for p in range(0, p0 + 1, T):
        inp = {n: v.contiguous() for n, v in synth.step_inputs(wl, 0, p, T, device=DEV).items()}
        if p == p0:
            ring0 = np_(gc.raw_kv)
            compare_cache(gc, oc, "bf16", "history")
        lib.ds4a_compress_append(gc, p, T, inp, raw_chunk_out=chunk)
        lib.ds4a_index_topk(gc, p, T, inp["q_idx"], inp["w"], s.index_heads, k, topk, ws)
        lib.ds4a_sparse_attn_prefill_chunk(gc, p, T, inp["q"], s.n_heads, chunk, topk, k,
                                           scale, out, wa)
        ninp = {n: np_(inp[n]) for n in comp_keys}
        rows = olayer.compress_append(oc, p, ninp, chunk=True)
        if p < p0:
            olayer.commit_ring(oc, p, rows)
    torch.cuda.synchronize()
    assert lib.ds4a_workspace_status(ws) == 0 and lib.ds4a_workspace_status(wa) == 0
    assert rel_l2(np_(chunk), rows) <= TOL["bf16"]
    assert oc.n_comp == 8192 and gc.n_tokens == p0 + T
    assert rel_l2(np_(gc.attn_comp_kv)[:, 7168:8192], oc.attn_comp_kv[:, 7168:8192]) <= TOL["bf16"]
    qs = [(0, t) for t in prefill_samples(T)]
    tk_ref = olayer.index_topk(oc, p0, np_(inp["q_idx"]), np_(inp["w"]), k, queries=qs)
    got_tk = topk.cpu().numpy()
    for b, t in qs:
        assert np.array_equal(got_tk[b, t], tk_ref[b, t]), t
    o_ref = olayer.attention(oc, p0, np_(inp["q"]), tk_ref, None, ring=ring0, chunk_rows=rows,
                             queries=qs)
    got = np.stack([np_(out[b, t]) for b, t in qs])
    ref = np.stack([o_ref[b, t] for b, t in qs])
    assert rel_l2(got, ref) <= TOL["bf16"]


def test_c128a_decode_full_size():
    """One sequence at 65,536 tokens on a ratio-128 layer: 128 window rows plus
    all 512 compressed rows."""
    run_attn(lib_(), synth.LayerShape(ratio=128), 1, 65536, 1, 65536, seed=41)


def test_c4a_decode_attn_b32():
    """Attention with random top-k lists at the 32-sequence decode shape."""
    run_attn(lib_(), synth.LayerShape(ratio=4), 32, 65536, 1, 65536, seed=42,
             queries=[(0, 0), (17, 0), (31, 0)])


@pytest.mark.parametrize("ratio,p0,T", [(4, 300, 50), (128, 1000, 70), (0, 60, 100), (4, 0, 40)])
def test_attn_tc_prefill(ratio, p0, T):
    """Tensor-core chunk attention (64 heads x 512): window across the old ring
    and the chunk, padded / ending top-k lists, ring commit."""
    run_attn(lib_(), synth.LayerShape(ratio=ratio), 2, p0, T, p0, topk_mode="pad", seed=43)


@pytest.mark.parametrize("ratio,p0,T", [(4, 700, 20), (128, 5000, 3)])
def test_attn_tc_prefill_running_max_raised(ratio, p0, T):
    """Scale 1.0 spreads the scores over hundreds of units, so later rows
    exceed the first row's score by far more than 2^8: the running max must be
    raised and the partial output and sums rescaled."""
    run_attn(lib_(), synth.LayerShape(ratio=ratio), 2, p0, T, p0, seed=44, scale=1.0)


@pytest.mark.parametrize("ratio,p", [(4, 900), (128, 65536), (0, 40)])
def test_attn_tc_decode_running_max_raised(ratio, p):
    run_attn(lib_(), synth.LayerShape(ratio=ratio), 3, p, 1, p, topk_mode="pad", seed=45,
             scale=1.0)
