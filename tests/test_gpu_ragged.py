"""Ragged batches (seq_pos): every sequence of one call at its own
position, for decode steps and prefill chunks. Each sequence must match the oracle run on that sequence alone at
its position: exact top-k, attention within the bf16 bound, state
bit-identical and rows within the bound."""
import numpy as np
import pytest
import torch

import synth
from helpers import TOL, gpu_cache, np_, oracle_cache, rel_l2, to_dev
from oracle import layer as olayer
from test_gpu_parity import lib_

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {4: [8191, 8000, 5003, 700], 128: [65535, 40000, 1023, 200]}


@pytest.mark.parametrize("ratio", [4, 128])
def test_ragged_decode_matches_oracle_per_sequence(ratio):
    lib = lib_()
    shape = synth.LayerShape(ratio=ratio)
    pos = CASES[ratio]
    B, P = len(pos), max(pos)
    cap = (P + 1) // ratio + 1
    hists = [synth.cache_history(synth.Workload(f"ragged{b}", 60 + b, 1, (shape,), pos[b],
                                                "decode"), 0, pos[b], comp_cap=cap)
             for b in range(B)]
    hist = {k: torch.cat([h[k] for h in hists]) for k in hists[0]}
    inp = synth.step_inputs(synth.Workload("ragged", 70, B, (shape,), P, "decode"), 0, P, 1)
    dinp = to_dev(inp)
    gc = gpu_cache(shape, B, cap, P + 2, hist, P)
    seq_pos = torch.tensor(pos, dtype=torch.int32, device=DEV)
    gc.set_seq_pos(seq_pos)
    lib.ds4a_compress_append(gc, P, 1, dinp)
    k = shape.top_k
    topk = None
    if ratio == 4:
        topk = torch.empty((B, k), dtype=torch.int32, device=DEV)
        ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, 1, shape.index_heads, k))
        lib.ds4a_index_topk(gc, P, 1, dinp["q_idx"], dinp["w"], shape.index_heads, k, topk, ws)
    out = torch.empty((B, shape.n_heads, shape.head_dim), dtype=torch.bfloat16, device=DEV)
    wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_DECODE, 1, shape.n_heads, k))
    lib.ds4a_sparse_attn_decode(gc, P, dinp["q"][:, 0].contiguous(), shape.n_heads, topk, k,
                                1 / np.sqrt(shape.head_dim), out, wa)
    torch.cuda.synchronize()
    seq_pos_host = pos
    for b in range(B):
        p = seq_pos_host[b]
        oc = oracle_cache(shape, {n: t[b:b + 1] for n, t in hist.items()}, p)
        one = {n: (np_(t[b:b + 1]) if t.dim() > 2 else np_(t)) for n, t in inp.items()}
        o_ref, tk_ref = olayer.decode_step(oc, p, one, k)
        if ratio == 4:
            assert np.array_equal(topk[b].cpu().numpy(), tk_ref[0]), b
        assert rel_l2(np_(out[b]), o_ref[0]) <= TOL["bf16"], b
        for name in ("attn_state_kv", "attn_state_score", "index_state_kv", "index_state_score"):
            g = getattr(gc, name)
            if g is not None:
                assert np.array_equal(np_(g[b:b + 1]), getattr(oc, name)), (b, name)
        n = oc.n_comp
        for name in ("raw_kv", "attn_comp_kv", "index_comp_kv"):
            g = getattr(gc, name)
            if g is not None:
                o = getattr(oc, name)
                m = min(n, o.shape[1]) if name != "raw_kv" else o.shape[1]
                assert rel_l2(np_(g[b:b + 1])[:, :m], o[:, :m]) <= TOL["bf16"], (b, name)


PREFILL = {4: [4093, 3000, 1025, 64], 128: [4000, 2047, 1000, 130], 0: [500, 77, 3, 0]}


@pytest.mark.parametrize("ratio", [4, 128, 0])
def test_ragged_prefill_matches_oracle_per_sequence(ratio):
    """A 300-token chunk per sequence, each sequence starting at its own
    position (seq_pos): append with the chunk's compressor boundaries at each
    sequence's positions, per-query top-k and chunk attention over each
    sequence's own window, then the window commit. Each sequence must match the
    oracle's prefill of that sequence alone: exact top-k, outputs within the
    bf16 bound, state bit-identical, rows within the bound, window rows equal."""
    lib = lib_()
    shape = synth.LayerShape(ratio=ratio)
    pos = PREFILL[ratio]
    B, T, P = len(pos), 300, max(pos)
    cap = (P + T) // ratio + 1 if ratio else 0
    wls = [synth.Workload(f"rgp{b}", 80 + b, 1, (shape,), pos[b], "prefill") for b in range(B)]
    hists = [synth.cache_history(wls[b], 0, pos[b], comp_cap=cap) if pos[b]
             else synth.empty_history(wls[b], 0, cap) for b in range(B)]
    hist = {k: torch.cat([h[k] for h in hists]) for k in hists[0]}
    inp = synth.step_inputs(synth.Workload("rgp", 90, B, (shape,), P, "prefill"), 0, P, T)
    dinp = to_dev(inp)
    gc = gpu_cache(shape, B, cap, P + T + 1, hist, P)
    gc.set_seq_pos(torch.tensor(pos, dtype=torch.int32, device=DEV))
    chunk = torch.empty((B, T, shape.head_dim), dtype=torch.bfloat16, device=DEV)
    lib.ds4a_compress_append(gc, P, T, dinp, raw_chunk_out=chunk)
    k = shape.top_k
    topk = None
    if ratio == 4:
        topk = torch.empty((B, T, k), dtype=torch.int32, device=DEV)
        ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, T, shape.index_heads, k))
        lib.ds4a_index_topk(gc, P, T, dinp["q_idx"], dinp["w"], shape.index_heads, k, topk, ws)
    out = torch.empty((B, T, shape.n_heads, shape.head_dim), dtype=torch.bfloat16, device=DEV)
    wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_PREFILL, T, shape.n_heads, k))
    lib.ds4a_sparse_attn_prefill_chunk(gc, P, T, dinp["q"], shape.n_heads, chunk, topk, k,
                                       1 / np.sqrt(shape.head_dim), out, wa)
    torch.cuda.synchronize()
    for b in range(B):
        p0 = pos[b]
        oc = oracle_cache(shape, {n: t[b:b + 1] for n, t in hist.items()}, p0)
        one = {n: (np_(t[b:b + 1]) if t.dim() > 2 else np_(t)) for n, t in inp.items()}
        o_ref, tk_ref = olayer.prefill_chunk(oc, p0, one, k)
        if ratio == 4:
            assert np.array_equal(topk[b].cpu().numpy(), tk_ref[0]), b
        assert rel_l2(np_(out[b]), o_ref[0]) <= TOL["bf16"], b
        for name in ("attn_state_kv", "attn_state_score", "index_state_kv", "index_state_score"):
            g = getattr(gc, name)
            if g is not None:
                assert np.array_equal(np_(g[b:b + 1]), getattr(oc, name)), (b, name)
        for name in ("attn_comp_kv", "index_comp_kv"):
            g = getattr(gc, name)
            if g is not None:
                n = oc.n_comp
                assert rel_l2(np_(g[b:b + 1])[:, :n], getattr(oc, name)[:, :n]) <= TOL["bf16"], \
                    (b, name)
        assert rel_l2(np_(gc.raw_kv[b:b + 1]), oc.raw_kv) <= TOL["bf16"], b
