"""Ragged decode batches (seq_pos): every sequence of one call at its own
position. Each sequence must match the oracle run on that sequence alone at
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


def test_ragged_refuses_chunks():
    """seq_pos is for decode steps: calls with T > 1 are refused before any launch."""
    lib = lib_()
    shape = synth.LayerShape(ratio=4)
    gc = gpu_cache(shape, 2, 64, 300)
    gc.set_seq_pos(torch.zeros(2, dtype=torch.int32, device=DEV))
    inp = to_dev(synth.step_inputs(synth.Workload("rgc", 71, 2, (shape,), 0, "prefill"), 0, 0, 8))
    chunk = torch.empty((2, 8, 512), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(lib.Ds4aError):
        lib.ds4a_compress_append(gc, 0, 8, inp, raw_chunk_out=chunk)
