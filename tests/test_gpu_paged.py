"""Paged compressed rows (block_table): every call must give bit-identical
results to the contiguous cache holding the same logical rows, and match the
oracle run on those logical rows (vLLM page, "DeepSeek V4 アテンション
アーキテクチャ": 256-position logical blocks).

Blocks are 256 token positions, so 64 rows on c4a and 2 on c128a. The tables
here are random permutations of a pool larger than the batch needs, and
optionally share a prefix of blocks between sequences (the rows in them are
the same). The contiguous path is the one the oracle parity tests cover."""
import numpy as np
import pytest
import torch

import synth
from helpers import TOL, gpu_cache, np_, oracle_cache, rel_l2, to_dev, to_np
from oracle import layer as olayer
from test_gpu_parity import lib_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make_table(B, max_blocks, n_blocks, seed, share=0):
    perm = np.random.default_rng(seed).permutation(n_blocks)[:B * max_blocks]
    tb = perm.reshape(B, max_blocks).copy()
    if share:
        tb[1:, :share] = tb[0, :share]
    return torch.tensor(tb, dtype=torch.int32, device=DEV)


def share_rows(hist, rows):
    """Make every sequence's first `rows` compressed rows those of sequence 0."""
    for name in ("attn_comp_kv", "index_comp_kv"):
        if name in hist and rows:
            hist[name][1:, :rows] = hist[name][:1, :rows]
    return hist


def run_calls(lib, shape, gc, p0, T, inp):
    """Append, top-k (ratio 4) and attention on one cache; returns outputs."""
    k = shape.top_k
    out = {}
    chunk = None
    if T > 1:
        chunk = torch.empty((gc.batch, T, shape.head_dim), dtype=gc.torch_dtype, device=DEV)
    lib.ds4a_compress_append(gc, p0, T, inp, raw_chunk_out=chunk)
    tk = None
    if shape.ratio == 4:
        tk = torch.full((gc.batch, T, k), -7, dtype=torch.int32, device=DEV)
        ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, T, shape.index_heads, k))
        lib.ds4a_index_topk(gc, p0, T, inp["q_idx"], inp["w"], shape.index_heads, k, tk, ws)
        out["topk"] = tk
    scale = lib.default_scale(shape.head_dim)
    if T == 1:
        o = torch.empty((gc.batch, shape.n_heads, shape.head_dim), dtype=gc.torch_dtype,
                        device=DEV)
        wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_DECODE, 1, shape.n_heads, k))
        lib.ds4a_sparse_attn_decode(gc, p0, inp["q"][:, 0].contiguous(), shape.n_heads,
                                    None if tk is None else tk[:, 0].contiguous(), k, scale, o,
                                    wa)
    else:
        o = torch.empty((gc.batch, T, shape.n_heads, shape.head_dim), dtype=gc.torch_dtype,
                        device=DEV)
        wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_PREFILL, T, shape.n_heads, k))
        lib.ds4a_sparse_attn_prefill_chunk(gc, p0, T, inp["q"], shape.n_heads, chunk, tk, k,
                                           scale, o, wa)
    out["out"] = o
    torch.cuda.synchronize()
    return out


CASES = [
    # ratio, dtype, batch, p0, T, share (blocks)
    (4, "bf16", 4, 8191, 1, 0),       # decode at a row boundary, tensor-core paths
    (4, "bf16", 3, 8190, 1, 3),       # decode off the boundary, shared prefix
    (4, "bf16", 1, 4096, 1024, 0),    # prefill chunk
    (128, "bf16", 2, 65535, 1, 2),    # c128a decode at a boundary (2 rows per block)
    (128, "bf16", 1, 1000, 300, 0),   # c128a prefill chunk
    (4, "f32", 2, 1023, 1, 1),        # exact paths (fp32 indexer, CUDA-core attention)
]


@pytest.mark.parametrize("ratio,dtype,B,p0,T,share", CASES)
def test_paged_equals_contiguous(ratio, dtype, B, p0, T, share):
    lib = lib_()
    shape = synth.LayerShape(ratio=ratio, head_dim=128 if dtype == "f32" else 512,
                             index_dim=32 if dtype == "f32" else 128,
                             index_heads=2 if dtype == "f32" else 64,
                             n_heads=4 if dtype == "f32" else 64,
                             top_k=16 if dtype == "f32" else 512, dtype=dtype)
    rpb = 256 // ratio
    rows_needed = (p0 + T) // ratio
    max_blocks = rows_needed // rpb + 2
    cap = max_blocks * rpb
    n_blocks = B * max_blocks + 7
    wl = synth.Workload("paged", 40 + ratio, B, (shape,), p0, "decode" if T == 1 else "prefill")
    hist = share_rows(synth.cache_history(wl, 0, p0, comp_cap=cap), share * rpb)
    inp = to_dev(synth.step_inputs(wl, 0, p0, T))
    ref = gpu_cache(shape, B, cap, p0 + T + 1, hist, p0)
    table = make_table(B, max_blocks, n_blocks, seed=ratio + p0, share=share)
    from compressed_kv_sparse_gb300 import lib as L
    pg = L.LayerCache(ratio=ratio, head_dim=shape.head_dim, n_rot=shape.n_rot, batch=B,
                      comp_cap=cap, dtype=dtype, base=shape.rope_base, rope_max_pos=p0 + T + 1,
                      index_dim=shape.index_dim, index_rot=shape.index_rot,
                      cap_raw=shape.cap_raw, device=DEV, block_table=table, n_blocks=n_blocks)
    pg.load_state({k: v.to(DEV) for k, v in hist.items()}, p0)
    a = run_calls(lib, shape, ref, p0, T, inp)
    b = run_calls(lib, shape, pg, p0, T, inp)
    for name in a:
        assert torch.equal(a[name], b[name]), name
    n = (p0 + T) // ratio
    for name in ("attn_comp_kv", "index_comp_kv", "index_norm"):
        if getattr(ref, name) is None:
            continue
        assert torch.equal(ref.logical(name)[:, :n], pg.logical(name)[:, :n]), name
    for name in ("raw_kv", "attn_state_kv", "attn_state_score", "index_state_kv",
                 "index_state_score", "index_norm_max"):
        if getattr(ref, name) is not None:
            assert torch.equal(getattr(ref, name), getattr(pg, name)), name
    # the paged results against the oracle on the same logical rows (shared
    # prefix blocks included)
    oc = oracle_cache(shape, hist, p0)
    k = shape.top_k
    if T == 1:
        o_ref, tk_ref = olayer.decode_step(oc, p0, to_np(inp), k)
        got_o = np_(b["out"])
        got_tk = None if tk_ref is None else b["topk"][:, 0].cpu().numpy()
    else:
        o_ref, tk_ref = olayer.prefill_chunk(oc, p0, to_np(inp), k)
        got_o = np_(b["out"])
        got_tk = None if tk_ref is None else b["topk"].cpu().numpy()
    if tk_ref is not None:
        assert np.array_equal(got_tk, tk_ref)
    assert rel_l2(got_o, o_ref) <= TOL[dtype]
    for name in ("attn_comp_kv", "index_comp_kv"):
        if getattr(pg, name) is not None:
            assert rel_l2(np_(pg.logical(name))[:, :n], getattr(oc, name)[:, :n]) <= TOL[dtype], name
    for name in ("attn_state_kv", "attn_state_score", "index_state_kv", "index_state_score"):
        if getattr(pg, name) is not None:
            assert np.array_equal(np_(getattr(pg, name)), getattr(oc, name)), name
