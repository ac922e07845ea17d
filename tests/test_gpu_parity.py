"""GPU parity: each C-ABI call against the CPU oracle on identical seeded inputs.

Top-k lists must be identical (exact sets, ascending, -1 padded); continuous
outputs within relative L2 1e-5 (fp32 layers) or 1e-2 (bf16 layers); the
compressor state (copies of the inputs) must be bit-identical.
"""
import numpy as np
import pytest
import torch

import synth
from helpers import TOL, gpu_cache, np_, oracle_cache, rel_l2, to_dev, to_np
from oracle import layer as olayer

pytestmark = pytest.mark.gpu

DEV = "cuda"


def lib_():
    from compressed_kv_sparse_gb300 import lib
    lib.load()
    return lib


def wl_with(base: synth.Workload, batch=None, **shape_kw):
    s = base.layers[0].replace(**shape_kw) if shape_kw else base.layers[0]
    return synth.Workload(name=base.name + "_t", seed=base.seed + 100, batch=batch or base.batch,
                          layers=(s,), context=base.context, mode=base.mode, hidden=0)


def compare_cache(gc, oc, dtype, what=""):
    for name in ("attn_state_kv", "attn_state_score", "index_state_kv", "index_state_score"):
        g = getattr(gc, name)
        if g is None:
            continue
        assert np.array_equal(np_(g), getattr(oc, name)), f"{what} {name}"
    for name in ("raw_kv", "attn_comp_kv", "index_comp_kv"):
        g = getattr(gc, name)
        if g is None:
            continue
        o = getattr(oc, name)
        n = o.shape[1]
        e = rel_l2(np_(g)[:, :n], o)
        assert e <= TOL[dtype], f"{what} {name} rel L2 {e}"


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("ratio,dtype,p", [(4, "f32", 255), (4, "f32", 256), (4, "bf16", 1027),
                                           (128, "bf16", 65535), (128, "f32", 300),
                                           (0, "bf16", 70)])
def test_append_decode_step(ratio, dtype, p):
    """One token at a ratio boundary (p % 4 == 3, p % 128 == 127) and off it."""
    lib = lib_()
    shape = synth.LayerShape(ratio=ratio, head_dim=128 if dtype == "f32" else 512,
                             index_dim=32 if dtype == "f32" else 128,
                             index_heads=2, n_heads=4, dtype=dtype)
    wl = synth.Workload("app", 7, 3, (shape,), p, "decode")
    cap = max(1, (p + 1) // ratio) if ratio else 0
    hist = synth.cache_history(wl, 0, p, comp_cap=cap)
    inp = synth.step_inputs(wl, 0, p, 1)
    gc = gpu_cache(shape, 3, cap, p + 2, hist, p)
    lib.ds4a_compress_append(gc, p, 1, to_dev(inp))
    torch.cuda.synchronize()
    oc = oracle_cache(shape, hist, p)
    olayer.compress_append(oc, p, to_np(inp), chunk=False)
    assert gc.n_tokens == p + 1
    compare_cache(gc, oc, dtype, f"r{ratio} p{p}")


@pytest.mark.parametrize("ratio,dtype,p0,T", [(4, "bf16", 0, 37), (4, "f32", 2, 3), (4, "bf16", 1021, 300),
                                              (128, "bf16", 200, 300), (128, "f32", 0, 129),
                                              (0, "bf16", 5, 200)])
def test_append_chunk(ratio, dtype, p0, T):
    """A chunk of T tokens (chunk mode: ring untouched, rows to raw_chunk_out),
    ragged with respect to the ratio, from an existing history."""
    lib = lib_()
    shape = synth.LayerShape(ratio=ratio, head_dim=128 if dtype == "f32" else 512,
                             index_dim=32 if dtype == "f32" else 128, dtype=dtype)
    wl = synth.Workload("appc", 8, 2, (shape,), p0, "prefill")
    cap = (p0 + T) // ratio + 1 if ratio else 0
    hist = synth.cache_history(wl, 0, p0, comp_cap=cap) if p0 else synth.empty_history(wl, 0, cap)
    inp = synth.step_inputs(wl, 0, p0, T)
    gc = gpu_cache(shape, 2, cap, p0 + T + 1, hist, p0)
    chunk = torch.empty((2, T, shape.head_dim), dtype=gc.torch_dtype, device=DEV)
    lib.ds4a_compress_append(gc, p0, T, to_dev(inp), raw_chunk_out=chunk)
    torch.cuda.synchronize()
    oc = oracle_cache(shape, hist, p0)
    rows = olayer.compress_append(oc, p0, to_np(inp), chunk=True)
    compare_cache(gc, oc, dtype, f"r{ratio} p0{p0} T{T}")
    assert rel_l2(np_(chunk), rows) <= TOL[dtype]


def test_append_chunked_equals_one_call_on_gpu_and_oracle():
    """4096-token chunk at 28,672 over a history that was itself appended on the
    GPU in 4096-token chunks from position 24,576: row counts 7,168 -> 8,192,
    state continuity across the boundary."""
    lib = lib_()
    shape = synth.LayerShape(ratio=4)
    wl = synth.Workload("cont", 9, 1, (shape,), 24576, "prefill")
    p_start, cap = 24576, 8192
    hist = synth.cache_history(wl, 0, p_start, comp_cap=cap)
    gc = gpu_cache(shape, 1, cap, 32769, hist, p_start)
    oc = oracle_cache(shape, hist, p_start)
    for p0 in (24576, 28672):
        inp = synth.step_inputs(wl, 0, p0, 4096)
        chunk = torch.empty((1, 4096, 512), dtype=torch.bfloat16, device=DEV)
        lib.ds4a_compress_append(gc, p0, 4096, to_dev(inp), raw_chunk_out=chunk)
        rows = olayer.compress_append(oc, p0, to_np(inp), chunk=True)
        torch.cuda.synchronize()
        assert rel_l2(np_(chunk), rows) <= TOL["bf16"]
    assert oc.n_comp == 8192 and gc.n_tokens == 32768
    compare_cache(gc, oc, "bf16", "continuity")


@pytest.mark.parametrize("T", [1, 37])
def test_append_lanes_on_two_streams_equal_one_call(T):
    """The indexer lane on one stream and the raw rows plus attention lane on
    another (ds4a_compress_append_lanes, then n_tokens set by the caller) leave
    exactly the cache of one ds4a_compress_append, and that cache matches the
    oracle's append (vLLM page, "GPU 計算飽和": multi-stream partitioning)."""
    lib = lib_()
    shape = synth.LayerShape(ratio=4)
    p0 = 1023 if T == 1 else 1021
    wl = synth.Workload("lanes", 14, 2, (shape,), p0, "decode" if T == 1 else "prefill")
    cap = (p0 + T) // 4 + 1
    hist = synth.cache_history(wl, 0, p0, comp_cap=cap)
    inp = to_dev(synth.step_inputs(wl, 0, p0, T))
    ref = gpu_cache(shape, 2, cap, p0 + T + 1, hist, p0)
    got = gpu_cache(shape, 2, cap, p0 + T + 1, hist, p0)
    mk = lambda: torch.empty((2, T, 512), dtype=torch.bfloat16, device=DEV) if T > 1 else None
    chunk_ref, chunk_got = mk(), mk()
    lib.ds4a_compress_append(ref, p0, T, inp, raw_chunk_out=chunk_ref)
    main, aux = torch.cuda.current_stream(), torch.cuda.Stream()
    aux.wait_stream(main)
    with torch.cuda.stream(aux):
        lib.ds4a_compress_append_lanes(got, p0, T, lib.LANE_INDEX, inp)
    lib.ds4a_compress_append_lanes(got, p0, T, lib.LANE_RAW | lib.LANE_ATTN, inp,
                                   raw_chunk_out=chunk_got)
    main.wait_stream(aux)
    assert got.n_tokens == p0
    got.n_tokens = p0 + T
    torch.cuda.synchronize()
    for name in ("raw_kv", "attn_comp_kv", "attn_state_kv", "attn_state_score", "index_comp_kv",
                 "index_state_kv", "index_state_score", "index_norm", "index_norm_max"):
        assert torch.equal(getattr(ref, name), getattr(got, name)), name
    if T > 1:
        assert torch.equal(chunk_ref, chunk_got)
    # and the two-stream cache against the oracle directly
    oc = oracle_cache(shape, hist, p0)
    rows = olayer.compress_append(oc, p0, to_np(inp), chunk=T > 1)
    compare_cache(got, oc, "bf16", f"two streams T{T}")
    if T > 1:
        assert rel_l2(np_(chunk_got), rows) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_index_norms_written_at_append(dtype):
    """Every indexer row appended (chunk and decode paths) gets an upper bound
    of its Euclidean norm, within 1e-4, in index_norm and the running maximum
    in index_norm_max; ds4a_index_norms recomputes such bounds from the rows
    (the certified top-k bounds its tensor-core scores with them)."""
    lib = lib_()
    shape = synth.LayerShape(ratio=4, head_dim=128 if dtype == "f32" else 512,
                             index_dim=32 if dtype == "f32" else 128, dtype=dtype)
    wl = synth.Workload("norm", 12, 2, (shape,), 0, "prefill")
    T, n_dec = 301, 9
    cap = (T + n_dec) // 4 + 1
    gc = gpu_cache(shape, 2, cap, T + n_dec + 1, synth.empty_history(wl, 0, cap), 0)
    chunk = torch.empty((2, T, shape.head_dim), dtype=gc.torch_dtype, device=DEV)
    lib.ds4a_compress_append(gc, 0, T, to_dev(synth.step_inputs(wl, 0, 0, T)),
                             raw_chunk_out=chunk)
    for p in range(T, T + n_dec):
        lib.ds4a_compress_append(gc, p, 1, to_dev(synth.step_inputs(wl, 0, p, 1)))
    torch.cuda.synchronize()
    n = (T + n_dec) // 4
    exact = torch.linalg.vector_norm(gc.index_comp_kv[:, :n].double(), dim=-1)

    def upper_bound_within_1e4(got):   # the error bound needs ||k|| <= norm <= (1 + 1e-4) ||k||
        got = got.double()
        return bool((got >= exact).all()) and bool((got <= exact * (1 + 1e-4)).all())

    assert upper_bound_within_1e4(gc.index_norm[:, :n])
    appended = gc.index_norm[:, :n].clone()
    assert torch.equal(gc.index_norm_max.view(torch.float32), appended.max(dim=1).values)
    lib.ds4a_index_norms(gc)
    torch.cuda.synchronize()
    assert upper_bound_within_1e4(gc.index_norm[:, :n])
    assert torch.equal(gc.index_norm_max.view(torch.float32), gc.index_norm[:, :n].max(dim=1).values)


# ------------------------------------------------------------------ indexer

def run_index(lib, shape, B, p0, T, seed=11, grid=False, queries=None):
    wl = synth.Workload("idx", seed, B, (shape,), p0 + T, "prefill")
    cap = (p0 + T) // 4 + 1
    hist = synth.cache_history(wl, 0, p0 + T, comp_cap=cap)
    q_idx = synth.normal((B, T, shape.index_heads, shape.index_dim), seed, "q", dtype=shape.dtype)
    w = synth.normal((B, T, shape.index_heads), seed, "w", dtype=shape.dtype)
    if grid:
        hist["index_comp_kv"] = synth.grid_values(hist["index_comp_kv"].shape, seed, "gk",
                                                  dtype=shape.dtype)
        q_idx = synth.grid_values(q_idx.shape, seed, "gq", dtype=shape.dtype)
        w = synth.grid_values(w.shape, seed, "gw", lo=0, hi=4, dtype=shape.dtype)
    gc = gpu_cache(shape, B, cap, p0 + T + 1, hist, p0 + T)
    k = shape.top_k
    topk = torch.full((B, T, k), -7, dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, T, shape.index_heads, k))
    lib.ds4a_index_topk(gc, p0, T, q_idx.to(DEV), w.to(DEV), shape.index_heads, k, topk, ws)
    torch.cuda.synchronize()
    oc = oracle_cache(shape, hist, p0 + T)
    ref = olayer.index_topk(oc, p0, np_(q_idx), np_(w), k, queries=queries)
    got = topk.cpu().numpy()
    if queries is not None:
        for b, t in queries:
            assert np.array_equal(got[b, t], ref[b, t]), (b, t)
    else:
        assert np.array_equal(got, ref)
    return got


def test_index_tc_query_unaligned():
    """bf16 indexer with q_idx at a 2-byte offset (not 16-byte aligned): the
    query rotation loads element by element; the lists must equal the
    oracle's, at one decode token and across a chunk whose tail queries see
    rows past the first 4 k."""
    lib = lib_()
    shape = synth.LayerShape(ratio=4)
    for B, p0, T in ((3, 6000, 1), (1, 4000, 9)):
        wl = synth.Workload("qun16", 26, B, (shape,), p0 + T, "prefill")
        cap = (p0 + T) // 4 + 1
        hist = synth.cache_history(wl, 0, p0 + T, comp_cap=cap)
        q_idx = synth.normal((B, T, 64, 128), 26, "q", dtype="bf16")
        w = synth.normal((B, T, 64), 26, "w", dtype="bf16")
        buf = torch.empty(q_idx.numel() + 1, dtype=torch.bfloat16, device=DEV)
        qd = buf[1:].view(q_idx.shape)
        qd.copy_(q_idx.to(DEV))
        assert qd.data_ptr() % 16 != 0
        gc = gpu_cache(shape, B, cap, p0 + T + 1, hist, p0 + T)
        topk = torch.empty((B, T, 512), dtype=torch.int32, device=DEV)
        ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, T, 64, 512))
        lib.ds4a_index_topk(gc, p0, T, qd, w.to(DEV), 64, 512, topk, ws)
        torch.cuda.synchronize()
        ref = olayer.index_topk(oracle_cache(shape, hist, p0 + T), p0, np_(q_idx), np_(w), 512)
        assert np.array_equal(topk.cpu().numpy(), ref), (B, p0, T)


@pytest.mark.parametrize("q_exp,k_exp", [(-70, -60), (-100, -40)])
def test_index_tc_tiny_magnitudes(q_exp, k_exp):
    """bf16 indexer with query and key entries near the bottom of the fp32
    range: head dots and their products are subnormal, so the certified top-k
    rests on its absolute underflow term and the exact rescoring must use
    separately rounded products; the lists must still equal the oracle's."""
    lib = lib_()
    shape = synth.LayerShape(ratio=4)
    B, p0, T = 2, 3000, 1
    wl = synth.Workload("tinymag", 31, B, (shape,), p0 + T, "prefill")
    cap = (p0 + T) // 4 + 1
    hist = synth.cache_history(wl, 0, p0 + T, comp_cap=cap)
    hist["index_comp_kv"] = (hist["index_comp_kv"].float() * 2.0 ** k_exp).to(torch.bfloat16)
    q_idx = (synth.normal((B, T, 64, 128), 31, "q", dtype="f32") * 2.0 ** q_exp).to(torch.bfloat16)
    w = synth.normal((B, T, 64), 31, "w", dtype="bf16")
    gc = gpu_cache(shape, B, cap, p0 + T + 1, hist, p0 + T)
    k = shape.top_k
    topk = torch.full((B, T, k), -7, dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, T, 64, k))
    lib.ds4a_index_topk(gc, p0, T, q_idx.to(DEV), w.to(DEV), 64, k, topk, ws)
    torch.cuda.synchronize()
    oc = oracle_cache(shape, hist, p0 + T)
    ref = olayer.index_topk(oc, p0, np_(q_idx), np_(w), k)
    assert np.array_equal(topk.cpu().numpy(), ref)


def test_index_tiny_fp32():
    """Tiny workload's indexer: 2 heads x 32, top-k 16, 64 visible rows."""
    run_index(lib_(), synth.TINY.layers[0], 1, 256, 1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_index_grid_ties(dtype):
    """1/8-grid inputs: exact scores with many exact ties at the cut."""
    shape = synth.LayerShape(ratio=4, index_dim=16, index_heads=4, top_k=24, dtype=dtype)
    run_index(lib_(), shape, 2, 400, 9, grid=True)


def test_index_ragged_prefill_with_padding():
    """Queries whose visible count is below, at and above k (padding with -1),
    and no visible row at all (p < 3)."""
    shape = synth.LayerShape(ratio=4, index_dim=64, index_heads=8, top_k=20)
    run_index(lib_(), shape, 2, 0, 90)


def test_index_flash_shape_decode():
    """Flash indexer (64 heads x 128, k 512) at 16,384 rows, 2 sequences."""
    shape = synth.LayerShape(ratio=4)
    run_index(lib_(), shape, 2, 65536, 1)


# ------------------------------------------------------------------ attention

def run_attn(lib, shape, B, p0, T, n_hist, topk_mode="random", seed=21, queries=None,
             scale=None):
    wl = synth.Workload("att", seed, B, (shape,), n_hist, "prefill")
    r = shape.ratio
    cap = max(1, (p0 + T) // r) if r else 0
    hist = synth.cache_history(wl, 0, p0 + T, comp_cap=cap)   # rows through p0+T
    q = synth.normal((B, T, shape.n_heads, shape.head_dim), seed, "q", dtype=shape.dtype)
    chunk = None
    if T > 1:
        chunk = synth.normal((B, T, shape.head_dim), seed, "chunk", dtype=shape.dtype)
        hist["raw_kv"] = synth.normal(hist["raw_kv"].shape, seed, "ring", dtype=shape.dtype)
    k = shape.top_k
    topk = None
    if r == 4:
        vis = (p0 + T) // 4
        topk = synth.random_topk(B, T, k, vis, seed, "tk")
        if topk_mode == "pad":       # -1 holes and entries past the visible rows
            topk[..., ::5] = -1
            topk[..., -3:] = vis + 5
    gc = gpu_cache(shape, B, cap, p0 + T + 1, hist, p0 + T)
    out = torch.empty((B, T, shape.n_heads, shape.head_dim), dtype=gc.torch_dtype, device=DEV)
    scale = 1.0 / np.sqrt(shape.head_dim) if scale is None else scale
    tk_dev = topk.to(DEV) if topk is not None else None
    if T == 1 and chunk is None:
        ws = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_DECODE, 1, shape.n_heads, k))
        lib.ds4a_sparse_attn_decode(gc, p0, q[:, 0].contiguous().to(DEV), shape.n_heads,
                                    None if tk_dev is None else tk_dev[:, 0].contiguous(), k,
                                    scale, out[:, 0], ws)
    else:
        ring_before = gc.raw_kv.clone()
        ws = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_PREFILL, T, shape.n_heads, k))
        lib.ds4a_sparse_attn_prefill_chunk(gc, p0, T, q.to(DEV), shape.n_heads, chunk.to(DEV),
                                           tk_dev, k, scale, out, ws)
    torch.cuda.synchronize()
    oc = oracle_cache(shape, hist, p0 + T)
    ref = olayer.attention(oc, p0, np_(q), None if topk is None else topk.numpy(), scale,
                           ring=np_(hist["raw_kv"]),
                           chunk_rows=None if chunk is None else np_(chunk), queries=queries)
    got = np_(out)
    if queries is not None:
        got = np.stack([got[b, t] for b, t in queries])
        ref = np.stack([ref[b, t] for b, t in queries])
    e = rel_l2(got, ref)
    assert e <= TOL[shape.dtype], e
    if chunk is not None:
        n = min(T, shape.cap_raw)
        ring = np_(gc.raw_kv)
        for t in range(T - n, T):
            assert np.array_equal(ring[:, (p0 + t) % shape.cap_raw], np_(chunk)[:, t])
    return e


@pytest.mark.parametrize("ratio", [0, 4, 128])
def test_attn_decode_tiny_fp32(ratio):
    shape = synth.TINY.layers[0].replace(ratio=ratio)
    run_attn(lib_(), shape, 2, 300, 1, 300)


# (0, 500) and (128, 20000) take the TMA tiles: the whole ring, and 156
# compressed rows as one full and one part-filled tile (rows past 156 zero)
@pytest.mark.parametrize("ratio,p", [(4, 1000), (128, 65536), (0, 77), (4, 5), (0, 500),
                                     (128, 20000)])
def test_attn_decode_bf16(ratio, p):
    shape = synth.LayerShape(ratio=ratio)
    run_attn(lib_(), shape, 3, p, 1, p, topk_mode="pad")


@pytest.mark.parametrize("ratio,p0,T", [(4, 300, 50), (128, 1000, 70), (0, 60, 100), (4, 0, 40)])
def test_attn_prefill(ratio, p0, T):
    """Window spanning the old ring and the chunk, causal visibility, ring commit."""
    shape = synth.LayerShape(ratio=ratio, n_heads=16)
    run_attn(lib_(), shape, 2, p0, T, p0, topk_mode="pad")


def test_attn_prefill_tiny_fp32_window_only_ring():
    shape = synth.TINY.layers[0]
    run_attn(lib_(), shape, 1, 200, 7, 200)


# ------------------------------------------------------------------ end to end

def test_tiny_workload_end_to_end():
    """The tiny fp32 workload: 256-token prefill (two chunks) then the decode
    step at 256, each side running its own chain from an empty cache."""
    lib = lib_()
    wl = synth.TINY
    s = wl.layers[0]
    cap = 80
    gc = gpu_cache(s, 1, cap, 1024)
    lib.ds4a_cache_reset(gc)
    oc = oracle_cache(s, {k: v for k, v in synth.empty_history(wl, 0, cap).items()}, 0)
    k = s.top_k
    for p0, T in ((0, 100), (100, 156)):
        inp = synth.step_inputs(wl, 0, p0, T)
        d = to_dev(inp)
        chunk = torch.empty((1, T, s.head_dim), device=DEV)
        lib.ds4a_compress_append(gc, p0, T, d, raw_chunk_out=chunk)
        topk = torch.empty((1, T, k), dtype=torch.int32, device=DEV)
        ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, T, s.index_heads, k))
        lib.ds4a_index_topk(gc, p0, T, d["q_idx"], d["w"], s.index_heads, k, topk, ws)
        out = torch.empty((1, T, s.n_heads, s.head_dim), device=DEV)
        wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_PREFILL, T, s.n_heads, k))
        lib.ds4a_sparse_attn_prefill_chunk(gc, p0, T, d["q"], s.n_heads, chunk, topk, k,
                                           1 / np.sqrt(s.head_dim), out, wa)
        o_ref, tk_ref = olayer.prefill_chunk(oc, p0, to_np(inp), k)
        torch.cuda.synchronize()
        assert np.array_equal(topk.cpu().numpy(), tk_ref)
        assert rel_l2(np_(out), o_ref) <= TOL["f32"]
    compare_cache(gc, oc, "f32", "after prefill")
    inp = synth.step_inputs(wl, 0, 256, 1)
    d = to_dev(inp)
    lib.ds4a_compress_append(gc, 256, 1, d)
    topk = torch.empty((1, k), dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, 1, s.index_heads, k))
    lib.ds4a_index_topk(gc, 256, 1, d["q_idx"], d["w"], s.index_heads, k, topk, ws)
    out = torch.empty((1, s.n_heads, s.head_dim), device=DEV)
    wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_DECODE, 1, s.n_heads, k))
    lib.ds4a_sparse_attn_decode(gc, 256, d["q"][:, 0].contiguous(), s.n_heads, topk, k,
                                1 / np.sqrt(s.head_dim), out, wa)
    o_ref, tk_ref = olayer.decode_step(oc, 256, to_np(inp), k)
    torch.cuda.synchronize()
    assert np.array_equal(topk.cpu().numpy(), tk_ref)
    assert rel_l2(np_(out), o_ref) <= TOL["f32"]
