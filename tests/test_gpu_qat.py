"""GPU parity of the compressor's step 8 (FP8 attention rows, FP4 QAT indexer
rows and queries) against the oracle.

The scales and codes are integers that the GPU and the oracle decide in fp32
with the same recipe. The indexer query's input is identical on both sides,
so its round trip, and the top-k that follows, must match exactly. A
compressed row's input is the fp32 row. The GPU computes it in fp32, the
oracle in fp64 (then rounds it). The two can differ by a few ulps, so a code
may differ where the oracle's value lies within 2^-12 of a quantum of a
rounding midpoint, or of a scale boundary. Those are accepted; every other
element must match exactly. Decisions further down (top-k, attention) are
then compared on the GPU's own rows."""
import numpy as np
import pytest
import torch

import synth
from helpers import TOL, gpu_cache, np_, oracle_cache, rel_l2, to_dev, to_np
from oracle import layer as olayer
from oracle import qat
from oracle.numerics import round_store
from test_gpu_parity import lib_

pytestmark = pytest.mark.gpu
DEV = "cuda"
QAT_ALL = olayer.QAT_FP8_ATTN | olayer.QAT_FP4_INDEX
BORDER = 2.0 ** -12


def _near_midpoint(r, vals):
    """|r| within BORDER steps of a midpoint between neighbouring table values."""
    a = abs(r)
    i = np.searchsorted(vals, a)
    for j in (i - 1, i):
        if 0 <= j < len(vals) - 1:
            mid, step = (vals[j] + vals[j + 1]) / 2, vals[j + 1] - vals[j]
            if abs(a - mid) <= BORDER * step:
                return True
    return False


def _near_scale_edge(amax, qmax):
    k = qat.block_scale_exp(amax, qmax)
    return amax > 0 and abs(amax / (qmax * 2.0 ** (k - 1)) - 1) <= BORDER


def check_fp8_rows(got, pre, n_rot):
    """got: stored attention rows [N, D]; pre: the oracle's rows before step 8.
    Non-RoPE dims: exact up to borderline codes. Returns the count of those."""
    n_nope = got.shape[-1] - n_rot
    x = pre[:, :n_nope].astype(np.float32)
    want = qat.fp8_round_trip(x)
    g = got[:, :n_nope]
    vals = qat.e4m3_table()[0]
    n_border = 0
    for r, d in np.argwhere(g != want):
        b0 = (d // qat.FP8_BLOCK) * qat.FP8_BLOCK
        seg = x[r, b0:b0 + qat.FP8_BLOCK].astype(np.float64)
        amax = np.abs(seg).max()
        if _near_scale_edge(amax, qat.E4M3_MAX):
            n_border += 1
            continue
        k = qat.block_scale_exp(amax, qat.E4M3_MAX)
        rr = float(x[r, d]) * 2.0 ** -k
        gc, wc = abs(g[r, d]) * 2.0 ** -k, abs(want[r, d]) * 2.0 ** -k
        assert gc in vals, (r, d, g[r, d])
        assert _near_midpoint(rr, vals), (r, d, rr, g[r, d], want[r, d])
        assert abs(np.searchsorted(vals, gc) - np.searchsorted(vals, wc)) == 1, (r, d)
        n_border += 1
    return n_border


def _fp4_variants(x):
    """The FP4 round trip of one fp32 row, and its variants with one
    borderline decision taken the other way: a code within BORDER of a
    midpoint moved to the other neighbour, or a block whose amax sits within
    BORDER of a scale boundary requantised at the other scale."""
    vals = qat.e2m1_table()
    c = qat.hadamard_scale(x.size)
    z = (qat.fwht_f32(x) * c).astype(np.float64)
    n = z.size
    ks, zq = [], np.empty(n)
    for b0 in range(0, n, qat.FP4_BLOCK):
        seg = z[b0:b0 + qat.FP4_BLOCK]
        k = qat.block_scale_exp(np.abs(seg).max(), qat.E2M1_MAX)
        ks.append(k)
        zq[b0:b0 + qat.FP4_BLOCK] = qat.round_to_table(seg * 2.0 ** -k, vals) * 2.0 ** k
    out = [zq]
    for bi, b0 in enumerate(range(0, n, qat.FP4_BLOCK)):
        seg, k = z[b0:b0 + qat.FP4_BLOCK], ks[bi]
        if _near_scale_edge(np.abs(seg).max(), qat.E2M1_MAX):
            for k2 in (k - 1, k + 1):
                r = seg * 2.0 ** -k2
                if np.abs(r).max() <= qat.E2M1_MAX:
                    v = zq.copy()
                    v[b0:b0 + qat.FP4_BLOCK] = qat.round_to_table(r, vals) * 2.0 ** k2
                    out.append(v)
        for j, zz in enumerate(seg):
            r = zz * 2.0 ** -k
            if _near_midpoint(r, vals[0]):
                a, i = abs(r), np.searchsorted(vals[0], abs(r))
                lo, hi = vals[0][max(i - 1, 0)], vals[0][min(i, len(vals[0]) - 1)]
                cur = abs(zq[b0 + j]) * 2.0 ** -k
                alt = hi if cur == lo else lo
                v = zq.copy()
                v[b0 + j] = np.copysign(alt, r) * 2.0 ** k
                out.append(v)
    return [qat.fwht_f32(v.astype(np.float32)) * c for v in out]


def check_fp4_rows(got, pre, dtype):
    """got: stored indexer rows [N, Di]; pre: the oracle's rows before step 8.
    A row matches the oracle's exactly or one of its single borderline
    variants. Returns the count of rows that differ from the oracle's."""
    x = pre.astype(np.float32)
    want = round_store(qat.index_row_round_trip(pre), dtype)
    rows = np.nonzero(np.any(got != want, axis=1))[0]
    for r in rows:
        ok = any(np.array_equal(got[r], round_store(v.astype(np.float64), dtype))
                 for v in _fp4_variants(x[r])[1:])
        assert ok, f"row {r} differs from every borderline variant"
    return len(rows)


def _shape(dtype, ratio=4):
    return synth.LayerShape(ratio=ratio, head_dim=128 if dtype == "f32" else 512,
                            index_dim=32 if dtype == "f32" else 128,
                            index_heads=2 if dtype == "f32" else 64,
                            n_heads=4 if dtype == "f32" else 64,
                            top_k=16 if dtype == "f32" else 512, dtype=dtype)


def compare_rows(gc, oc, n0, n1, shape):
    """Rows n0..n1-1 of both lanes: state exact, step-8 dims by the rules above."""
    for name in ("attn_state_kv", "attn_state_score", "index_state_kv", "index_state_score"):
        g = getattr(gc, name)
        if g is not None:
            assert np.array_equal(np_(g), getattr(oc, name)), name
    ga = np_(gc.attn_comp_kv)[:, n0:n1].reshape(-1, shape.head_dim).astype(np.float64)
    pa = oc.attn_pre[:, n0:n1].reshape(-1, shape.head_dim)
    oa = oc.attn_comp_kv[:, n0:n1].reshape(-1, shape.head_dim)
    nb = check_fp8_rows(ga, pa, shape.n_rot)
    assert nb <= max(2, ga[:, :-shape.n_rot].size // 10000), nb
    assert rel_l2(ga[:, -shape.n_rot:], oa[:, -shape.n_rot:]) <= TOL[shape.dtype]
    n_fp4 = 0
    if shape.ratio == 4:
        gi = np_(gc.index_comp_kv)[:, n0:n1].reshape(-1, shape.index_dim).astype(np.float64)
        pi = oc.index_pre[:, n0:n1].reshape(-1, shape.index_dim)
        n_fp4 = check_fp4_rows(gi, pi, shape.dtype)
        assert n_fp4 <= max(1, gi.shape[0] // 100), n_fp4
    return nb, n_fp4


@pytest.mark.parametrize("ratio,dtype,p0,T", [(4, "bf16", 1021, 300), (4, "f32", 2, 61),
                                              (128, "bf16", 200, 300), (4, "bf16", 1023, 1)])
def test_append_qat_chunk(ratio, dtype, p0, T):
    """Chunk (and single-token) appends with both round trips on: state exact,
    rows by the borderline rule, raw rows untouched by step 8."""
    lib = lib_()
    shape = _shape(dtype, ratio)
    wl = synth.Workload("qat", 21, 2, (shape,), p0, "prefill")
    cap = (p0 + T) // ratio + 1
    hist = synth.cache_history(wl, 0, p0, comp_cap=cap) if p0 else synth.empty_history(wl, 0, cap)
    inp = synth.step_inputs(wl, 0, p0, T)
    qflag = QAT_ALL if ratio == 4 else olayer.QAT_FP8_ATTN
    gc = gpu_cache(shape, 2, cap, p0 + T + 1, hist, p0, qat=qflag)
    chunk = torch.empty((2, T, shape.head_dim), dtype=gc.torch_dtype, device=DEV)
    lib.ds4a_compress_append(gc, p0, T, to_dev(inp), raw_chunk_out=chunk if T > 1 else None)
    torch.cuda.synchronize()
    oc = oracle_cache(shape, hist, p0, qat=qflag, keep_pre=True)
    rows = olayer.compress_append(oc, p0, to_np(inp), chunk=T > 1)
    if T > 1:
        assert rel_l2(np_(chunk), rows) <= TOL[dtype]
    compare_rows(gc, oc, p0 // ratio, (p0 + T) // ratio, shape)


def test_append_qat_changes_rows_and_keeps_norm_bounds():
    """The flag takes effect (rows differ from the plain cache's) and the
    indexer row norms still bound the stored, round-tripped rows."""
    lib = lib_()
    shape = _shape("bf16")
    wl = synth.Workload("qatn", 22, 2, (shape,), 0, "prefill")
    T, cap = 512, 129
    inp = to_dev(synth.step_inputs(wl, 0, 0, T))
    out = {}
    for q in (0, QAT_ALL):
        gc = gpu_cache(shape, 2, cap, T + 1, synth.empty_history(wl, 0, cap), 0, qat=q)
        chunk = torch.empty((2, T, 512), dtype=torch.bfloat16, device=DEV)
        lib.ds4a_compress_append(gc, 0, T, inp, raw_chunk_out=chunk)
        torch.cuda.synchronize()
        out[q] = gc
    a0, a1 = out[0].attn_comp_kv[:, :128], out[QAT_ALL].attn_comp_kv[:, :128]
    assert not torch.equal(a0[..., :448], a1[..., :448])
    assert torch.equal(a0[..., 448:], a1[..., 448:])
    assert not torch.equal(out[0].index_comp_kv[:, :128], out[QAT_ALL].index_comp_kv[:, :128])
    g = out[QAT_ALL]
    exact = torch.linalg.vector_norm(g.index_comp_kv[:, :128].double(), dim=-1)
    got = g.index_norm[:, :128].double()
    assert bool((got >= exact).all()) and bool((got <= exact * (1 + 1e-4)).all())


@pytest.mark.parametrize("dtype,B,p0,T", [("bf16", 2, 3001, 37), ("bf16", 8, 16383, 1),
                                          ("f32", 2, 300, 9)])
def test_index_qat_query_exact(dtype, B, p0, T):
    """Same keys on both sides: the QAT query is the same fp32 recipe, so the
    top-k lists must be identical (tensor-core path for bf16, exact path for
    f32), and must differ from the lists without the round trip somewhere."""
    lib = lib_()
    shape = _shape(dtype)
    wl = synth.Workload("qidx", 23, B, (shape,), p0 + T, "prefill")
    cap = (p0 + T) // 4 + 1
    hist = synth.cache_history(wl, 0, p0 + T, comp_cap=cap)
    q_idx = synth.normal((B, T, shape.index_heads, shape.index_dim), 23, "q", dtype=dtype)
    w = synth.normal((B, T, shape.index_heads), 23, "w", dtype=dtype)
    gc = gpu_cache(shape, B, cap, p0 + T + 1, hist, p0 + T, qat=QAT_ALL)
    k = shape.top_k
    topk = torch.full((B, T, k), -7, dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, T, shape.index_heads, k))
    lib.ds4a_index_topk(gc, p0, T, q_idx.to(DEV), w.to(DEV), shape.index_heads, k, topk, ws)
    torch.cuda.synchronize()
    oc = oracle_cache(shape, hist, p0 + T, qat=QAT_ALL)
    ref = olayer.index_topk(oc, p0, np_(q_idx), np_(w), k)
    assert np.array_equal(topk.cpu().numpy(), ref)
    plain = olayer.index_topk(oracle_cache(shape, hist, p0 + T), p0, np_(q_idx), np_(w), k)
    assert not np.array_equal(ref, plain)


def test_index_qat_query_unaligned():
    """q_idx at a 2-byte offset (not 16-byte aligned): element loads, same result."""
    lib = lib_()
    shape = _shape("bf16")
    B, p0, T = 1, 4000, 5
    wl = synth.Workload("qun", 24, B, (shape,), p0 + T, "prefill")
    cap = (p0 + T) // 4 + 1
    hist = synth.cache_history(wl, 0, p0 + T, comp_cap=cap)
    q_idx = synth.normal((B, T, 64, 128), 24, "q", dtype="bf16")
    w = synth.normal((B, T, 64), 24, "w", dtype="bf16")
    buf = torch.empty(q_idx.numel() + 1, dtype=torch.bfloat16, device=DEV)
    qd = buf[1:].view(q_idx.shape)
    qd.copy_(q_idx.to(DEV))
    assert qd.data_ptr() % 16 != 0
    gc = gpu_cache(shape, B, cap, p0 + T + 1, hist, p0 + T, qat=QAT_ALL)
    topk = torch.empty((B, T, 512), dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, T, 64, 512))
    lib.ds4a_index_topk(gc, p0, T, qd, w.to(DEV), 64, 512, topk, ws)
    torch.cuda.synchronize()
    ref = olayer.index_topk(oracle_cache(shape, hist, p0 + T, qat=QAT_ALL), p0, np_(q_idx),
                            np_(w), 512)
    assert np.array_equal(topk.cpu().numpy(), ref)


def test_qat_decode_step_layer():
    """One Flash-shape c4a decode step at a ratio boundary with both round
    trips: new rows by the borderline rule; top-k and attention on the GPU's
    rows equal the oracle's."""
    lib = lib_()
    shape = _shape("bf16")
    B, p = 4, 8191
    wl = synth.Workload("qdec", 25, B, (shape,), p, "decode")
    cap = (p + 1) // 4 + 1
    hist = synth.cache_history(wl, 0, p, comp_cap=cap)
    inp = synth.step_inputs(wl, 0, p, 1)
    gc = gpu_cache(shape, B, cap, p + 2, hist, p, qat=QAT_ALL)
    dinp = to_dev(inp)
    lib.ds4a_compress_append(gc, p, 1, dinp)
    k = shape.top_k
    topk = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, 1, 64, k))
    lib.ds4a_index_topk(gc, p, 1, dinp["q_idx"], dinp["w"], 64, k, topk, ws)
    out = torch.empty((B, 64, 512), dtype=torch.bfloat16, device=DEV)
    wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_DECODE, 1, 64, k))
    lib.ds4a_sparse_attn_decode(gc, p, dinp["q"][:, 0].contiguous(), 64, topk, k,
                                1 / np.sqrt(512), out, wa)
    torch.cuda.synchronize()
    oc = oracle_cache(shape, hist, p, qat=QAT_ALL, keep_pre=True)
    olayer.compress_append(oc, p, to_np(inp), chunk=False)
    i = (p + 1) // 4 - 1
    compare_rows(gc, oc, i, i + 1, shape)
    oc.attn_comp_kv[:, i] = np_(gc.attn_comp_kv)[:, i]   # decide on the GPU's rows
    oc.index_comp_kv[:, i] = np_(gc.index_comp_kv)[:, i]
    ninp = to_np(inp)
    tk = olayer.index_topk(oc, p, ninp["q_idx"], ninp["w"], k)
    assert np.array_equal(topk.cpu().numpy(), tk[:, 0])
    o_ref = olayer.attention(oc, p, ninp["q"], tk)
    assert rel_l2(np_(out), o_ref[:, 0]) <= TOL["bf16"]


def test_qat_flag_checks():
    """Unknown bits, FP8 on a window-only layer and FP4 off ratio 4 are
    refused before any launch."""
    lib = lib_()
    for ratio, q in ((4, 4), (0, 1), (128, 2)):
        shape = _shape("bf16", ratio)
        gc = gpu_cache(shape, 1, 4, 64, qat=q)
        inp = to_dev(synth.step_inputs(synth.Workload("qf", 26, 1, (shape,), 0, "decode"), 0, 0, 1))
        with pytest.raises(lib.Ds4aError):
            lib.ds4a_compress_append(gc, 0, 1, inp)
