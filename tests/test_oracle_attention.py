"""Pins of oracle.attention and oracle.layer: one row, brute-force softmax,
k >= visible equals dense, relative-position invariance of the output,
window-only layers, and prefill == repeated decode."""
import math

import numpy as np

from oracle import attention, rope
from oracle.layer import OracleCache, decode_step, prefill_chunk

NEG = -np.inf


def rng(seed=0):
    return np.random.default_rng(seed)


def test_single_row_returns_that_row_rotated_back():
    r = rng()
    row = r.standard_normal(128)
    q = r.standard_normal((4, 128))
    o = attention.attention_query(q, 300, row[None], np.zeros((0, 128)), 1e4, 64, 0.1, "f32")
    want = rope.rope_tail(row, 300, 1e4, 64, inverse=True)
    assert np.allclose(o, np.broadcast_to(want, (4, 128)), rtol=1e-6, atol=1e-7)


def test_brute_force_softmax_tiny():
    """Python-loop softmax with math.exp on a tiny case."""
    r = rng(1)
    H, D, n = 2, 6, 5
    q, K = r.standard_normal((H, D)), r.standard_normal((n, D))
    o = attention.attend(q, K, 0.5)
    for h in range(H):
        e = [math.exp(0.5 * sum(q[h, d] * K[j, d] for d in range(D))) for j in range(n)]
        z = sum(e)
        want = [sum(e[j] * K[j, d] for j in range(n)) / z for d in range(D)]
        assert np.allclose(o[h], want, rtol=1e-12)


def test_comp_row_ids_rules():
    # skip negatives, stop at the first index >= visible
    ids = attention.comp_row_ids(4, 39, 1000, np.array([-1, 2, 5, 9, 10, 3]))
    assert list(ids) == [2, 5, 9]
    assert list(attention.comp_row_ids(128, 1000, 1000)) == list(range(7))
    assert len(attention.comp_row_ids(0, 1000, 0)) == 0
    assert list(attention.window_positions(5, 128)) == list(range(6))
    assert list(attention.window_positions(1000, 128)) == list(range(873, 1001))


def test_relative_position_invariance_of_output():
    """Shift the query and every key's position by the same amount: with the
    inverse rotation on the output, the output does not change."""
    r = rng(2)
    H, D, n = 3, 16, 9
    base, n_rot = 160000.0, 8
    x = r.standard_normal((n, D))
    q = r.standard_normal((H, D))
    pk = np.arange(n) * 3 + 100
    outs = []
    for shift in (0, 50000):
        rows = rope.rope_tail(x, (pk + shift)[:, None].squeeze(-1), base, n_rot)
        outs.append(attention.attention_query(q, 140 + shift, rows, np.zeros((0, D)), base,
                                              n_rot, 0.3, "f32"))
    assert np.allclose(outs[0], outs[1], rtol=2e-5, atol=2e-6)


def _layer(ratio, B=1, D=16, n_rot=4, Di=8, cap=64, dtype="f32"):
    W = {0: 0, 4: 8, 128: 128}[ratio]
    kw = dict(ratio=ratio, head_dim=D, n_rot=n_rot, cap_raw=8, base=160000.0, dtype=dtype,
              n_tokens=0, raw_kv=np.zeros((B, 8, D)), index_dim=Di, index_rot=Di)
    if ratio:
        kw.update(attn_comp_kv=np.zeros((B, cap, D)), attn_state_kv=np.zeros((B, W, D)),
                  attn_state_score=np.full((B, W, D), NEG))
    if ratio == 4:
        kw.update(index_comp_kv=np.zeros((B, cap, Di)), index_state_kv=np.zeros((B, 8, Di)),
                  index_state_score=np.full((B, 8, Di), NEG))
    return OracleCache(**kw)


def _inputs(r, ratio, B, T, D=16, H=2, Di=8, Hi=2):
    inp = {"raw_kv_in": r.standard_normal((B, T, D)), "q": r.standard_normal((B, T, H, D))}
    if ratio:
        W = 8 if ratio == 4 else 128
        inp.update(attn_cand=r.standard_normal((B, T, D)), attn_score=r.standard_normal((B, T, D)),
                   ape_attn=0.02 * r.standard_normal((W, D)),
                   gamma_attn=1 + 0.02 * r.standard_normal(D))
    if ratio == 4:
        inp.update(idx_cand=r.standard_normal((B, T, Di)), idx_score=r.standard_normal((B, T, Di)),
                   ape_idx=0.02 * r.standard_normal((8, Di)), gamma_idx=np.ones(Di),
                   q_idx=r.standard_normal((B, T, Hi, Di)).astype(np.float32),
                   w=r.standard_normal((B, T, Hi)).astype(np.float32))
    return inp


def _split(inp, t0, t1):
    return {k: (v[:, t0:t1] if k not in ("ape_attn", "gamma_attn", "ape_idx", "gamma_idx") else v)
            for k, v in inp.items()}


def test_prefill_chunk_equals_decode_steps():
    """A prefill chunk (window spanning the old ring and the chunk, causal
    visibility, ring committed at the end) gives the same outputs, top-k lists
    and final cache as the same tokens decoded one by one."""
    for ratio in (0, 4, 128):
        r = rng(3 + ratio)
        T0, T = 141 if ratio != 128 else 300, 29 if ratio != 128 else 140
        inp = _inputs(r, ratio, 2, T0 + T)
        a, b = _layer(ratio, B=2), _layer(ratio, B=2)
        for c in (a, b):
            prefill_chunk(c, 0, _split(inp, 0, T0), top_k=5)
        oa, ta = prefill_chunk(a, T0, _split(inp, T0, T0 + T), top_k=5)
        for t in range(T):
            ob, tb = decode_step(b, T0 + t, _split(inp, T0 + t, T0 + t + 1), top_k=5)
            assert np.array_equal(oa[:, t], ob), (ratio, t)
            if ratio == 4:
                assert np.array_equal(ta[:, t], tb)
        for name in ("raw_kv", "attn_comp_kv", "attn_state_kv", "attn_state_score",
                     "index_comp_kv"):
            x, y = getattr(a, name), getattr(b, name)
            assert (x is None and y is None) or np.array_equal(x, y), (ratio, name)


def test_topk_covering_all_rows_equals_dense_c128a_style():
    """k >= visible on a ratio-4 layer: the output equals attention over the
    window plus every visible compressed row."""
    r = rng(7)
    c = _layer(4)
    T0 = 90
    inp = _inputs(r, 4, 1, T0 + 1)
    prefill_chunk(c, 0, _split(inp, 0, T0), top_k=64)
    o, tk = decode_step(c, T0, _split(inp, T0, T0 + 1), top_k=64)
    vis = (T0 + 1) // 4
    assert np.array_equal(tk[0, :vis], np.arange(vis))
    win = np.array([c.raw_kv[0, t % 8] for t in range(T0 - 7, T0 + 1)])
    rows = np.concatenate([win, c.attn_comp_kv[0, :vis]])
    q_rot = rope.rope_tail(inp["q"][0, T0], T0, c.base, c.n_rot)
    dense = rope.rope_tail(attention.attend(q_rot, rows, 0.25), T0, c.base, c.n_rot, inverse=True)
    assert np.array_equal(o[0], dense.astype(np.float32).astype(np.float64))


def test_window_only_layer_uses_last_cap_rows():
    """Ratio 0: the output only depends on the last cap_raw raw rows."""
    r = rng(8)
    c1, c2 = _layer(0), _layer(0)
    inp1 = _inputs(r, 0, 1, 40)
    inp2 = {k: v.copy() for k, v in inp1.items()}
    inp2["raw_kv_in"][:, :30] = r.standard_normal((1, 30, 16))   # older than the window
    o1, _ = prefill_chunk(c1, 0, inp1, top_k=1)
    o2, _ = prefill_chunk(c2, 0, inp2, top_k=1)
    assert np.array_equal(o1[:, 39], o2[:, 39])
    assert not np.allclose(o1[:, 35], o2[:, 35])
