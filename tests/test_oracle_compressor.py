"""Pins of oracle.compressor: pooling special cases and closed forms, the
window geometry of c4a / c128a rows, row counts, RMSNorm, chunk invariance."""
import numpy as np
import pytest

from oracle import compressor, schedule
from oracle.layer import OracleCache, compress_append

NEG = -np.inf


def rng(seed=0):
    return np.random.default_rng(seed)


def test_equal_scores_give_plain_mean():
    r = rng()
    kv = r.standard_normal((3, 8, 16))
    sc = np.broadcast_to(r.standard_normal((3, 1, 16)), (3, 8, 16))
    out = compressor.softmax_pool(kv, sc, np.zeros((8, 16)))
    assert np.allclose(out, kv.mean(axis=1), rtol=1e-14, atol=1e-14)


def test_empty_slots_excluded_and_all_empty_gives_zero():
    """First c4a window: slots 0..3 empty -> mean of the 4 present tokens (R2);
    no slot present -> 0 (the denominator guard)."""
    r = rng(1)
    kv = r.standard_normal((1, 8, 4))
    sc = np.zeros((1, 8, 4))
    sc[:, :4] = NEG
    out = compressor.softmax_pool(kv, sc, np.zeros((8, 4)))
    assert np.allclose(out[0], kv[0, 4:].mean(axis=0), rtol=1e-14)
    out0 = compressor.softmax_pool(kv, np.full((1, 8, 4), NEG), np.zeros((8, 4)))
    assert np.array_equal(out0, np.zeros((1, 4)))


def test_two_slot_closed_form_and_dominant_slot():
    """Two slots: out = kv1 + (kv0 - kv1) * sigmoid(s0 - s1); a dominant score
    selects its slot; APE adds to the score of its own slot."""
    r = rng(2)
    kv = r.standard_normal((1, 2, 5))
    s = r.standard_normal((1, 2, 5))
    ape = r.standard_normal((2, 5))
    out = compressor.softmax_pool(kv, s, ape)
    d = (s[0, 0] + ape[0]) - (s[0, 1] + ape[1])
    want = kv[0, 1] + (kv[0, 0] - kv[0, 1]) / (1.0 + np.exp(-d))
    assert np.allclose(out[0], want, rtol=1e-13, atol=1e-14)
    s2 = s.copy()
    s2[0, 0] += 80.0
    assert np.allclose(compressor.softmax_pool(kv, s2, ape)[0], kv[0, 0], rtol=1e-12)


def test_permuting_slots_with_ape_rows_is_invariant():
    r = rng(3)
    kv, sc, ape = r.standard_normal((2, 8, 6)), r.standard_normal((2, 8, 6)), r.standard_normal((8, 6))
    perm = r.permutation(8)
    a = compressor.softmax_pool(kv, sc, ape)
    b = compressor.softmax_pool(kv[:, perm], sc[:, perm], ape[perm])
    assert np.allclose(a, b, rtol=1e-13)


def test_rms_norm_unit_rms_and_scale_invariance():
    r = rng(4)
    c = r.standard_normal((3, 512)) * 7.0
    g = 1.0 + 0.02 * r.standard_normal(512)
    y = compressor.rms_norm(c, g)
    rms = np.sqrt(np.mean((y / g) ** 2, axis=-1))
    assert np.allclose(rms, 1.0, rtol=1e-7)          # eps = 1e-6 against mean(c^2) ~ 49
    assert np.allclose(compressor.rms_norm(3.0 * c, g), y, rtol=1e-7)


def _cache(ratio, D, n_rot, cap, dtype="f32", Di=0, index_rot=0):
    W = {4: 8, 128: 128, 0: 0}[ratio]
    kw = dict(ratio=ratio, head_dim=D, n_rot=n_rot, cap_raw=8, base=10000.0, dtype=dtype,
              n_tokens=0, raw_kv=np.zeros((1, 8, D)), index_dim=Di, index_rot=index_rot)
    if ratio:
        kw.update(attn_comp_kv=np.zeros((1, cap, D)), attn_state_kv=np.zeros((1, W, D)),
                  attn_state_score=np.full((1, W, D), NEG))
    if ratio == 4:
        kw.update(index_comp_kv=np.zeros((1, cap, Di)), index_state_kv=np.zeros((1, 8, Di)),
                  index_state_score=np.full((1, 8, Di), NEG))
    return OracleCache(**kw)


def _onehot_inputs(ratio, T, D, n_keep, Di=4):
    """Token t's candidate is the one-hot e_(t mod n_keep); scores are equal."""
    cand = np.zeros((1, T, D))
    for t in range(T):
        cand[0, t, t % n_keep] = 1.0
    inp = {"raw_kv_in": np.zeros((1, T, D)), "attn_cand": cand,
           "attn_score": np.zeros((1, T, D)),
           "ape_attn": np.zeros((8 if ratio == 4 else ratio, D)), "gamma_attn": np.ones(D)}
    if ratio == 4:
        inp.update(idx_cand=np.zeros((1, T, Di)), idx_score=np.zeros((1, T, Di)),
                   ape_idx=np.zeros((8, Di)), gamma_idx=np.ones(Di))
    return inp


@pytest.mark.parametrize("ratio,window,stride", [(4, 8, 4), (128, 128, 128)])
def test_window_geometry(ratio, window, stride):
    """Row i pools exactly the tokens the vLLM page describes: c4a 8 tokens at
    stride 4 (4i-4 .. 4i+3, row 0 only 0..3), c128a 128 tokens at stride 128.
    Read back from the support of one-hot candidates (dims below the rotated
    tail are not rotated)."""
    n_keep = 1000
    D = n_keep + 2
    T = 3 * stride
    c = _cache(ratio, D, 2, 4, Di=4, index_rot=4)
    compress_append(c, 0, _onehot_inputs(ratio, T, D, n_keep), chunk=False)
    assert c.n_comp == 3
    for i in range(3):
        support = set(np.nonzero(np.abs(c.attn_comp_kv[0, i, :n_keep]) > 1e-12)[0])
        first = max(0, i * stride - (window - stride))
        assert support == set(range(first, i * stride + stride)), (ratio, i)
        vals = c.attn_comp_kv[0, i, sorted(support)]
        assert np.allclose(vals, vals[0])                  # equal weights


@pytest.mark.parametrize("ratio", [4, 128])
def test_row_counts_and_chunk_invariance(ratio):
    """After n tokens the cache holds floor(n / ratio) rows, and feeding the
    same tokens in one call or in chunks of 1, 3 and 200 gives identical state
    and rows (absolute-position boundaries carry across chunks)."""
    r = rng(5)
    n, D, Di = 1037 if ratio == 4 else 700, 8, 4
    inp = {"raw_kv_in": r.standard_normal((1, n, D)), "attn_cand": r.standard_normal((1, n, D)),
           "attn_score": r.standard_normal((1, n, D)),
           "ape_attn": 0.02 * r.standard_normal((8 if ratio == 4 else 128, D)),
           "gamma_attn": 1 + 0.02 * r.standard_normal(D),
           "idx_cand": r.standard_normal((1, n, Di)), "idx_score": r.standard_normal((1, n, Di)),
           "ape_idx": 0.02 * r.standard_normal((8, Di)), "gamma_idx": np.ones(Di)}
    caches = []
    for chunks in ([n], [1] * 5 + [3] * 7 + [n - 26], [200] * (n // 200) + [n % 200]):
        c = _cache(ratio, D, 4, n // ratio + 1, Di=Di, index_rot=4)
        p = 0
        for T in chunks:
            part = {k: (v[:, p:p + T] if v.ndim == 3 else v) for k, v in inp.items()}
            compress_append(c, p, part, chunk=False)
            p += T
        caches.append(c)
    ref = caches[0]
    assert ref.n_comp == schedule.n_comp_rows(ratio, n)
    assert np.all(np.abs(ref.attn_comp_kv[0, :ref.n_comp]).sum(-1) > 0)
    assert np.all(ref.attn_comp_kv[0, ref.n_comp:] == 0)
    for c in caches[1:]:
        for name in ("attn_comp_kv", "attn_state_kv", "attn_state_score", "raw_kv",
                     "index_comp_kv", "index_state_kv", "index_state_score"):
            a, b = getattr(ref, name), getattr(c, name)
            assert np.array_equal(a, b), name


def test_bf16_rows_are_bf16_exact():
    r = rng(6)
    c = _cache(4, 16, 4, 4, dtype="bf16", Di=4, index_rot=4)
    n = 8
    inp = {"raw_kv_in": r.standard_normal((1, n, 16)), "attn_cand": r.standard_normal((1, n, 16)),
           "attn_score": r.standard_normal((1, n, 16)), "ape_attn": np.zeros((8, 16)),
           "gamma_attn": np.ones(16), "idx_cand": r.standard_normal((1, n, 4)),
           "idx_score": r.standard_normal((1, n, 4)), "ape_idx": np.zeros((8, 4)),
           "gamma_idx": np.ones(4)}
    compress_append(c, 0, inp, chunk=False)
    rows = c.attn_comp_kv[0, :2].astype(np.float32)
    bits = rows.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)
