"""Pins of oracle.indexer: exact integer-grid scores, the lower-index tie
rule, k >= visible, visibility at a boundary, brute-force ranking, the ReLU."""
from fractions import Fraction

import numpy as np

from oracle import indexer
from oracle.numerics import round_bf16


def grid(r, shape):
    return (r.integers(-8, 9, size=shape) * 0.125).astype(np.float32)


def exact_score(q, w, k):
    """Exact rational score sum_h w_h max(0, q_h . k) (brute force, Fractions)."""
    tot = Fraction(0)
    for h in range(q.shape[0]):
        d = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(q[h], k))
        tot += Fraction(float(w[h])) * max(d, Fraction(0))
    return tot


def test_grid_scores_are_exact_and_ties_go_to_lower_index():
    """On the 1/8 grid every product and partial sum is exact in fp32, so the
    fp32 recipe must equal the exact rational score, whatever the order; ties
    are common and the kept set must prefer lower indices."""
    r = np.random.default_rng(0)
    Hi, Di, n, k = 3, 8, 60, 7
    q, w, keys = grid(r, (Hi, Di)), grid(r, Hi), grid(r, (n, Di))
    keys[30:40] = keys[10]                   # force exact ties
    s = indexer.index_scores(q, w, keys)
    ex = [exact_score(q, w, keys[i]) for i in range(n)]
    assert all(Fraction(float(s[i])) == ex[i] for i in range(n))
    order = sorted(range(n), key=lambda i: (-ex[i], i))
    want = np.sort(np.array(order[:k], np.int32))
    got = indexer.topk_select(s, n, k)
    assert np.array_equal(got, want)
    # a tie straddling the cut: the tied rows with lower index win
    s2 = np.zeros(20, np.float32)
    s2[[3, 8, 12, 17]] = 5.0
    s2[[1, 19]] = 9.0
    assert np.array_equal(indexer.topk_select(s2, 20, 4), np.array([1, 3, 8, 19]))


def test_k_at_least_visible_keeps_all_padded():
    out = indexer.topk_select(np.arange(5, dtype=np.float32), 5, 8)
    assert np.array_equal(out, np.array([0, 1, 2, 3, 4, -1, -1, -1]))
    q = np.ones((2, 4), np.float32)
    keys = np.ones((100, 4), np.float32)
    # position 39 sees floor(40 / 4) = 10 rows; with k = 16 every one is kept
    out = indexer.index_topk_query(q, np.ones(2, np.float32), keys, 39, 1e4, 4, "f32", 16)
    assert np.array_equal(out[:10], np.arange(10)) and np.all(out[10:] == -1)


def test_visibility_at_boundary():
    assert indexer.visible_rows(4, 3) == 1        # row 0 is emitted at p = 3
    assert indexer.visible_rows(4, 2) == 0
    assert indexer.visible_rows(4, 65536) == 16384
    assert indexer.visible_rows(4, 28675) == 7169


def test_brute_force_ranking_on_gaussian():
    """fp32 recipe against a fp64 brute force of the same sum: values within
    the fp32 rounding bound, same top-k set when the k-th gap is clear."""
    r = np.random.default_rng(1)
    Hi, Di, n, k = 4, 16, 200, 20
    q = r.standard_normal((Hi, Di)).astype(np.float32)
    w = r.standard_normal(Hi).astype(np.float32)
    keys = r.standard_normal((n, Di)).astype(np.float32)
    s = indexer.index_scores(q, w, keys)
    bf = np.array([sum(float(w[h]) * max(0.0, sum(float(q[h, d]) * float(keys[i, d])
                                                   for d in range(Di))) for h in range(Hi))
                   for i in range(n)])
    bound = (Di + Hi + 2) * 2.0**-23 * np.sum(np.abs(w)[None, :] *
                                             (np.abs(keys) @ np.abs(q).T), axis=1)
    assert np.all(np.abs(s - bf) <= bound)
    srt = np.sort(bf)[::-1]
    assert srt[k - 1] - srt[k] > 2 * bound.max()
    assert np.array_equal(indexer.topk_select(s, n, k), np.sort(np.argsort(-bf)[:k]))


def test_relu_drops_negative_heads():
    """A head whose dot products are all negative adds nothing, whatever its weight."""
    r = np.random.default_rng(2)
    keys = np.abs(r.standard_normal((30, 8))).astype(np.float32)
    q = r.standard_normal((2, 8)).astype(np.float32)
    q[1] = -np.abs(q[1])
    w1 = np.array([1.5, 0.0], np.float32)
    w2 = np.array([1.5, 1e6], np.float32)
    assert np.array_equal(indexer.index_scores(q, w1, keys), indexer.index_scores(q, w2, keys))


def test_rotated_query_rounded_to_storage():
    r = np.random.default_rng(3)
    q = round_bf16(r.standard_normal((2, 4, 128))).astype(np.float32)
    out = indexer.rotate_index_query(q, 12345, 160000.0, 64, "bf16")
    assert np.all(out.view(np.uint32) & 0xFFFF == 0)
    assert np.array_equal(out[..., :64], q[..., :64])
