"""Pins of oracle.rope: tail-only placement, norm preservation, inverse,
relative-position property, the per-pair angle, and the fp32 recipe."""
import numpy as np

from oracle import rope


def rng(seed=0):
    return np.random.default_rng(seed)


def test_head_dims_untouched_and_position_zero_identity():
    x = rng().standard_normal((3, 512))
    y = rope.rope_tail(x, np.array([5, 77, 131071]), 160000.0, 64)
    assert np.array_equal(y[:, :448], x[:, :448])       # first D - 64 dims
    assert not np.allclose(y[:, 448:], x[:, 448:])
    assert np.array_equal(rope.rope_tail(x, 0, 10000.0, 64), x)


def test_pair_norms_preserved_and_inverse():
    x = rng(1).standard_normal((4, 128))
    p = np.array([1, 999, 65536, 131072])
    y = rope.rope_tail(x, p, 10000.0, 64)
    n0 = np.hypot(x[:, 64::2], x[:, 65::2])
    n1 = np.hypot(y[:, 64::2], y[:, 65::2])
    assert np.allclose(n0, n1, rtol=3e-7, atol=0)       # fp32 cos/sin: |c^2+s^2-1| < 2^-22
    z = rope.rope_tail(y, p, 10000.0, 64, inverse=True)
    assert np.allclose(z, x, rtol=0, atol=1e-6)


def test_pair_angle_is_p_times_base_power():
    """Rotating the unit vector e_a of pair i at position p gives the angle
    p * base^(-2i/n_rot) (mod 2 pi), read back with atan2; the rotation is
    counter-clockwise (a, b) -> (a cos - b sin, a sin + b cos)."""
    n_rot, base, D = 64, 10000.0, 64
    for p in (1, 3, 1000):
        for i in (0, 1, 17, 31):
            x = np.zeros(D)
            x[2 * i] = 1.0
            y = rope.rope_tail(x, p, base, n_rot)
            got = np.arctan2(y[2 * i + 1], y[2 * i])
            want = np.remainder(p * base ** (-2.0 * i / n_rot) + np.pi, 2 * np.pi) - np.pi
            assert abs(got - want) < 1e-6, (p, i, got, want)


def test_relative_position_property():
    """<R(p) q, R(p') k> depends on p - p' only (in the rotated dims)."""
    r = rng(2)
    q, k = r.standard_normal(128), r.standard_normal(128)
    base = 160000.0
    d1 = rope.rope_tail(q, 5000, base, 64) @ rope.rope_tail(k, 4000, base, 64)
    d2 = rope.rope_tail(q, 131000, base, 64) @ rope.rope_tail(k, 130000, base, 64)
    assert abs(d1 - d2) < 1e-5 * (np.abs(q) @ np.abs(k))
    d3 = rope.rope_tail(q, 5000, base, 64) @ rope.rope_tail(k, 4001, base, 64)
    assert abs(d1 - d3) > 1e-4


def test_fp32_recipe_close_to_fp64_and_exact_on_grid():
    x = rng(3).standard_normal((8, 2, 32)).astype(np.float32)
    p = np.arange(8)[:, None] * 4093
    y32 = rope.rope_tail_f32(x, p, 160000.0, 32)
    y64 = rope.rope_tail(x.astype(np.float64), p, 160000.0, 32)
    assert y32.dtype == np.float32
    assert np.allclose(y32, y64, rtol=0, atol=4 * 2.0**-24 * np.abs(x).max() * 2)
    # at p = 0 the recipe is exact: a*1 - b*0 = a
    assert np.array_equal(rope.rope_tail_f32(x, 0, 160000.0, 32), x)
