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


def _mp_f32(v, mp):
    """fp32 nearest to the mpmath value v (v converted exactly to a binary64
    first only when that cannot change the fp32 rounding, i.e. the value is
    not within 2^-40 relative of an fp32 rounding midpoint)."""
    x = float(v)
    f = np.float32(x)
    lo, hi = np.nextafter(f, np.float32(-np.inf)), np.nextafter(f, np.float32(np.inf))
    for nb in (lo, hi):
        mid = (mp.mpf(float(f)) + mp.mpf(float(nb))) / 2
        if mid != 0 and abs((v - mid) / mid) < mp.mpf(2) ** -40:
            return None          # too close to a midpoint to decide from a binary64 copy
    return f


def test_coefficients_against_independent_high_precision_evaluation():
    """rope_coeffs (fp64 libm angle, cos and sin each rounded once to fp32) pinned
    against mpmath at 50 digits, positions up to 131,072, both bases and both
    rotation widths. theta_i = base^(-2i/n_rot) must be the binary64 nearest (or
    adjacent, as C pow allows) to the exact power, and cos / sin of the fp64
    angle p * theta_i, evaluated at 50 digits and rounded once to fp32, must
    equal the oracle's coefficients. A wrong exponent (-i/n_rot), a swapped
    cos / sin, an fp32 angle or a missing pair fails here."""
    import pytest
    mp = pytest.importorskip("mpmath").mp
    mp.dps = 50
    r = np.random.default_rng(5)
    pos = np.unique(np.concatenate([np.arange(0, 70), [127, 128, 255, 256, 4095, 4096, 28671,
                                                       28672, 32767, 32768, 65535, 65536,
                                                       131071, 131072],
                                    r.integers(0, 131073, 300)]))
    undecided = 0
    for base in (10000.0, 160000.0):
        for n_rot in (64, 32):
            theta = rope.inv_freq(base, n_rot)
            for i, t in enumerate(theta):
                exact = mp.power(mp.mpf(base), mp.mpf(-2 * i) / n_rot)
                ulp = mp.mpf(np.spacing(t))
                assert abs(mp.mpf(float(t)) - exact) <= ulp, (base, n_rot, i)
            c, s = rope.rope_coeffs(pos, base, n_rot)
            assert c.dtype == np.float32 and c.shape == (len(pos), n_rot // 2)
            for a, p in enumerate(pos):
                for i in range(n_rot // 2):
                    ang = mp.mpf(float(p) * float(theta[i]))   # the reading's fp64 angle
                    for got, fn in ((c[a, i], mp.cos), (s[a, i], mp.sin)):
                        want = _mp_f32(fn(ang), mp)
                        if want is None:
                            undecided += 1
                            continue
                        assert got == want, (base, n_rot, int(p), i, fn.__name__, got, want)
    assert undecided < 4
