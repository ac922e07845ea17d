"""Pins of oracle.numerics.round_bf16, the storage rounding of every bf16 row,
rotated indexer query and output the parity tests compare.

The rule it must follow is round to nearest, ties to even (bf16 keeps the top
16 bits of an fp32 value). Two independent references pin it:
  * for fp32 inputs, torch's fp32 -> bf16 cast (round to nearest even), on
    exact midpoints, neighbours of midpoints, subnormals, overflow and signs;
  * for fp64 inputs (the oracle rounds fp64 results once), a brute-force
    nearest search: the result is a bf16 value, no bf16 neighbour is strictly
    closer in exact rational arithmetic, and on an exact tie the kept value has
    an even last mantissa bit.
Truncation, ties away from zero, ties to odd or a double rounding through fp32
each fail one of these."""
from fractions import Fraction

import numpy as np
import torch

from oracle.numerics import round_bf16, round_f32_to_bf16


def bits32(x):
    return np.asarray(x, np.float32).view(np.uint32)


def from_bits32(u):
    return np.asarray(u, np.uint32).view(np.float32)


def torch_rne(x32):
    return torch.from_numpy(np.asarray(x32, np.float32)).to(torch.bfloat16).float().numpy()


def special_fp32():
    """Midpoints and their neighbours over many exponents, subnormals, the
    overflow edge, zeros and infinities, both signs."""
    out = []
    for e in list(range(-149, -120)) + list(range(-20, 21)) + list(range(120, 128)):
        for m in (0, 1, 2, 3, 0x7F, 0x80, 0x81, 0x7E):          # bf16 mantissa patterns
            base = (max(e + 127, 0) << 23) | (m << 16)
            for low in (0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF):
                out.append(base | low)
    u = np.array(out, np.uint64)
    u = u[(u & 0x7F800000) != 0x7F800000].astype(np.uint32)   # finite only here
    x = from_bits32(u)
    extra = np.array([0.0, 3.3895313892515355e38, 3.3961775292304172e38, 3.3961776e38,
                      np.finfo(np.float32).max, np.inf, 1.0 + 2**-8, 1.0 + 3 * 2**-8,
                      2**-133, 3 * 2**-134, 2**-134, 2**-135, 1e-45], np.float32)
    x = np.concatenate([x, extra])
    return np.concatenate([x, -x])


def test_fp32_inputs_match_torch_round_to_nearest_even():
    x = special_fp32()
    got = round_bf16(x.astype(np.float64))
    want = torch_rne(x).astype(np.float64)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    bad = np.nonzero(~same)[0]
    assert bad.size == 0, [(hex(int(bits32(x[i]))), got[i], want[i]) for i in bad[:8]]
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[x == 0]), np.signbit(want[x == 0]))


def test_random_fp32_match_torch():
    r = np.random.default_rng(7)
    u = r.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    u = u[(u & 0x7F800000) != 0x7F800000]
    x = from_bits32(u)
    assert np.array_equal(round_bf16(x.astype(np.float64)), torch_rne(x).astype(np.float64))
    assert np.array_equal(round_f32_to_bf16(x), torch_rne(x))


def test_exact_ties_go_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even neighbour is 1
    assert round_bf16(1.0 + 2.0**-8) == 1.0
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert round_bf16(1.0 + 3 * 2.0**-8) == 1.0 + 2.0**-6
    # just above a midpoint rounds up, just below rounds down (no truncation)
    assert round_bf16(1.0 + 2.0**-8 + 2.0**-40) == 1.0 + 2.0**-7
    assert round_bf16(1.0 + 2.0**-7 - 2.0**-40) == 1.0 + 2.0**-7
    assert round_bf16(-(1.0 + 2.0**-8)) == -1.0


def _bf16_neighbours(r):
    """bf16 values just below and above the bf16 value r (as exact Fractions)."""
    b = int(bits32(np.float32(r))) >> 16
    lo = from_bits32(np.uint32(((b - 1) & 0xFFFF) << 16)) if (b & 0x7FFF) else None
    hi = from_bits32(np.uint32(((b + 1) & 0xFFFF) << 16))
    return lo, hi


def test_fp64_inputs_are_rounded_once_to_the_nearest_bf16():
    """Brute force in exact arithmetic: no bf16 value is closer than the result,
    and exact ties keep the even mantissa. A double rounding through fp32 fails
    the inputs that sit just past a bf16 midpoint by less than an fp32 ulp."""
    r = np.random.default_rng(11)
    mids = []
    for e in (-130, -100, -3, 0, 5, 60):
        m = r.integers(0, 128, size=40)
        base = np.ldexp(1.0 + m / 128.0, e)
        half = np.ldexp(1.0, e - 8)
        mids += list(base + half)                               # exact midpoints
        mids += list(base + half + np.ldexp(1.0, e - 8 - 30))   # past them by << fp32 ulp
        mids += list(base + half - np.ldexp(1.0, e - 8 - 30))
    xs = np.concatenate([np.array(mids), r.standard_normal(3000) * 10.0 ** r.integers(-30, 30, 3000)])
    xs = np.concatenate([xs, -xs])
    got = round_bf16(xs)
    for x, g in zip(xs, got):
        gf = np.float32(g)
        assert float(gf) == g and (int(bits32(gf)) & 0xFFFF) == 0, (x, g)   # a bf16 value
        fx, fg = Fraction(float(x)), Fraction(float(g))
        for nb in _bf16_neighbours(g):
            if nb is None or not np.isfinite(nb):
                continue
            d_nb, d_g = abs(fx - Fraction(float(nb))), abs(fx - fg)
            assert d_g <= d_nb, (x, g, float(nb))
            if d_g == d_nb:       # exact tie: the kept value is the even one
                assert (int(bits32(gf)) >> 16) & 1 == 0, (x, g)
    # the double-rounding trap: just past the midpoint 1 + 2^-8 by 2^-38 must round up
    assert round_bf16(1.0 + 2.0**-8 + 2.0**-38) == 1.0 + 2.0**-7


def test_overflow_and_non_finite():
    big = 3.3895313892515355e38            # largest finite bf16
    step = 2.0 ** (127 - 7)                # its spacing
    assert round_bf16(big) == big
    assert round_bf16(big + 0.49 * step) == big
    assert round_bf16(big + 0.5 * step) == np.inf     # the tie rounds to the even (infinity)
    assert round_bf16(-(big + 0.6 * step)) == -np.inf
    assert np.isnan(round_bf16(np.nan))
    assert round_bf16(np.inf) == np.inf and round_bf16(-np.inf) == -np.inf
