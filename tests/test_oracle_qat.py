"""Pins of oracle.qat (the compressor's step 8 round trips), each checked
against something other than the oracle's own formula:

* the E4M3 and E2M1 value tables against facts of the OCP formats (extremes,
  counts, known codes) and, for E4M3, torch's own fp8 conversion;
* rounding ties against hand-worked cases;
* the power-of-two block scale at its boundaries;
* the fp32 butterfly against the Hadamard matrix written out entry by entry,
  and the transform's involution;
* closed forms of both round trips (the all-ones indexer row, rows already on
  the grid), their error bounds, block independence, and their place in the
  compressor (RoPE dims untouched, the indexer query)."""
import numpy as np
import pytest
import torch

from oracle import qat
from oracle.compressor import Lane, lane_step, rms_norm, softmax_pool
from oracle.indexer import rotate_index_query
from oracle.layer import OracleCache, QAT_FP4_INDEX, QAT_FP8_ATTN, compress_append
from oracle.rope import rope_tail, rope_tail_f32


def rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ tables

def test_e4m3_table_facts():
    vals, codes = qat.e4m3_table()
    assert len(vals) == 127 and vals[0] == 0.0 and vals[-1] == 448.0
    assert np.all(np.diff(vals) > 0)                 # codes are ordered
    by = dict(zip(codes.tolist(), vals.tolist()))
    assert by[0x01] == 2.0 ** -9                     # smallest subnormal
    assert by[0x07] == 7 * 2.0 ** -9                 # largest subnormal
    assert by[0x08] == 2.0 ** -6                     # smallest normal
    assert by[0x38] == 1.0 and by[0x40] == 2.0 and by[0x7E] == 448.0
    assert 0x7F not in by                            # NaN


def test_e2m1_table():
    vals, codes = qat.e2m1_table()
    assert vals.tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert codes.tolist() == list(range(8))


def test_e4m3_rounding_matches_torch_fp8_cast():
    """Nearest-even rounding to E4M3 equals torch's float8_e4m3fn cast on
    fp32 values within range (normals, subnormals, exact ties)."""
    r = rng(1)
    x = np.concatenate([
        r.uniform(-448, 448, 4000), r.uniform(-1, 1, 2000) * 2.0 ** -6,
        r.standard_normal(2000),
        # every midpoint between neighbouring values (exact ties)
        (qat.e4m3_table()[0][1:] + qat.e4m3_table()[0][:-1]) / 2,
    ]).astype(np.float32)
    got = qat.round_to_table(x, qat.e4m3_table())
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(got.astype(np.float32), ref)


@pytest.mark.parametrize("x,want", [
    (0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0),
    (5.0, 4.0), (5.01, 6.0), (0.26, 0.5), (0.24, 0.0), (6.0, 6.0), (-1.75, -2.0),
    (-0.1, -0.0)])
def test_e2m1_rounding_ties_to_even(x, want):
    got = qat.round_to_table(np.array([x]), qat.e2m1_table())[0]
    assert got == want and np.signbit(got) == np.signbit(want)


# ------------------------------------------------------------------ scales

@pytest.mark.parametrize("amax,qmax,k", [
    (448.0, 448.0, 0), (448.0 * (1 + 2.0 ** -40), 448.0, 1), (224.0, 448.0, -1),
    (224.0 * (1 + 2.0 ** -40), 448.0, 0), (1.0, 448.0, -8), (6.0, 6.0, 0), (6.5, 6.0, 1),
    (3.0, 6.0, -1), (0.0, 6.0, -127), (1e-45, 448.0, -127), (1e30, 6.0, 98)])
def test_block_scale_boundaries(amax, qmax, k):
    assert qat.block_scale_exp(amax, qmax) == k
    if amax > 0 and k > -127:
        assert amax <= qmax * 2.0 ** k and amax > qmax * 2.0 ** (k - 1)


# ------------------------------------------------------------------ Hadamard

@pytest.mark.parametrize("n", [1, 2, 8, 32, 128])
def test_fwht_equals_sylvester_matrix(n):
    """Small-integer inputs keep every fp32 sum exact, so the butterfly must
    equal H x with H[i][j] = (-1)^popcount(i & j) written out entry by entry."""
    H = np.array([[(-1) ** bin(i & j).count("1") for j in range(n)] for i in range(n)],
                 np.float64)
    x = rng(n).integers(-50, 50, (5, n)).astype(np.float32)
    assert np.array_equal(qat.fwht_f32(x).astype(np.float64), x.astype(np.float64) @ H.T)


def test_fwht_involution_and_orthonormal_scale():
    x = rng(3).integers(-1000, 1000, (4, 128)).astype(np.float32)
    assert np.array_equal(qat.fwht_f32(qat.fwht_f32(x)), 128 * x)
    c = qat.hadamard_scale(128)
    assert c == np.float32(0.08838834764831845)
    y = rng(4).standard_normal((4, 128)).astype(np.float32)
    z = qat.fwht_f32(y) * c
    assert np.allclose(np.linalg.norm(z, axis=1), np.linalg.norm(y, axis=1), rtol=1e-5)


# ------------------------------------------------------------------ FP8 rows

def test_fp8_round_trip_grid_bound_and_idempotence():
    r = rng(5)
    x = (r.standard_normal((6, 448)) * r.uniform(0.01, 100, (6, 1))).astype(np.float32)
    y = qat.fp8_round_trip(x)
    vals = qat.e4m3_table()[0]
    for row in range(6):
        for b in range(7):
            seg, q = x[row, 64 * b:64 * b + 64].astype(np.float64), y[row, 64 * b:64 * b + 64]
            k = qat.block_scale_exp(np.abs(seg).max(), 448.0)
            assert np.all(np.isin(np.abs(q) * 2.0 ** -k, vals))        # on the scaled grid
            # at most half a step: relative 2^-4 for normals, 2^-10 * 2^k below
            assert np.all(np.abs(q - seg) <= np.maximum(np.abs(seg) * 2.0 ** -4,
                                                        2.0 ** (k - 10)))
    assert np.array_equal(qat.fp8_round_trip(y.astype(np.float32)), y)


def test_fp8_blocks_are_independent_and_scale_exactly():
    """Scaling one 64-dim block by 2^j scales its output by 2^j and leaves the
    other blocks alone; a block-wide scale would quantise the small block to 0."""
    x = rng(6).standard_normal((1, 448)).astype(np.float32)
    y = qat.fp8_round_trip(x)
    x2 = x.copy()
    x2[0, 64:128] *= np.float32(2.0 ** 20)
    y2 = qat.fp8_round_trip(x2)
    assert np.array_equal(y2[0, 64:128], y[0, 64:128] * 2.0 ** 20)
    assert np.array_equal(np.delete(y2, np.s_[64:128], axis=1), np.delete(y, np.s_[64:128], axis=1))
    assert np.count_nonzero(y2[0, :64]) > 50


def test_fp8_ragged_last_block_and_zero_block():
    x = rng(7).standard_normal((2, 100)).astype(np.float32)
    x[1, :64] = 0
    y = qat.fp8_round_trip(x)
    assert np.array_equal(y[1, :64], np.zeros(64))
    k = qat.block_scale_exp(np.abs(x[0, 64:]).max(), 448.0)
    assert np.all(np.isin(np.abs(y[0, 64:]) * 2.0 ** -k, qat.e4m3_table()[0]))


def test_attn_row_round_trip_leaves_rope_tail():
    row = rng(8).standard_normal((3, 512))
    out = qat.attn_row_round_trip(row, 64)
    assert np.array_equal(out[:, 448:], row[:, 448:])
    assert np.array_equal(out[:, :448], qat.fp8_round_trip(row[:, :448].astype(np.float32)))
    assert np.array_equal(qat.attn_row_round_trip(row, 512), row)   # all dims rotated


# ------------------------------------------------------------------ FP4 QAT

def test_fp4_all_ones_closed_form():
    """H 1 = 128 e_0, so z = 128 c e_0 = 11.31; its block scale is 2 (11.31 <= 12),
    z/2 = 5.66 rounds to 6, z' = 12 e_0 and x' = c H (12 e_0) = 12 c everywhere."""
    x = np.ones((1, 128), np.float32)
    c = qat.hadamard_scale(128)
    y = qat.fp4_qat_round_trip(x)
    assert np.array_equal(y, np.full((1, 128), np.float32(12) * c, np.float32))


def test_fp4_on_grid_rows_survive_and_blocks_are_independent():
    """x = c H z with z on each block's own grid (block 0 small, block 1 large)
    comes back within fp32 rounding; one scale for the whole row would wipe
    block 0."""
    z = np.zeros((1, 128), np.float32)
    z[0, 0:4] = [0.5, -1.5, 3.0, 4.0]       # amaxes kept off the scale boundaries
    z[0, 32:36] = [4.0 * 2 ** 8, -3.0 * 2 ** 8, 2 ** 8, 0.5 * 2 ** 8]
    c = qat.hadamard_scale(128)
    x = qat.fwht_f32(z) * c
    y = qat.fp4_qat_round_trip(x)
    zz = qat.fwht_f32(y) * c
    assert np.allclose(zz, z, rtol=0, atol=5e-3)
    assert np.count_nonzero(np.abs(zz[0, :4]) > 0.4) == 4


def test_fp4_error_bound_and_zero():
    r = rng(9)
    x = r.standard_normal((8, 128)).astype(np.float32)
    y = qat.fp4_qat_round_trip(x)
    c = qat.hadamard_scale(128)
    z = (qat.fwht_f32(x) * c).astype(np.float64)
    bound = 0
    for b in range(4):
        amax = np.abs(z[:, 32 * b:32 * b + 32]).max(axis=1)
        s = np.array([2.0 ** qat.block_scale_exp(a, 6.0) for a in amax])
        bound = bound + 32 * (s * 1.0) ** 2          # half of the widest step (2 s)
    err = np.linalg.norm(y.astype(np.float64) - x, axis=1)
    assert np.all(err <= np.sqrt(bound) * 1.001)
    assert np.all(err > 0)
    assert np.array_equal(qat.fp4_qat_round_trip(np.zeros((1, 32), np.float32)),
                          np.zeros((1, 32), np.float32))


def test_fp4_quantiser_fixes_its_own_grid():
    """The block quantiser maps its own output to itself (every block's amax
    is then a grid value times its scale, so the scale and codes repeat). The
    whole round trip is not idempotent in fp32: a block whose largest code is 6
    can come back a rounding above 6 * 2^k and take the next scale."""
    r = rng(10)
    z = (r.standard_normal((16, 128)) * r.uniform(0.1, 50, (16, 1))).astype(np.float32)
    t = qat.e2m1_table()
    zq = qat.quantise_blocks(z, 32, 6.0, t)
    assert np.array_equal(qat.quantise_blocks(zq, 32, 6.0, t), zq)


# ------------------------------------------------------------------ in the layer

def _lane(width, n_rot, quant, seed):
    r = rng(seed)
    W = 8
    skv = r.standard_normal((2, W, width)).astype(np.float32)
    ssc = r.standard_normal((2, W, width)).astype(np.float32)
    ape = r.standard_normal((W, width)) * 0.1
    gam = 1 + 0.1 * r.standard_normal(width)
    return Lane(skv.copy(), ssc.copy(), np.zeros((2, 4, width)), ape, gam, n_rot, quant,
                np.zeros((2, 4, width))), (skv, ssc, ape, gam)


@pytest.mark.parametrize("quant,width,n_rot", [("fp8", 512, 64), ("fp4", 128, 64)])
def test_lane_step_applies_step8_after_rope(quant, width, n_rot):
    """The round trip sits after RMSNorm and the tail RoPE (and before the
    storage rounding): the stored row equals the round trip of the row the
    lane builds without it."""
    lane, (skv, ssc, ape, gam) = _lane(width, n_rot, quant, 11)
    p = 7                                   # row 1 of a ratio-4 lane
    lane_step(lane, 4, p, skv[:, 4 + p % 4], ssc[:, 4 + p % 4], 10000.0, "bf16")
    pooled = softmax_pool(skv, ssc, ape)
    row = rope_tail(rms_norm(pooled, gam), 4, 10000.0, n_rot)
    assert np.allclose(lane.pre[:, 1], row, rtol=1e-12, atol=1e-12)
    fn = qat.attn_row_round_trip if quant == "fp8" else (
        lambda r_, n: qat.index_row_round_trip(r_))
    from oracle.numerics import round_bf16
    assert np.array_equal(lane.comp[:, 1], round_bf16(fn(lane.pre[:, 1], n_rot)))
    if quant == "fp8":   # E4M3 values times 2^k are bf16 values: no second rounding
        assert np.array_equal(lane.comp[:, 1, :448], fn(lane.pre[:, 1], n_rot)[:, :448])


def test_index_query_qat_between_rope_and_storage():
    r = rng(12)
    q = r.standard_normal((2, 64, 128)).astype(np.float32)
    plain = rotate_index_query(q, 1000, 10000.0, 64, "bf16")
    got = rotate_index_query(q, 1000, 10000.0, 64, "bf16", qat=True)
    rot = rope_tail_f32(q, 1000, 10000.0, 64)
    from oracle.numerics import round_f32_to_bf16
    assert np.array_equal(got, round_f32_to_bf16(qat.fp4_qat_round_trip(rot)))
    assert not np.array_equal(got, plain)


def test_cache_flags_select_lanes():
    """qat bit 0 touches only attention rows, bit 1 only indexer rows."""
    r = rng(13)
    B, D, Di, T = 1, 512, 128, 8
    base = dict(ratio=4, head_dim=D, n_rot=64, cap_raw=128, base=10000.0, dtype="bf16",
                n_tokens=0, index_dim=Di, index_rot=64)

    def mk(q):
        return OracleCache(**base, qat=q, raw_kv=np.zeros((B, 128, D)),
                           attn_comp_kv=np.zeros((B, 4, D)),
                           attn_state_kv=np.zeros((B, 8, D)),
                           attn_state_score=np.full((B, 8, D), -np.inf),
                           index_comp_kv=np.zeros((B, 4, Di)),
                           index_state_kv=np.zeros((B, 8, Di)),
                           index_state_score=np.full((B, 8, Di), -np.inf))
    inp = {"raw_kv_in": r.standard_normal((B, T, D)),
           "attn_cand": r.standard_normal((B, T, D)), "attn_score": r.standard_normal((B, T, D)),
           "idx_cand": r.standard_normal((B, T, Di)), "idx_score": r.standard_normal((B, T, Di)),
           "ape_attn": 0.1 * r.standard_normal((8, D)), "gamma_attn": np.ones(D),
           "ape_idx": 0.1 * r.standard_normal((8, Di)), "gamma_idx": np.ones(Di)}
    cs = {q: mk(q) for q in (0, QAT_FP8_ATTN, QAT_FP4_INDEX)}
    for c in cs.values():
        compress_append(c, 0, inp, chunk=True)
    assert not np.array_equal(cs[QAT_FP8_ATTN].attn_comp_kv, cs[0].attn_comp_kv)
    assert np.array_equal(cs[QAT_FP8_ATTN].index_comp_kv, cs[0].index_comp_kv)
    assert np.array_equal(cs[QAT_FP4_INDEX].attn_comp_kv, cs[0].attn_comp_kv)
    assert not np.array_equal(cs[QAT_FP4_INDEX].index_comp_kv, cs[0].index_comp_kv)
    assert np.array_equal(cs[QAT_FP8_ATTN].attn_comp_kv[..., 448:], cs[0].attn_comp_kv[..., 448:])
