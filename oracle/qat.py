"""FP8 / FP4 quantisation round trips of compressed rows (step 8 of the
compressor) — TEST INFRASTRUCTURE, part of the CPU oracle.

"【#3】ds4.c を読み解く" §4 (step 8) and §9: after RMS normalisation and the
tail RoPE, a compressed row is quantised and dequantised in place before it is
appended. A 512-wide attention row takes an FP8 E4M3 round trip on its
non-RoPE dims; a 128-wide indexer row takes a 128-point Hadamard transform and
an FP4 activation quantisation. The indexer query takes the same QAT round
trip. The round trips exist to match the model's own graph, not to shrink the
cache. §5 gives the order: RMSNorm -> tail RoPE -> round trip -> append. vLLM's
DeepSeek V4 page (memory section) quotes fp8 for the attention cache and fp4 for
the indexer cache.

Readings (the pages give neither the scale granularity nor the arithmetic):
* Q1 FP8: the non-RoPE dims are the leading D - n_rot dims (the RoPE is on the
  tail). They are split into blocks of 64 consecutive dims (the last block may
  be shorter). Each block has one power-of-two scale 2^k, the smallest with
  amax <= 448 * 2^k (448 is E4M3's largest finite value), with k >= -127 (the
  range of an 8-bit exponent scale). Every dim becomes the E4M3 value nearest
  x / 2^k (ties to the even code), times 2^k. The RoPE dims are unchanged.
* Q2 FP4: with n = Di (a power of two, >= 32), z = c * H x, where H is the
  Sylvester Hadamard matrix (H[i][j] = (-1)^popcount(i & j)) and
  c = 1/sqrt(n) rounded to fp32 (n = 128: the 128-point transform). z is
  split into blocks of 32. Each block has a power-of-two scale 2^k, the smallest
  with amax <= 6 * 2^k (6 is E2M1's largest value), k >= -127. Every element
  becomes the E2M1 value nearest z / 2^k (ties to the even code), times 2^k.
  The result goes back through the same transform, x' = c * H z'. H / sqrt(n)
  is its own inverse, so the row stays in its own basis.
* Q3 the decisions (scales, codes) are integers, so both round trips run in
  fp32 (the pages' CPU reference is float code) in one fixed order:
  - the row arrives rounded to fp32;
  - H is the radix-2 butterfly over stages h = 1, 2, 4, ..., n/2, each pair
    (a at i, b at i + h, i & h == 0) becoming (a + b, a - b), one rounding per
    operation;
  - then the multiplication by c.
  Scaling by 2^k is exact. The attention row's RoPE dims keep their fp64
  value, and the row is rounded once to the storage dtype. The FP8 dims are
  exact in bf16 and fp32.
* Q4 the cache keeps the dequantised values in its storage dtype. The pages'
  round trip is in place.

The function names say which step they implement. The GPU library has its own
code for each, and none of it is shared with this module.
"""
import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0
FP8_BLOCK = 64
FP4_BLOCK = 32
MIN_SCALE_EXP = -127


def _decode_table(exp_bits: int, man_bits: int, bias: int, nan_codes=()):
    """Non-negative finite values of a sign/exponent/mantissa format with
    subnormals, indexed by code (sign bit clear). Codes in nan_codes are
    dropped. Returns (values, codes) in code order."""
    vals, codes = [], []
    for code in range(1 << (exp_bits + man_bits)):
        if code in nan_codes:
            continue
        e, m = code >> man_bits, code & ((1 << man_bits) - 1)
        if e == 0:
            v = (m / (1 << man_bits)) * 2.0 ** (1 - bias)
        else:
            v = (1 + m / (1 << man_bits)) * 2.0 ** (e - bias)
        vals.append(v)
        codes.append(code)
    return np.array(vals, np.float64), np.array(codes, np.int64)


def e4m3_table():
    """OCP FP8 E4M3 (the 'fn' variant: no infinities, exponent bias 7, code
    0x7F is NaN): 127 finite non-negative values, 0 .. 448."""
    return _decode_table(4, 3, 7, nan_codes=(0x7F,))


def e2m1_table():
    """OCP FP4 E2M1 (exponent bias 1, no NaN or infinity): 0, 0.5, 1, 1.5, 2,
    3, 4, 6."""
    return _decode_table(2, 1, 1)


def round_to_table(r, table) -> np.ndarray:
    """Nearest table value to each r (|r| <= the table's max), ties to the
    value whose code is even; the sign of r is kept (-0 for a negative r that
    rounds to 0)."""
    vals, codes = table
    r = np.asarray(r, np.float64)
    a = np.abs(r).ravel()
    assert np.all(a <= vals[-1]), "value beyond the format's range"
    d = np.abs(a[:, None] - vals[None, :])
    best = d.min(axis=1, keepdims=True)
    near = d == best
    # among equidistant values (at most two), the even code wins
    pick = np.where(near & (codes[None, :] % 2 == 0), 1, 0) + near
    idx = np.argmax(pick, axis=1)
    out = vals[idx].reshape(r.shape)
    return np.copysign(out, r)


def block_scale_exp(amax: float, qmax: float) -> int:
    """Smallest integer k >= -127 with amax <= qmax * 2^k (exact comparisons)."""
    amax = float(amax)
    if amax <= qmax * 2.0 ** MIN_SCALE_EXP:
        return MIN_SCALE_EXP
    k = int(np.frexp(amax)[1]) - int(np.frexp(qmax)[1])
    while amax > qmax * 2.0 ** k:
        k += 1
    while k - 1 >= MIN_SCALE_EXP and amax <= qmax * 2.0 ** (k - 1):
        k -= 1
    return k


def quantise_blocks(x, block: int, qmax: float, table) -> np.ndarray:
    """Round trip of the last axis of x through a block-scaled format (Q1/Q2):
    per block of `block` consecutive elements a power-of-two scale, then the
    nearest format value. Exact arithmetic (float64 holds every step)."""
    x = np.asarray(x, np.float64)
    out = np.empty_like(x)
    flat, res = x.reshape(-1, x.shape[-1]), out.reshape(-1, x.shape[-1])
    n = x.shape[-1]
    for row in range(flat.shape[0]):
        for b0 in range(0, n, block):
            seg = flat[row, b0:b0 + block]
            k = block_scale_exp(np.max(np.abs(seg)) if seg.size else 0.0, qmax)
            res[row, b0:b0 + block] = round_to_table(seg * 2.0 ** -k, table) * 2.0 ** k
    return out


def fwht_f32(x) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform of the last axis in fp32 (Q3):
    radix-2 butterflies over stages h = 1, 2, ..., n/2."""
    v = np.array(x, np.float32, copy=True)
    n = v.shape[-1]
    assert n >= 1 and n & (n - 1) == 0
    h = 1
    while h < n:
        shp = v.shape[:-1] + (n // (2 * h), 2, h)
        w = v.reshape(shp)
        a, b = w[..., 0, :].copy(), w[..., 1, :].copy()
        w[..., 0, :] = a + b
        w[..., 1, :] = a - b
        v = w.reshape(v.shape)
        h *= 2
    return v


def hadamard_scale(n: int) -> np.float32:
    """c = 1/sqrt(n) rounded to fp32."""
    return np.float32(1.0 / np.sqrt(np.float64(n)))


def fp8_round_trip(x32, block: int = FP8_BLOCK) -> np.ndarray:
    """Q1 on fp32 values (last axis): E4M3 with per-block power-of-two scales.
    Returns the exact dequantised values as float64."""
    return quantise_blocks(np.asarray(x32, np.float32), block, E4M3_MAX, e4m3_table())


def fp4_qat_round_trip(x32) -> np.ndarray:
    """Q2/Q3 on fp32 vectors (last axis, length a power of two >= 32):
    Hadamard, E2M1 with per-32 power-of-two scales, Hadamard back; fp32."""
    x32 = np.asarray(x32, np.float32)
    c = hadamard_scale(x32.shape[-1])
    z = fwht_f32(x32) * c
    zq = quantise_blocks(z, FP4_BLOCK, E2M1_MAX, e2m1_table()).astype(np.float32)
    return fwht_f32(zq) * c


def attn_row_round_trip(row, n_rot: int) -> np.ndarray:
    """Q1 applied to compressed attention rows (last axis D): the leading
    D - n_rot dims go through the FP8 round trip from their fp32 values, the
    RoPE tail keeps its value. float64 out (rounded to storage by the caller)."""
    row = np.asarray(row, np.float64)
    out = row.copy()
    n_nope = row.shape[-1] - n_rot
    if n_nope > 0:
        out[..., :n_nope] = fp8_round_trip(row[..., :n_nope].astype(np.float32))
    return out


def index_row_round_trip(row) -> np.ndarray:
    """Q2 applied to compressed indexer rows (last axis Di) from their fp32
    values; float64 out (rounded to storage by the caller)."""
    return fp4_qat_round_trip(np.asarray(row, np.float64).astype(np.float32)).astype(np.float64)
