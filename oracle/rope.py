"""Tail-only rotary position embedding.

"【#3】ds4.c を読み解く" §8: only the last n_rot = 64 dims of a head rotate; the
first head_dim - n_rot dims are left alone; a compressed layer (ratio != 0)
uses the compression frequency base instead of the normal one. vLLM's page
("DeepSeek V4 アテンションアーキテクチャ", shared K=V) applies the inverse
rotation to the attention output.

Readings (the pages do not give them):
* pairs are adjacent, (x[n_nope + 2i], x[n_nope + 2i + 1]) for i < n_rot / 2,
  rotated by angle p * theta_i with theta_i = base^(-2i / n_rot);
* the angle and its cos / sin are computed in fp64 and each cos / sin is then
  rounded to fp32: these fp32 numbers ARE the rotation's coefficients (an fp32
  angle at p ~ 1.3e5 would be off by ~1e-2 rad);
* the indexer rotates min(64, Di) tail dims of its rows and queries.
"""
import math

import numpy as np

_cos = np.vectorize(math.cos, otypes=[np.float64])
_sin = np.vectorize(math.sin, otypes=[np.float64])


def inv_freq(base: float, n_rot: int) -> np.ndarray:
    """theta_i = base^(-2i / n_rot), fp64 (C library pow)."""
    return np.array([math.pow(base, -2.0 * i / n_rot) for i in range(n_rot // 2)])


def rope_coeffs(pos, base: float, n_rot: int):
    """fp32 cos / sin of p * theta_i, shape pos.shape + (n_rot/2,), as float32.
    The angle is one fp64 product; cos and sin are the C library's fp64
    functions (argument reduction included), each rounded once to fp32."""
    pos = np.asarray(pos, dtype=np.float64)
    ang = pos[..., None] * inv_freq(base, n_rot)
    return _cos(ang).astype(np.float32), _sin(ang).astype(np.float32)


def rope_tail(x, pos, base: float, n_rot: int, inverse: bool = False) -> np.ndarray:
    """Rotate the tail of x[..., D] in fp64; ``pos`` broadcasts to x.shape[:-1]."""
    x = np.array(x, dtype=np.float64, copy=True)
    D = x.shape[-1]
    n_nope = D - n_rot
    c, s = rope_coeffs(np.broadcast_to(pos, x.shape[:-1]), base, n_rot)
    c = c.astype(np.float64)
    s = -s.astype(np.float64) if inverse else s.astype(np.float64)
    a = x[..., n_nope::2].copy()
    b = x[..., n_nope + 1::2].copy()
    x[..., n_nope::2] = a * c - b * s
    x[..., n_nope + 1::2] = a * s + b * c
    return x


def rope_tail_f32(x32, pos, base: float, n_rot: int) -> np.ndarray:
    """The same rotation in fp32, one rounding per operation and no fused
    multiply-add: a' = (a c) - (b s), b' = (a s) + (b c). Used where the result
    feeds an integer decision (the indexer's top-k)."""
    x = np.array(x32, dtype=np.float32, copy=True)
    D = x.shape[-1]
    n_nope = D - n_rot
    c, s = rope_coeffs(np.broadcast_to(pos, x.shape[:-1]), base, n_rot)
    a = x[..., n_nope::2].copy()
    b = x[..., n_nope + 1::2].copy()
    x[..., n_nope::2] = (a * c) - (b * s)
    x[..., n_nope + 1::2] = (a * s) + (b * c)
    return x
