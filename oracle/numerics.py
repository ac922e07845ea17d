"""Storage rounding used by the oracle (fp32 and bf16, round to nearest even)."""
import numpy as np


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as
    float64. bf16 keeps 8 significant bits; the quantum of a value with binary
    exponent e (0.5 <= |m| < 1, x = m 2^e) is 2^(e-8), floored at the subnormal
    quantum 2^-133. ``np.round`` rounds half to even."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    _, e = np.frexp(x[fin])
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    out[fin] = np.round(x[fin] / q) * q
    big = np.abs(out) > 3.3895313892515355e38  # beyond the largest finite bf16
    out[big] = np.sign(out[big]) * np.inf
    return out


def round_store(x, dtype: str) -> np.ndarray:
    """Round to the storage dtype ('f32' or 'bf16'); result is float64."""
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        return round_bf16(x)
    raise ValueError(dtype)


def round_f32_to_bf16(x32) -> np.ndarray:
    """Round fp32 values to bf16 (ties to even) and return float32."""
    return round_bf16(np.asarray(x32, dtype=np.float32).astype(np.float64)).astype(np.float32)
