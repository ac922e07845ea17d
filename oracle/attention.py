"""Sparse attention over the raw window plus compressed rows (K = V).

"【#3】ds4.c を読み解く" §7: the attended set is the raw window rows of positions
max(first_raw, qpos + 1 - window) .. min(qpos, raw_last) together with the
top-k compressed rows (negative index: skipped; index >= visible: stop), all
under one softmax. vLLM's page: keys and values are the same vectors, the
output gets the inverse rotation; c128a layers attend every visible compressed
row (no indexer on ratio-128 layers); a ratio-0 layer sees the window only.

Readings:
* R10 scale 1/sqrt(D) unless given; no sink or bias; rows attended twice (a
  token in the window and inside a selected compressed row) are not merged.
* The query's tail is rotated at its position with the layer's base; the
  output's tail is rotated back by the same angle (R12).
* Computed in fp64 from the stored values; the output is rounded to the
  storage dtype.
"""
import numpy as np

from .numerics import round_store
from .rope import rope_tail


def attend(q_rot, rows, scale: float) -> np.ndarray:
    """softmax(q_rot rows^T * scale) rows for q_rot [H, D], rows [n, D] (fp64)."""
    q = np.asarray(q_rot, np.float64)
    K = np.asarray(rows, np.float64)
    if K.shape[0] == 0:
        return np.zeros_like(q)
    s = (q @ K.T) * scale
    s = s - np.max(s, axis=-1, keepdims=True)
    e = np.exp(s)
    return (e / np.sum(e, axis=-1, keepdims=True)) @ K


def window_positions(p: int, cap_raw: int) -> np.ndarray:
    return np.arange(max(0, p - cap_raw + 1), p + 1)


def comp_row_ids(ratio: int, p: int, n_comp: int, topk=None) -> np.ndarray:
    """Compressed rows attended by a query at p (ratio 4: the top-k list)."""
    if ratio == 0:
        return np.zeros(0, np.int64)
    vis = min((p + 1) // ratio, n_comp)
    if ratio == 128:
        return np.arange(vis)
    ids = []
    for idx in np.asarray(topk):
        if idx < 0:
            continue
        if idx >= vis:
            break
        ids.append(int(idx))
    return np.asarray(ids, np.int64)


def attention_query(q, p: int, window_rows, comp_rows, base: float, n_rot: int, scale: float,
                    dtype: str) -> np.ndarray:
    """One query: q [H, D] before rotation; window_rows [nw, D] and comp_rows
    [nc, D] stored (already rotated) rows. Returns [H, D] in storage precision."""
    q_rot = rope_tail(q, p, base, n_rot)
    rows = np.concatenate([np.asarray(window_rows, np.float64).reshape(-1, q.shape[-1]),
                           np.asarray(comp_rows, np.float64).reshape(-1, q.shape[-1])])
    o = attend(q_rot, rows, scale)
    return round_store(rope_tail(o, p, base, n_rot, inverse=True), dtype)
