"""Ratio-4 indexer: score every visible compressed index row, keep the top k.

"【#3】ds4.c を読み解く" §6: on ratio-4 layers an indexer with its own heads
(Flash: 64 heads x 128 dims, top-k 512) scores the compressed index rows and
its output decides which compressed rows the attention sees; §7 the attention
skips negative indices and stops at indices >= the visible count. vLLM's page
(DSA): only the top-k compressed tokens are attended.

Readings (the pages give no formula):
* R9 score I(t, s) = sum_h w_h(t) * ReLU(q'_h(t) . k_s), q' = the indexer query
  with its tail rotated at the query's position. Any positive scale leaves the
  ranking alone; the ReLU is the one assumption.
* The score decides integers, so it is defined in fp32 (the pages' CPU
  reference works in float) in this exact order, one rounding per operation and
  no fused multiply-add: dot_h = ((q_0 k_0) + (q_1 k_1)) + ... in ascending d;
  r_h = dot_h if dot_h > 0 else +0; I = ((w_0 r_0) + (w_1 r_1)) + ... in
  ascending h, starting from +0. The rotated query is rounded to the storage
  dtype before scoring (it is a bf16 activation in the bf16 workloads).
  With the QAT round trip enabled (§9: the indexer query takes it too), it
  runs on the fp32 rotated query before that rounding (``qat.py``).
* Visible rows for a query at position p: s < floor((p + 1) / 4) (a row emitted
  at p is visible to p: the append runs before the indexer).
* Top-k: the k largest scores, ties to the lower row index; the kept indices
  are returned in ascending order, padded with -1 when fewer than k are visible.
"""
import numpy as np

from .numerics import round_f32_to_bf16
from .qat import fp4_qat_round_trip
from .rope import rope_tail_f32


def visible_rows(ratio: int, p: int) -> int:
    return (p + 1) // ratio


def rotate_index_query(q_idx, p, base: float, index_rot: int, dtype: str,
                       qat: bool = False) -> np.ndarray:
    """q' = tail rotation of q_idx[..., Hi, Di] at p (fp32 recipe), then the
    FP4 QAT round trip when enabled, stored dtype."""
    q = rope_tail_f32(np.asarray(q_idx, np.float32), p, base, index_rot)
    if qat:
        q = fp4_qat_round_trip(q)
    return round_f32_to_bf16(q) if dtype == "bf16" else q


def index_scores(q_rot, w, keys) -> np.ndarray:
    """fp32 scores of rows keys[n, Di] for one query (q_rot [Hi, Di], w [Hi])."""
    q = np.asarray(q_rot, np.float32)
    w = np.asarray(w, np.float32)
    k = np.asarray(keys, np.float32)
    n, Di = k.shape
    Hi = q.shape[0]
    dot = np.zeros((n, Hi), np.float32)
    for d in range(Di):
        dot = dot + k[:, d:d + 1] * q[None, :, d]
    tot = np.zeros(n, np.float32)
    for h in range(Hi):
        r = np.where(dot[:, h] > 0, dot[:, h], np.float32(0.0)).astype(np.float32)
        tot = tot + w[h] * r
    return tot


def topk_select(scores, vis: int, k: int) -> np.ndarray:
    """Indices of the k largest of scores[:vis] (ties: lower index), ascending,
    padded with -1."""
    out = np.full(k, -1, np.int32)
    if vis <= k:
        out[:vis] = np.arange(vis, dtype=np.int32)
        return out
    sc = np.asarray(scores[:vis], np.float64)
    order = np.lexsort((np.arange(vis), -sc))    # by score desc, then index asc
    out[:] = np.sort(order[:k]).astype(np.int32)
    return out


def index_topk_query(q_idx, w, keys, p: int, base: float, index_rot: int, dtype: str,
                     k: int, qat: bool = False) -> np.ndarray:
    """Top-k row list of one query at position p."""
    vis = min(visible_rows(4, p), keys.shape[0])
    if vis <= k:
        return topk_select(None, vis, k)
    q_rot = rotate_index_query(q_idx, p, base, index_rot, dtype, qat)
    return topk_select(index_scores(q_rot, w, keys[:vis]), vis, k)
