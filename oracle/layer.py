"""One attention layer of the compressed-KV family: cache, append, indexer
top-k and sparse attention, composed in the order a step runs them.

Per-layer cache ("【#3】ds4.c を読み解く" §2): raw_kv ring of cap_raw rows
(slot = position mod cap_raw), attn_comp_kv with the attention lane's state,
and on ratio-4 layers index_comp_kv with the indexer lane's state. Order of a
step (§4-§7): append (raw row, both lanes' compressor) -> indexer top-k
(ratio 4) -> attention. A prefill chunk keeps the ring as it was before the
chunk until its attention is done (early queries of the chunk still need the
older window rows) and then writes the chunk's last rows into the ring.

``qat`` enables step 8 of the compressor (§4, §9): bit 0 the FP8 round trip of
compressed attention rows, bit 1 the FP4 QAT round trip of compressed indexer
rows and of the indexer query (``qat.py``). ``keep_pre`` records every
compressed row as it was before that step (``attn_pre`` / ``index_pre``).
"""
import numpy as np

from .attention import attention_query, comp_row_ids, window_positions
from .compressor import Lane, lane_step, raw_rows
from .indexer import index_topk_query

QAT_FP8_ATTN = 1
QAT_FP4_INDEX = 2


class OracleCache:
    """Numpy copy of one layer's cache for B sequences.

    Rows hold the exact values of their storage dtype as float64; the state is
    float32 (the library keeps the state in fp32)."""

    def __init__(self, *, ratio, head_dim, n_rot, cap_raw, base, dtype, n_tokens,
                 raw_kv, index_dim=0, index_rot=0, attn_comp_kv=None, attn_state_kv=None,
                 attn_state_score=None, index_comp_kv=None, index_state_kv=None,
                 index_state_score=None, qat=0, keep_pre=False):
        self.ratio, self.head_dim, self.n_rot = ratio, head_dim, n_rot
        self.cap_raw, self.base, self.dtype = cap_raw, base, dtype
        self.index_dim, self.index_rot = index_dim, index_rot
        self.n_tokens = n_tokens
        f64 = lambda a: None if a is None else np.array(a, np.float64)
        f32 = lambda a: None if a is None else np.array(a, np.float32)
        self.raw_kv = f64(raw_kv)
        self.attn_comp_kv, self.index_comp_kv = f64(attn_comp_kv), f64(index_comp_kv)
        self.attn_state_kv, self.attn_state_score = f32(attn_state_kv), f32(attn_state_score)
        self.index_state_kv, self.index_state_score = f32(index_state_kv), f32(index_state_score)
        self.qat = qat
        pre = lambda a: None if (a is None or not keep_pre) else np.full(a.shape, np.nan)
        self.attn_pre, self.index_pre = pre(self.attn_comp_kv), pre(self.index_comp_kv)

    @property
    def n_comp(self) -> int:
        return 0 if self.ratio == 0 else self.n_tokens // self.ratio

    def lanes(self, w):
        out = []
        if self.ratio:
            out.append((Lane(self.attn_state_kv, self.attn_state_score, self.attn_comp_kv,
                             w["ape_attn"], w["gamma_attn"], self.n_rot,
                             "fp8" if self.qat & QAT_FP8_ATTN else None, self.attn_pre),
                        "attn_cand", "attn_score"))
        if self.ratio == 4:
            out.append((Lane(self.index_state_kv, self.index_state_score, self.index_comp_kv,
                             w["ape_idx"], w["gamma_idx"], self.index_rot,
                             "fp4" if self.qat & QAT_FP4_INDEX else None, self.index_pre),
                        "idx_cand", "idx_score"))
        return out


def compress_append(c: OracleCache, pos0: int, inp, chunk: bool):
    """Append tokens pos0 .. pos0+T-1. Returns the rotated raw rows [B, T, D].

    chunk=False (decode): each raw row goes into the ring at once.
    chunk=True (prefill): the ring is left alone; ``commit_ring`` writes it."""
    assert pos0 == c.n_tokens
    raw_in = np.asarray(inp["raw_kv_in"], np.float64)
    T = raw_in.shape[1]
    rows = raw_rows(raw_in, pos0, c.base, c.n_rot, c.dtype)
    lanes = c.lanes(inp)
    for t in range(T):
        p = pos0 + t
        if not chunk:
            c.raw_kv[:, p % c.cap_raw] = rows[:, t]
        for lane, kc, ks in lanes:
            lane_step(lane, c.ratio, p, np.asarray(inp[kc], np.float32)[:, t],
                      np.asarray(inp[ks], np.float32)[:, t], c.base, c.dtype)
    c.n_tokens = pos0 + T
    return rows


def commit_ring(c: OracleCache, pos0: int, rows):
    T = rows.shape[1]
    for t in range(max(0, T - c.cap_raw), T):
        c.raw_kv[:, (pos0 + t) % c.cap_raw] = rows[:, t]


def index_topk(c: OracleCache, pos0: int, q_idx, w, k: int, queries=None) -> np.ndarray:
    """[B, T, k] top-k lists for queries at pos0 .. pos0+T-1 (``queries``: a
    subset of (b, t) pairs to compute; others stay -1)."""
    q_idx = np.asarray(q_idx, np.float32)
    w = np.asarray(w, np.float32)
    B, T = q_idx.shape[:2]
    out = np.full((B, T, k), -1, np.int32)
    todo = queries if queries is not None else [(b, t) for b in range(B) for t in range(T)]
    for b, t in todo:
        out[b, t] = index_topk_query(q_idx[b, t], w[b, t], c.index_comp_kv[b], pos0 + t,
                                     c.base, c.index_rot, c.dtype, k,
                                     bool(c.qat & QAT_FP4_INDEX))
    return out


def _window_rows(c: OracleCache, b: int, p: int, pos0: int, ring, chunk_rows):
    pos = window_positions(p, c.cap_raw)
    rows = []
    for t in pos:
        if chunk_rows is not None and t >= pos0:
            rows.append(chunk_rows[b, t - pos0])
        else:
            rows.append(ring[b, t % c.cap_raw])
    return np.asarray(rows)


def attention(c: OracleCache, pos0: int, q, topk=None, scale=None, ring=None,
              chunk_rows=None, queries=None) -> np.ndarray:
    """Attention outputs [B, T, H, D] for queries at pos0 .. pos0+T-1.

    ring: the raw ring as it was before the chunk (defaults to the cache's);
    chunk_rows: the chunk's rotated raw rows (prefill) or None (decode)."""
    q = np.asarray(q, np.float64)
    B, T, H, D = q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    ring = c.raw_kv if ring is None else ring
    out = np.zeros((B, T, H, D))
    todo = queries if queries is not None else [(b, t) for b in range(B) for t in range(T)]
    for b, t in todo:
        p = pos0 + t
        win = _window_rows(c, b, p, pos0, ring, chunk_rows)
        ids = comp_row_ids(c.ratio, p, c.n_comp, None if topk is None else topk[b, t])
        comp = c.attn_comp_kv[b, ids] if len(ids) else np.zeros((0, D))
        out[b, t] = attention_query(q[b, t], p, win, comp, c.base, c.n_rot, scale, c.dtype)
    return out


def decode_step(c: OracleCache, p: int, inp, top_k: int, scale=None):
    """Append token p, select (ratio 4) and attend. Returns (out [B,H,D], topk [B,k] | None)."""
    compress_append(c, p, inp, chunk=False)
    tk = None
    if c.ratio == 4:
        tk = index_topk(c, p, inp["q_idx"], inp["w"], top_k)
    o = attention(c, p, inp["q"], tk, scale)
    return o[:, 0], (None if tk is None else tk[:, 0])


def prefill_chunk(c: OracleCache, pos0: int, inp, top_k: int, scale=None):
    """Prefill tokens pos0 .. pos0+T-1. Returns (out [B,T,H,D], topk [B,T,k] | None)."""
    ring = c.raw_kv.copy()
    rows = compress_append(c, pos0, inp, chunk=True)
    tk = None
    if c.ratio == 4:
        tk = index_topk(c, pos0, inp["q_idx"], inp["w"], top_k)
    o = attention(c, pos0, inp["q"], tk, scale, ring=ring, chunk_rows=rows)
    commit_ring(c, pos0, rows)
    return o, tk
