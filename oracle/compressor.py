"""KV compressor: per-token state store, softmax pooling at ratio boundaries,
RMSNorm, tail RoPE, append; plus the raw sliding-window insert.

Follows "【#3】ds4.c を読み解く":
* §2 the per-layer cache (raw_kv ring of cap_raw rows, attn_comp_kv with the
  attn_state_kv / attn_state_score recurrent state, and index_comp_kv with the
  index state on ratio-4 layers);
* §4 the per-token compressor steps: candidate (wkv) and score (wgate) come in
  projected; APE bias; store in the recurrent state; at a ratio boundary pool
  with per-channel softmax weights exp(score - max) (denominator 0 gives 0);
  RMS normalisation; tail-only RoPE; step 8, the FP8 (attention lane) or
  FP4 QAT (indexer lane) round trip, when the cache enables it (``qat.py``);
* §5 ratio 4 keeps an 8-row frontier: token p is written to row 4 + p % 4, at
  (p + 1) % 4 == 0 the 8 rows are pooled into one row and rows 4..7 move to
  rows 0..3. With vLLM's page (c4a: one compressed token is a weighted sum of
  8 raw tokens at stride 4; c128a: 128 tokens at stride 128).

Readings:
* R1 row i of a ratio-4 layer pools tokens 4i-4 .. 4i+3 (slot s <-> token
  4i-4+s); row i of a ratio-128 layer pools tokens 128i .. 128i+127 (slot =
  p mod 128). n_comp = floor(n_tokens / ratio).
* R2 slots of tokens before position 0 are empty (score -inf, weight 0).
* R3 the state keeps scores without APE; APE row = slot within the window
  (0 = oldest) is added when pooling. Each lane (attention, indexer) has its
  own width (D, Di) and its own APE [W, width].
* R5 RMSNorm: y = gamma * c / sqrt(mean(c^2) + 1e-6).
* R8 compressed row i is rotated at position i * ratio with the layer's base;
  raw rows at their own position.
"""
import numpy as np

from .numerics import round_store
from .qat import attn_row_round_trip, index_row_round_trip
from .rope import rope_tail

RMS_EPS = 1e-6


def window_slot(ratio: int, p: int) -> int:
    """State row that token p is stored in."""
    return 4 + p % 4 if ratio == 4 else p % ratio


def softmax_pool(state_kv, state_score, ape) -> np.ndarray:
    """Per-channel softmax-weighted pool over the window slots (axis -2).

    sigma = score + APE; m = max over slots; w = exp(sigma - m);
    out = sum(w * kv) / sum(w), or 0 where the sum of weights is 0."""
    sigma = np.asarray(state_score, np.float64) + np.asarray(ape, np.float64)
    m = np.max(sigma, axis=-2, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(sigma - m)                    # exp(-inf) = 0 for empty slots
    kv = np.where(w > 0, np.asarray(state_kv, np.float64), 0.0)
    den = np.sum(w, axis=-2)
    num = np.sum(w * kv, axis=-2)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)


def rms_norm(c, gamma, eps: float = RMS_EPS) -> np.ndarray:
    c = np.asarray(c, np.float64)
    rms = np.sqrt(np.mean(c * c, axis=-1, keepdims=True) + eps)
    return np.asarray(gamma, np.float64) * (c / rms)


class Lane:
    """One compressor lane's recurrent state and output rows (numpy views)."""

    def __init__(self, state_kv, state_score, comp, ape, gamma, n_rot, quant=None, pre=None):
        self.state_kv = state_kv          # [B, W, width] float32
        self.state_score = state_score    # [B, W, width] float32, pre-APE
        self.comp = comp                  # [B, cap, width] float64 (storage-exact)
        self.ape = ape                    # [W, width]
        self.gamma = gamma                # [width]
        self.n_rot = n_rot
        self.quant = quant                # None, "fp8" (attention) or "fp4" (indexer)
        self.pre = pre                    # optional [B, cap, width]: rows before step 8


def lane_step(lane: Lane, ratio: int, p: int, cand, score, base: float, dtype: str):
    """Compressor step for token p on one lane (cand / score: [B, width])."""
    slot = window_slot(ratio, p)
    lane.state_kv[:, slot] = cand
    lane.state_score[:, slot] = score
    if (p + 1) % ratio != 0:
        return
    i = (p + 1) // ratio - 1
    pooled = softmax_pool(lane.state_kv, lane.state_score, lane.ape)
    row = rope_tail(rms_norm(pooled, lane.gamma), i * ratio, base, lane.n_rot)
    if lane.pre is not None:
        lane.pre[:, i] = row
    if lane.quant == "fp8":
        row = attn_row_round_trip(row, lane.n_rot)
    elif lane.quant == "fp4":
        row = index_row_round_trip(row)
    lane.comp[:, i] = round_store(row, dtype)
    if ratio == 4:
        lane.state_kv[:, 0:4] = lane.state_kv[:, 4:8]
        lane.state_score[:, 0:4] = lane.state_score[:, 4:8]


def raw_rows(raw_kv_in, pos0: int, base: float, n_rot: int, dtype: str) -> np.ndarray:
    """Rotated raw rows of tokens pos0 .. pos0+T-1 ([B, T, D] in, storage-exact out)."""
    T = raw_kv_in.shape[1]
    pos = (pos0 + np.arange(T))[None, :]
    return round_store(rope_tail(raw_kv_in, pos, base, n_rot), dtype)
