"""Seeded synthetic inputs for the compressed-KV attention layer.

This module is shared by the tests, ``bench.py`` and the smoke check. It only
draws numbers and lays them out; it holds none of the method's arithmetic
(no pooling, normalisation, rotation, scoring or attention). Both the CUDA path
and the CPU oracle receive exactly the tensors produced here.

Recipe (stated once, used everywhere):
  * every tensor gets its own seed, derived from the workload seed and the
    tensor's name, layer and role by a stable hash (``subseed``);
  * values are drawn with ``torch.Generator`` as N(0, 1) in fp32 and, for bf16
    workloads, rounded to bf16 (round to nearest even, ``Tensor.to``);
  * projected per-token inputs (raw KV, compressor candidates and scores,
    queries, indexer queries and head weights) are drawn directly as N(0, 1):
    with hidden states x ~ N(0, 1) and weights W ~ N(0, 1/fan_in) each projected
    element is N(0, 1), so drawing them directly has the same distribution.
    The tiny fp32 workload projects real hidden states instead;
  * APE biases are N(0, 0.02^2); norm gains are 1 + 0.02 N(0, 1);
  * long histories (tens of thousands of tokens) are synthesised at cache level:
    compressed rows, indexer rows and raw-window rows are N(0, 1) (a normalised
    row has unit RMS, and the rotation keeps norms), and the compressor's
    recurrent state holds N(0, 1) candidates/scores for the tokens that are
    still pending, with score -inf marking an empty slot.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Dict, Optional

import torch

NEG_INF = float("-inf")


def subseed(seed: int, *keys) -> int:
    """Stable 63-bit seed for one tensor, from the workload seed and its keys."""
    h = hashlib.blake2b(repr((seed,) + tuple(keys)).encode(), digest_size=8)
    return int.from_bytes(h.digest(), "little") & ((1 << 63) - 1)


def normal(shape, seed: int, *keys, std: float = 1.0, mean: float = 0.0,
           dtype: str = "f32", device="cpu") -> torch.Tensor:
    """N(mean, std^2) draw, fp32 then rounded to ``dtype`` ('f32' or 'bf16')."""
    g = torch.Generator(device=device)
    g.manual_seed(subseed(seed, *keys))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch_dtype(dtype))


def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Shape of one attention layer of the compressed-KV family."""
    ratio: int            # 0 (raw window only), 4 (c4a) or 128 (c128a)
    head_dim: int = 512   # D, shared K = V head dimension
    n_rot: int = 64       # rotated tail dims
    n_heads: int = 64     # H query heads
    index_dim: int = 128  # Di (ratio 4 only)
    index_heads: int = 64 # Hi (ratio 4 only)
    top_k: int = 512
    cap_raw: int = 128    # raw sliding window
    base: float = 10000.0
    compress_base: float = 160000.0
    dtype: str = "bf16"

    @property
    def window(self) -> int:
        return {0: 0, 4: 8, 128: 128}[self.ratio]

    @property
    def index_rot(self) -> int:
        return min(64, self.index_dim)

    @property
    def rope_base(self) -> float:
        return self.compress_base if self.ratio != 0 else self.base

    def replace(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    batch: int
    layers: tuple          # tuple of LayerShape, one per layer
    context: int           # tokens already in the cache
    mode: str              # "decode" or "prefill"
    chunk: int = 1         # tokens processed by the step
    hidden: int = 0        # >0: project real hidden states (tiny workload only)

    @property
    def dtype(self) -> str:
        return self.layers[0].dtype


def flash_ratio(il: int) -> int:
    """Layer ratio of the 43-layer Flash stack (layout only; used to build shapes)."""
    if il < 2:
        return 0
    return 4 if il % 2 == 0 else 128


TINY = Workload(
    name="c4a_tiny_f32_b1_p256", seed=0, batch=1,
    layers=(LayerShape(ratio=4, head_dim=128, n_rot=64, n_heads=4, index_dim=32,
                       index_heads=2, top_k=16, dtype="f32"),),
    context=256, mode="decode", hidden=256)
C128A_DECODE = Workload(
    name="c128a_decode_b1_ctx65536", seed=1, batch=1,
    layers=(LayerShape(ratio=128),), context=65536, mode="decode")
C4A_DECODE = Workload(
    name="c4a_decode_b32_ctx65536", seed=2, batch=32,
    layers=(LayerShape(ratio=4),), context=65536, mode="decode")
C4A_PREFILL = Workload(
    name="c4a_prefill_b1_t4096_p28672", seed=3, batch=1,
    layers=(LayerShape(ratio=4),), context=28672, mode="prefill", chunk=4096)
FLASH_STACK = Workload(
    name="flash43_decode_b8_ctx131072", seed=4, batch=8,
    layers=tuple(LayerShape(ratio=flash_ratio(il)) for il in range(43)),
    context=131072, mode="decode")

# One c4a layer of the Flash stack alone (same shape, batch and context): a
# measurement case for counters that cannot be captured on the whole stack.
FLASH_C4A_LAYER = Workload(
    name="flash_c4a_layer_b8_ctx131072", seed=4, batch=8,
    layers=(LayerShape(ratio=4),), context=131072, mode="decode")

WORKLOADS = {w.name: w for w in (TINY, C128A_DECODE, C4A_DECODE, C4A_PREFILL, FLASH_STACK,
                                 FLASH_C4A_LAYER)}


def comp_capacity(shape: LayerShape, n_tokens: int) -> int:
    """Row capacity that holds every compressed row of ``n_tokens`` tokens."""
    if shape.ratio == 0:
        return 0
    return max(1, n_tokens // shape.ratio)


# --------------------------------------------------------------------------
# per-token projected inputs

def step_inputs(wl: Workload, layer: int, pos0: int, T: int, device="cpu",
                step: int = 0) -> Dict[str, torch.Tensor]:
    """Projected inputs and weights of one layer for tokens pos0 .. pos0+T-1.

    Keys: raw_kv_in [B,T,D], attn_cand/attn_score [B,T,D], q [B,T,H,D], and for
    ratio 4 idx_cand/idx_score [B,T,Di], q_idx [B,T,Hi,Di], w [B,T,Hi];
    weights ape_attn [W,D], gamma_attn [D], ape_idx [8,Di], gamma_idx [Di].
    """
    s = wl.layers[layer]
    B, D, dt, sd = wl.batch, s.head_dim, s.dtype, wl.seed
    key = ("step", layer, pos0, T, step)
    out: Dict[str, torch.Tensor] = {}
    if wl.hidden:
        return _projected_inputs(wl, layer, pos0, T, device)
    out["raw_kv_in"] = normal((B, T, D), sd, *key, "raw", dtype=dt, device=device)
    out["q"] = normal((B, T, s.n_heads, D), sd, *key, "q", dtype=dt, device=device)
    if s.ratio:
        out["attn_cand"] = normal((B, T, D), sd, *key, "acand", dtype=dt, device=device)
        out["attn_score"] = normal((B, T, D), sd, *key, "ascore", dtype=dt, device=device)
    if s.ratio == 4:
        Di, Hi = s.index_dim, s.index_heads
        out["idx_cand"] = normal((B, T, Di), sd, *key, "icand", dtype=dt, device=device)
        out["idx_score"] = normal((B, T, Di), sd, *key, "iscore", dtype=dt, device=device)
        out["q_idx"] = normal((B, T, Hi, Di), sd, *key, "qidx", dtype=dt, device=device)
        out["w"] = normal((B, T, Hi), sd, *key, "w", dtype=dt, device=device)
    out.update(layer_weights(wl, layer, device))
    return out


def layer_weights(wl: Workload, layer: int, device="cpu") -> Dict[str, torch.Tensor]:
    s = wl.layers[layer]
    dt, sd = s.dtype, wl.seed
    out = {}
    if s.ratio:
        out["ape_attn"] = normal((s.window, s.head_dim), sd, "ape_attn", layer, std=0.02,
                                 dtype=dt, device=device)
        out["gamma_attn"] = normal((s.head_dim,), sd, "gamma_attn", layer, std=0.02, mean=1.0,
                                   dtype=dt, device=device)
    if s.ratio == 4:
        out["ape_idx"] = normal((8, s.index_dim), sd, "ape_idx", layer, std=0.02,
                                dtype=dt, device=device)
        out["gamma_idx"] = normal((s.index_dim,), sd, "gamma_idx", layer, std=0.02, mean=1.0,
                                  dtype=dt, device=device)
    return out


def _projected_inputs(wl: Workload, layer: int, pos0: int, T: int, device):
    """Tiny workload: project N(0,1) hidden states with N(0, 1/fan_in) weights."""
    s = wl.layers[layer]
    B, Hd, D, dt, sd = wl.batch, wl.hidden, s.head_dim, s.dtype, wl.seed
    x = normal((B, T, Hd), sd, "hidden", layer, pos0, T, device=device).double()

    def proj(name, n_out):
        W = normal((Hd, n_out), sd, "W", name, layer, std=1.0 / math.sqrt(Hd),
                   device=device).double()
        return (x @ W).to(torch_dtype(dt))

    out = {"raw_kv_in": proj("kv", D),
           "q": proj("q", s.n_heads * D).reshape(B, T, s.n_heads, D)}
    if s.ratio:
        out["attn_cand"] = proj("wkv", D)
        out["attn_score"] = proj("wgate", D)
    if s.ratio == 4:
        Di, Hi = s.index_dim, s.index_heads
        out["idx_cand"] = proj("idx_wkv", Di)
        out["idx_score"] = proj("idx_wgate", Di)
        out["q_idx"] = proj("idx_q", Hi * Di).reshape(B, T, Hi, Di)
        out["w"] = proj("idx_w", Hi)
    out.update(layer_weights(wl, layer, device))
    return out


# --------------------------------------------------------------------------
# cache-level history

def cache_history(wl: Workload, layer: int, n_tokens: int, comp_cap: Optional[int] = None,
                  device="cpu") -> Dict[str, torch.Tensor]:
    """A cache that has seen ``n_tokens`` tokens, synthesised at cache level.

    Returns raw_kv [B,cap_raw,D] (slot = position mod cap_raw), attn_comp_kv
    [B,comp_cap,D] (rows beyond n_tokens // ratio are zero), attn_state_kv and
    attn_state_score [B,W,D] and, for ratio 4, index_comp_kv [B,comp_cap,Di],
    index_state_kv / index_state_score [B,8,Di].

    State layout (the cache convention of the library): ratio 4 keeps the last
    complete group of 4 tokens in slots 0..3 and the tokens of the current group
    in slots 4 + p % 4; ratio 128 keeps token p in slot p % 128. Scores are
    stored without the APE bias; an empty slot has score -inf and kv 0.
    """
    s = wl.layers[layer]
    B, D, dt, sd = wl.batch, s.head_dim, s.dtype, wl.seed
    r = s.ratio
    key = ("hist", layer, n_tokens)
    out: Dict[str, torch.Tensor] = {}
    out["raw_kv"] = normal((B, s.cap_raw, D), sd, *key, "raw", dtype=dt, device=device)
    if n_tokens < s.cap_raw:
        out["raw_kv"][:, n_tokens:] = 0
    if r == 0:
        return out
    cap = comp_cap if comp_cap is not None else comp_capacity(s, n_tokens)
    n_comp = n_tokens // r

    def rows(n_feat, name):
        t = torch.zeros((B, cap, n_feat), dtype=torch_dtype(dt), device=device)
        if n_comp:
            t[:, :n_comp] = normal((B, n_comp, n_feat), sd, *key, name, dtype=dt, device=device)
        return t

    def state(W, n_feat, name):
        kv = torch.zeros((B, W, n_feat), dtype=torch.float32, device=device)
        sc = torch.full((B, W, n_feat), NEG_INF, dtype=torch.float32, device=device)
        filled = []
        if r == 4:
            cur = n_tokens % 4
            if n_tokens >= 4:
                filled += [0, 1, 2, 3]
            filled += [4 + j for j in range(cur)]
        else:
            filled = list(range(n_tokens % r))
        for slot in filled:
            kv[:, slot] = normal((B, n_feat), sd, *key, name, "kv", slot, dtype=dt,
                                 device=device).float()
            sc[:, slot] = normal((B, n_feat), sd, *key, name, "score", slot, dtype=dt,
                                 device=device).float()
        return kv, sc

    out["attn_comp_kv"] = rows(D, "acomp")
    out["attn_state_kv"], out["attn_state_score"] = state(s.window, D, "astate")
    if r == 4:
        out["index_comp_kv"] = rows(s.index_dim, "icomp")
        out["index_state_kv"], out["index_state_score"] = state(8, s.index_dim, "istate")
    return out


def empty_history(wl: Workload, layer: int, comp_cap: int, device="cpu"):
    """A cache before its first token: zero rows, empty state."""
    s = wl.layers[layer]
    B, D = wl.batch, s.head_dim
    td = torch_dtype(s.dtype)
    out = {"raw_kv": torch.zeros((B, s.cap_raw, D), dtype=td, device=device)}
    if s.ratio == 0:
        return out
    out["attn_comp_kv"] = torch.zeros((B, comp_cap, D), dtype=td, device=device)
    out["attn_state_kv"] = torch.zeros((B, s.window, D), dtype=torch.float32, device=device)
    out["attn_state_score"] = torch.full((B, s.window, D), NEG_INF, dtype=torch.float32,
                                         device=device)
    if s.ratio == 4:
        Di = s.index_dim
        out["index_comp_kv"] = torch.zeros((B, comp_cap, Di), dtype=td, device=device)
        out["index_state_kv"] = torch.zeros((B, 8, Di), dtype=torch.float32, device=device)
        out["index_state_score"] = torch.full((B, 8, Di), NEG_INF, dtype=torch.float32,
                                              device=device)
    return out


def grid_values(shape, seed: int, *keys, lo: int = -8, hi: int = 8, scale: float = 0.125,
                device="cpu", dtype: str = "f32") -> torch.Tensor:
    """Integers in [lo, hi] times ``scale``: every product and short sum is exact,
    so ties are frequent and summation order cannot change a result."""
    g = torch.Generator(device=device)
    g.manual_seed(subseed(seed, *keys))
    x = torch.randint(lo, hi + 1, shape, generator=g, device=device).float() * scale
    return x.to(torch_dtype(dtype))


def random_topk(B: int, T: int, k: int, vis: int, seed: int, *keys, device="cpu"):
    """Random ascending index lists (distinct, < vis), -1 padded, for attention tests."""
    g = torch.Generator(device="cpu")
    g.manual_seed(subseed(seed, "topk", *keys))
    out = torch.full((B, T, k), -1, dtype=torch.int32)
    m = min(k, vis)
    for b in range(B):
        for t in range(T):
            if m:
                idx = torch.randperm(vis, generator=g)[:m].sort().values
                out[b, t, :m] = idx.to(torch.int32)
    return out.to(device)
