"""Thin Python binding of libds4a.so (ctypes): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; PyTorch only
provides device memory and streams. There is no CPU path: if the compiled
library is missing, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Dict, Optional

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libds4a.so")

DS4A_F32, DS4A_BF16 = 0, 1
CALL_APPEND, CALL_INDEX_TOPK, CALL_ATTN_DECODE, CALL_ATTN_PREFILL = 0, 1, 2, 3
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported or inconsistent shape",
          -3: "capacity exceeded", -4: "position does not match the cache",
          -5: "unknown dtype", -6: "CUDA error", -7: "device wait timed out",
          -8: "workspace too small"}


class Ds4aError(RuntimeError):
    def __init__(self, status: int, call: str):
        msg = f"{call}: {STATUS.get(status, status)} ({status})"
        if status == -6 and _lib is not None:
            msg += ": " + _lib.ds4a_last_error().decode()
        super().__init__(msg)
        self.status = status


class LayerCacheC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in
                ("ratio", "head_dim", "n_rot", "index_dim", "index_rot", "batch", "cap_raw",
                 "comp_cap")] + [
        ("dtype", ctypes.c_int32), ("n_tokens", ctypes.c_uint32),
        ("raw_kv", ctypes.c_void_p), ("attn_comp_kv", ctypes.c_void_p),
        ("attn_state_kv", ctypes.c_void_p), ("attn_state_score", ctypes.c_void_p),
        ("index_comp_kv", ctypes.c_void_p), ("index_state_kv", ctypes.c_void_p),
        ("index_state_score", ctypes.c_void_p), ("index_norm", ctypes.c_void_p),
        ("index_norm_max", ctypes.c_void_p), ("rope_cos", ctypes.c_void_p),
        ("rope_sin", ctypes.c_void_p), ("index_rope_cos", ctypes.c_void_p),
        ("index_rope_sin", ctypes.c_void_p), ("rope_max_pos", ctypes.c_uint32),
        ("qat", ctypes.c_uint32), ("block_table", ctypes.c_void_p),
        ("max_blocks", ctypes.c_uint32), ("n_blocks", ctypes.c_uint32),
        ("seq_pos", ctypes.c_void_p)]

QAT_FP8_ATTN = 1    # DS4A_QAT_FP8_ATTN
QAT_FP4_INDEX = 2   # DS4A_QAT_FP4_INDEX


EXPORTS = {
    "ds4a_cache_reset": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "ds4a_index_norms": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "ds4a_compress_append": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32]
                             + [ctypes.c_void_p] * 11),
    "ds4a_compress_append_lanes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32,
                                                  ctypes.c_uint32, ctypes.c_uint32]
                                   + [ctypes.c_void_p] * 11),
    "ds4a_index_topk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32,
                                       ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_size_t, ctypes.c_void_p]),
    "ds4a_sparse_attn_decode": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32,
                                               ctypes.c_void_p, ctypes.c_uint32,
                                               ctypes.c_void_p, ctypes.c_uint32, ctypes.c_float,
                                               ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_size_t, ctypes.c_void_p]),
    "ds4a_sparse_attn_prefill_chunk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32,
                                                      ctypes.c_uint32, ctypes.c_void_p,
                                                      ctypes.c_uint32, ctypes.c_void_p,
                                                      ctypes.c_void_p, ctypes.c_uint32,
                                                      ctypes.c_float, ctypes.c_void_p,
                                                      ctypes.c_void_p, ctypes.c_size_t,
                                                      ctypes.c_void_p]),
    "ds4a_index_topk_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32,
                                               ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]),
    "ds4a_noalloc_status": (ctypes.c_int, [ctypes.c_void_p]),
    "ds4a_workspace_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "ds4a_workspace_clear_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t,
                                                   ctypes.c_void_p]),
    "ds4a_wait_selftest": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32,
                                          ctypes.c_void_p]),
    "ds4a_set_decode_cluster": (ctypes.c_int, [ctypes.c_uint32]),
    "ds4a_decode_cluster_size": (ctypes.c_uint32, [ctypes.c_void_p, ctypes.c_uint32,
                                                   ctypes.c_uint32]),
    "ds4a_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_void_p, ctypes.c_uint32,
                                               ctypes.c_uint32, ctypes.c_uint32]),
    "ds4a_rope_table": (ctypes.c_int, [ctypes.c_double, ctypes.c_uint32, ctypes.c_uint32,
                                       ctypes.c_void_p, ctypes.c_void_p]),
    "ds4a_cache_bytes": (ctypes.c_uint64, [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                           ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]),
    "ds4a_layer_compress_ratio": (ctypes.c_uint32, [ctypes.c_int, ctypes.c_uint32]),
    "ds4a_prefill_chunk_cap": (ctypes.c_uint32, [ctypes.c_uint32]),
    "ds4a_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ds4a_launch_count": (ctypes.c_uint64, []),
    "ds4a_last_error": (ctypes.c_char_p, []),
}

_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libds4a.so and declare its signatures. Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m compressed_kv_sparse_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    assert t.is_contiguous(), "tensors passed to the library must be contiguous"
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(status: int, call: str):
    if status != 0:
        raise Ds4aError(status, call)


_tables: Dict[tuple, tuple] = {}


def rope_table(base: float, n_rot: int, n_pos: int, device) -> tuple:
    """Device cos / sin tables [n_pos][n_rot/2] built by ds4a_rope_table."""
    key = (float(base), int(n_rot), int(n_pos), str(device))
    if key not in _tables:
        lib = load()
        c = torch.empty((n_pos, n_rot // 2), dtype=torch.float32)
        s = torch.empty((n_pos, n_rot // 2), dtype=torch.float32)
        _check(lib.ds4a_rope_table(base, n_rot, n_pos, c.data_ptr(), s.data_ptr()),
               "ds4a_rope_table")
        _tables[key] = (c.to(device), s.to(device))
    return _tables[key]


class LayerCache:
    """Device memory of one layer's cache (torch tensors) and its C struct.

    block_table ([B][max_blocks] int32 on the device) makes the compressed rows
    paged: pools of n_blocks blocks of 256 token positions (256 / ratio rows);
    comp_cap is then max_blocks * 256 / ratio. ``logical(name)`` gathers a
    pool back into the contiguous [B][comp_cap][...] view."""

    def __init__(self, *, ratio: int, head_dim: int, n_rot: int, batch: int, comp_cap: int,
                 dtype: str, base: float, rope_max_pos: int, index_dim: int = 0,
                 index_rot: int = 0, cap_raw: int = 128, qat: int = 0, device="cuda",
                 block_table: Optional[torch.Tensor] = None, n_blocks: int = 0):
        td = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
        self.dtype, self.torch_dtype = dtype, td
        self.ratio, self.head_dim, self.n_rot = ratio, head_dim, n_rot
        self.index_dim, self.index_rot, self.batch = index_dim, index_rot, batch
        self.cap_raw, self.comp_cap, self.base = cap_raw, comp_cap, base
        W = {0: 0, 4: 8, 128: 128}[ratio]
        z = lambda *s, dt=td: torch.zeros(s, dtype=dt, device=device)
        self.block_table, self.n_blocks = block_table, n_blocks
        paged = block_table is not None
        if paged:
            assert block_table.dtype == torch.int32 and block_table.shape[0] == batch
            assert comp_cap == block_table.shape[1] * (256 // ratio)
        rpb = 256 // ratio if ratio else 0
        # comp rows: [B][comp_cap][w] or a pool [n_blocks][rows per block][w]
        rows = (lambda w, r, dt=td: z(n_blocks, r, w, dt=dt)) if paged else \
               (lambda w, r, dt=td: z(batch, comp_cap, w, dt=dt))
        self.raw_kv = z(batch, cap_raw, head_dim)
        self.attn_comp_kv = self.attn_state_kv = self.attn_state_score = None
        self.index_comp_kv = self.index_state_kv = self.index_state_score = None
        self.index_norm = self.index_norm_max = None
        if ratio:
            self.attn_comp_kv = rows(head_dim, rpb)
            self.attn_state_kv = z(batch, W, head_dim, dt=torch.float32)
            self.attn_state_score = torch.full((batch, W, head_dim), float("-inf"),
                                               device=device)
        if ratio == 4:
            self.index_comp_kv = rows(index_dim, 64)
            self.index_state_kv = z(batch, 8, index_dim, dt=torch.float32)
            self.index_state_score = torch.full((batch, 8, index_dim), float("-inf"),
                                                device=device)
            self.index_norm = (z(n_blocks, 64, dt=torch.float32) if paged
                               else z(batch, comp_cap, dt=torch.float32))
            self.index_norm_max = z(batch, dt=torch.int32)
        self.rope_cos, self.rope_sin = rope_table(base, n_rot, rope_max_pos, device)
        self.index_rope_cos = self.index_rope_sin = None
        if ratio == 4:
            self.index_rope_cos, self.index_rope_sin = rope_table(base, index_rot,
                                                                  rope_max_pos, device)
        self.c = LayerCacheC(
            ratio=ratio, head_dim=head_dim, n_rot=n_rot, index_dim=index_dim,
            index_rot=index_rot, batch=batch, cap_raw=cap_raw, comp_cap=comp_cap,
            dtype=DS4A_BF16 if dtype == "bf16" else DS4A_F32, n_tokens=0,
            raw_kv=_ptr(self.raw_kv), attn_comp_kv=_ptr(self.attn_comp_kv),
            attn_state_kv=_ptr(self.attn_state_kv), attn_state_score=_ptr(self.attn_state_score),
            index_comp_kv=_ptr(self.index_comp_kv), index_state_kv=_ptr(self.index_state_kv),
            index_state_score=_ptr(self.index_state_score), index_norm=_ptr(self.index_norm),
            index_norm_max=_ptr(self.index_norm_max), rope_cos=_ptr(self.rope_cos),
            rope_sin=_ptr(self.rope_sin), index_rope_cos=_ptr(self.index_rope_cos),
            index_rope_sin=_ptr(self.index_rope_sin), rope_max_pos=rope_max_pos, qat=qat,
            block_table=_ptr(block_table), max_blocks=block_table.shape[1] if paged else 0,
            n_blocks=n_blocks if paged else 0)

    def set_seq_pos(self, seq_pos: Optional[torch.Tensor]):
        """Ragged decode: [B] uint32/int32 device positions of this step's
        tokens (None: every sequence at the call's position). The tensor must
        stay alive while calls use it."""
        self.seq_pos = seq_pos
        self.c.seq_pos = _ptr(seq_pos)

    def logical(self, name: str) -> torch.Tensor:
        """[B][comp_cap][...] view of compressed rows / row norms (a gather
        through the block table when paged)."""
        t = getattr(self, name)
        if self.block_table is None or name not in ("attn_comp_kv", "index_comp_kv",
                                                     "index_norm"):
            return t
        tb = self.block_table.long()                       # [B][max_blocks]
        g = t[tb.clamp(0, self.n_blocks - 1)]              # [B][max_blocks][rpb](...)
        return g.reshape((self.batch, self.comp_cap) + tuple(t.shape[2:]))

    @property
    def n_tokens(self) -> int:
        return self.c.n_tokens

    @n_tokens.setter
    def n_tokens(self, v: int):
        self.c.n_tokens = v

    def ref(self):
        return ctypes.byref(self.c)

    def load_state(self, hist: Dict[str, torch.Tensor], n_tokens: int):
        """Copy a cache snapshot (same layout as the tensors here) in, set
        n_tokens and rebuild the indexer row norms (ds4a_index_norms)."""
        for name, t in hist.items():
            dst = getattr(self, name)
            if self.block_table is not None and name in ("attn_comp_kv", "index_comp_kv"):
                rpb, nb = dst.shape[1], (t.shape[1] + dst.shape[1] - 1) // dst.shape[1]
                src = torch.zeros((self.batch, nb * rpb) + tuple(t.shape[2:]), dtype=t.dtype,
                                  device=t.device)
                src[:, :t.shape[1]] = t
                idx = self.block_table[:, :nb].reshape(-1).long().to(dst.device)
                dst[idx] = src.reshape((self.batch * nb, rpb) + tuple(t.shape[2:])).to(dst.device)
            elif name in ("attn_comp_kv", "index_comp_kv") and t.shape[1] < dst.shape[1]:
                dst[:, :t.shape[1]].copy_(t)
            else:
                dst.copy_(t)
        self.n_tokens = n_tokens
        if self.ratio == 4:
            ds4a_index_norms(self)

    def snapshot(self) -> Dict[str, torch.Tensor]:
        names = ["raw_kv", "attn_comp_kv", "attn_state_kv", "attn_state_score",
                 "index_comp_kv", "index_state_kv", "index_state_score"]
        return {n: getattr(self, n).clone() for n in names if getattr(self, n) is not None}

    def workspace_bytes(self, call: int, T: int, n_heads: int, top_k: int) -> int:
        return load().ds4a_workspace_bytes(call, self.ref(), T, n_heads, top_k)


def ds4a_cache_reset(cache: LayerCache, stream=None):
    _check(load().ds4a_cache_reset(cache.ref(), _stream(stream)), "ds4a_cache_reset")


def ds4a_index_norms(cache: LayerCache, stream=None):
    _check(load().ds4a_index_norms(cache.ref(), _stream(stream)), "ds4a_index_norms")


def ds4a_compress_append(cache: LayerCache, pos0: int, T: int, inp: Dict[str, torch.Tensor],
                         raw_chunk_out: Optional[torch.Tensor] = None, stream=None):
    g = inp.get
    _check(load().ds4a_compress_append(
        cache.ref(), pos0, T, _ptr(g("raw_kv_in")), _ptr(g("attn_cand")), _ptr(g("attn_score")),
        _ptr(g("ape_attn")), _ptr(g("gamma_attn")), _ptr(g("idx_cand")), _ptr(g("idx_score")),
        _ptr(g("ape_idx")), _ptr(g("gamma_idx")), _ptr(raw_chunk_out), _stream(stream)),
        "ds4a_compress_append")


LANE_RAW, LANE_ATTN, LANE_INDEX = 1, 2, 4   # DS4A_LANE_*


def ds4a_compress_append_lanes(cache: LayerCache, pos0: int, T: int, lanes: int,
                               inp: Dict[str, torch.Tensor],
                               raw_chunk_out: Optional[torch.Tensor] = None, stream=None):
    """The parts `lanes` of an append; n_tokens is left for the caller to set."""
    g = inp.get
    _check(load().ds4a_compress_append_lanes(
        cache.ref(), pos0, T, lanes, _ptr(g("raw_kv_in")), _ptr(g("attn_cand")),
        _ptr(g("attn_score")), _ptr(g("ape_attn")), _ptr(g("gamma_attn")), _ptr(g("idx_cand")),
        _ptr(g("idx_score")), _ptr(g("ape_idx")), _ptr(g("gamma_idx")), _ptr(raw_chunk_out),
        _stream(stream)), "ds4a_compress_append_lanes")


def ds4a_index_topk(cache: LayerCache, pos0: int, T: int, q_idx: torch.Tensor, w: torch.Tensor,
                    n_heads: int, top_k: int, topk: torch.Tensor, ws: torch.Tensor, stream=None):
    _check(load().ds4a_index_topk(cache.ref(), pos0, T, _ptr(q_idx), _ptr(w), n_heads, top_k,
                                  _ptr(topk), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "ds4a_index_topk")


STATIC_SCRATCH_BYTES = 8 << 20


def ds4a_index_topk_noalloc(cache: LayerCache, pos0: int, T: int, q_idx: torch.Tensor,
                            w: torch.Tensor, n_heads: int, top_k: int, topk: torch.Tensor,
                            stream=None):
    """ds4a_index_topk with the library's static scratch instead of a workspace."""
    _check(load().ds4a_index_topk_noalloc(cache.ref(), pos0, T, _ptr(q_idx), _ptr(w), n_heads,
                                          top_k, _ptr(topk), _stream(stream)),
           "ds4a_index_topk_noalloc")


def ds4a_sparse_attn_decode(cache: LayerCache, pos: int, q: torch.Tensor, n_heads: int,
                            topk: Optional[torch.Tensor], top_k: int, scale: float,
                            out: torch.Tensor, ws: Optional[torch.Tensor], stream=None):
    nb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().ds4a_sparse_attn_decode(cache.ref(), pos, _ptr(q), n_heads, _ptr(topk), top_k,
                                          scale, _ptr(out), _ptr(ws), nb, _stream(stream)),
           "ds4a_sparse_attn_decode")


def ds4a_sparse_attn_prefill_chunk(cache: LayerCache, pos0: int, T: int, q: torch.Tensor,
                                   n_heads: int, raw_chunk: torch.Tensor,
                                   topk: Optional[torch.Tensor], top_k: int, scale: float,
                                   out: torch.Tensor, ws: Optional[torch.Tensor], stream=None):
    nb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().ds4a_sparse_attn_prefill_chunk(cache.ref(), pos0, T, _ptr(q), n_heads,
                                                 _ptr(raw_chunk), _ptr(topk), top_k, scale,
                                                 _ptr(out), _ptr(ws), nb, _stream(stream)),
           "ds4a_sparse_attn_prefill_chunk")


def ds4a_cache_bytes(ratio, head_dim, index_dim, ctx, batch, elem_bytes) -> int:
    return load().ds4a_cache_bytes(ratio, head_dim, index_dim, ctx, batch, elem_bytes)


def ds4a_layer_compress_ratio(variant: int, il: int) -> int:
    return load().ds4a_layer_compress_ratio(variant, il)


def ds4a_prefill_chunk_cap(prompt_len: int) -> int:
    return load().ds4a_prefill_chunk_cap(prompt_len)


def ds4a_launch_count() -> int:
    return load().ds4a_launch_count()


def workspace(nbytes: int, device="cuda") -> Optional[torch.Tensor]:
    """A workspace buffer (uint8) of at least nbytes, 256-byte aligned by torch.
    Its first 256 bytes are zeroed, so its wait status starts clear."""
    if nbytes == 0:
        return None
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
    ws[:min(nbytes, 256)].zero_()
    return ws


def _nbytes(ws: Optional[torch.Tensor]) -> int:
    return 0 if ws is None else ws.numel() * ws.element_size()


def ds4a_workspace_status(ws: torch.Tensor) -> int:
    """Timed-out device waits recorded in a workspace's error word (0: none).
    Synchronises nothing itself: call after the calls' stream is synchronised.
    Returns the count; the status (DS4A_OK / DS4A_ERR_TIMEOUT) follows from it."""
    n = ctypes.c_uint32(0)
    st = load().ds4a_workspace_status(_ptr(ws), _nbytes(ws), ctypes.byref(n))
    if st not in (0, -7):
        _check(st, "ds4a_workspace_status")
    assert (st == -7) == (n.value != 0)
    return n.value


def ds4a_workspace_clear_status(ws: torch.Tensor, stream=None):
    _check(load().ds4a_workspace_clear_status(_ptr(ws), _nbytes(ws), _stream(stream)),
           "ds4a_workspace_clear_status")


def ds4a_noalloc_status() -> int:
    """ds4a_workspace_status of the no-allocation variant's static scratch."""
    n = ctypes.c_uint32(0)
    st = load().ds4a_noalloc_status(ctypes.byref(n))
    if st not in (0, -7):
        _check(st, "ds4a_noalloc_status")
    return n.value


def ds4a_wait_selftest(ws: torch.Tensor, limit_us: int, stream=None):
    _check(load().ds4a_wait_selftest(_ptr(ws), _nbytes(ws), limit_us, _stream(stream)),
           "ds4a_wait_selftest")


def ds4a_set_decode_cluster(C: int):
    _check(load().ds4a_set_decode_cluster(C), "ds4a_set_decode_cluster")


def ds4a_decode_cluster_size(cache: "LayerCache", n_heads: int, top_k: int) -> int:
    return load().ds4a_decode_cluster_size(cache.ref(), n_heads, top_k)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
