"""Shared plumbing of the parity tests: build the same layer state on the GPU
(through the library) and in the oracle, and compare."""
import numpy as np
import torch

import synth

TOL = {"f32": 1e-5, "bf16": 1e-2}   # relative L2 bound on continuous outputs


def np_(t):
    return t.detach().float().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


def rel_l2(got, want):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def gpu_cache(shape: synth.LayerShape, batch: int, comp_cap: int, rope_max_pos: int,
              hist=None, n_tokens: int = 0, device="cuda", qat: int = 0):
    from compressed_kv_sparse_gb300 import lib
    c = lib.LayerCache(ratio=shape.ratio, head_dim=shape.head_dim, n_rot=shape.n_rot,
                       batch=batch, comp_cap=comp_cap, dtype=shape.dtype, base=shape.rope_base,
                       rope_max_pos=rope_max_pos, index_dim=shape.index_dim,
                       index_rot=shape.index_rot, cap_raw=shape.cap_raw, qat=qat, device=device)
    if hist is not None:
        c.load_state({k: v.to(device) for k, v in hist.items()}, n_tokens)
    return c


def oracle_cache(shape: synth.LayerShape, hist, n_tokens: int, qat: int = 0,
                 keep_pre: bool = False):
    from oracle.layer import OracleCache
    return OracleCache(ratio=shape.ratio, head_dim=shape.head_dim, n_rot=shape.n_rot,
                       cap_raw=shape.cap_raw, base=shape.rope_base, dtype=shape.dtype,
                       n_tokens=n_tokens, index_dim=shape.index_dim, index_rot=shape.index_rot,
                       qat=qat, keep_pre=keep_pre, **{k: np_(v) for k, v in hist.items()})


def to_dev(inp, device="cuda"):
    return {k: v.to(device).contiguous() for k, v in inp.items()}


def to_np(inp):
    return {k: np_(v) for k, v in inp.items()}
