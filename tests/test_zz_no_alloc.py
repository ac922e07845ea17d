"""ds4a_index_topk_noalloc: the indexer top-k for callers that cannot
allocate device memory (a C host without an allocator, a runtime that owns
all device memory, a loop that cannot afford cudaMalloc's synchronisation).
It uses the library's static scratch array instead of a workspace; its top-k
lists must equal those of ds4a_index_topk on the same inputs, call after call
(the shared scratch keeps the previous call's contents)."""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, shape, B, p):
    from compressed_kv_sparse_gb300 import lib
    wl = synth.Workload("noalloc", seed, B, (shape,), p, "decode")
    cap = (p + 1) // 4 + 1
    hist = synth.cache_history(wl, 0, p + 1, comp_cap=cap, device=DEV)
    c = lib.LayerCache(ratio=4, head_dim=shape.head_dim, n_rot=shape.n_rot, batch=B,
                       comp_cap=cap, dtype=shape.dtype, base=shape.rope_base, rope_max_pos=p + 2,
                       index_dim=shape.index_dim, index_rot=shape.index_rot, device=DEV)
    c.load_state(hist, p + 1)
    q_idx = synth.normal((B, 1, shape.index_heads, shape.index_dim), seed, "q",
                         dtype=shape.dtype, device=DEV)
    w = synth.normal((B, 1, shape.index_heads), seed, "w", dtype=shape.dtype, device=DEV)
    return c, q_idx, w


@pytest.mark.parametrize("shape,B,p", [
    (synth.LayerShape(ratio=4), 4, 65536),                 # Flash shape, tensor-core path
    (synth.TINY.layers[0], 2, 2000),                        # fp32 tiny shape, exact path
])
def test_noalloc_matches_workspace_entry_point(shape, B, p):
    from compressed_kv_sparse_gb300 import lib
    k = shape.top_k
    for call in range(2):
        c, q_idx, w = _case(50 + call, shape, B, p)
        ref = torch.full((B, k), -7, dtype=torch.int32, device=DEV)
        got = torch.full((B, k), -9, dtype=torch.int32, device=DEV)
        ws = lib.workspace(c.workspace_bytes(lib.CALL_INDEX_TOPK, 1, shape.index_heads, k))
        lib.ds4a_index_topk(c, p, 1, q_idx, w, shape.index_heads, k, ref, ws)
        lib.ds4a_index_topk_noalloc(c, p, 1, q_idx, w, shape.index_heads, k, got)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), ref.cpu().numpy()), f"call {call}"
        assert lib.ds4a_noalloc_status() == 0      # no device wait gave up


def test_noalloc_rejects_requests_beyond_the_scratch():
    """A 4096-query chunk needs far more than the static scratch: the call
    must refuse before launching anything and leave the output untouched."""
    from compressed_kv_sparse_gb300 import lib
    shape = synth.LayerShape(ratio=4)
    c, _, _ = _case(60, shape, 1, 32767)
    T = 4096
    need = c.workspace_bytes(lib.CALL_INDEX_TOPK, T, shape.index_heads, shape.top_k)
    assert need > lib.STATIC_SCRATCH_BYTES
    q_idx = torch.zeros((1, T, 64, 128), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((1, T, 64), dtype=torch.bfloat16, device=DEV)
    out = torch.full((1, T, shape.top_k), -3, dtype=torch.int32, device=DEV)
    st = lib.load().ds4a_index_topk_noalloc(c.ref(), 32768 - T, T, q_idx.data_ptr(),
                                            w.data_ptr(), 64, shape.top_k, out.data_ptr(), None)
    torch.cuda.synchronize()
    assert st == -8
    assert bool((out == -3).all())
