"""The bounded device waits and their host-visible status.

A wait that runs out must end its kernel, leave the context usable and show
up on the host as DS4A_ERR_TIMEOUT through the workspace's error word. The
self-test kernel waits, with the same bounded-wait code the kernels use, on a
barrier phase that nothing completes (no copy or MMA in flight) under a short
limit; ordinary calls must leave the word at zero."""
import time

import numpy as np
import pytest
import torch

import synth
from helpers import TOL, gpu_cache, np_, oracle_cache, rel_l2, to_dev, to_np
from oracle import layer as olayer

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_wait_that_runs_out_reports_timeout():
    from compressed_kv_sparse_gb300 import lib
    ws = lib.workspace(256)
    assert lib.ds4a_workspace_status(ws) == 0
    t0 = time.perf_counter()
    lib.ds4a_wait_selftest(ws, 2000)          # 2 ms limit
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    n = lib.ds4a_workspace_status(ws)
    assert n >= 1
    assert dt < 1.0, dt                       # it gave up near its limit
    st = lib.load().ds4a_workspace_status(ws.data_ptr(), 256, None)
    assert st == -7                           # DS4A_ERR_TIMEOUT
    # a later launch on the same word: the count keeps growing until cleared
    lib.ds4a_wait_selftest(ws, 500)
    torch.cuda.synchronize()
    assert lib.ds4a_workspace_status(ws) > n
    lib.ds4a_workspace_clear_status(ws)
    torch.cuda.synchronize()
    assert lib.ds4a_workspace_status(ws) == 0


def test_context_usable_after_timeout_and_calls_leave_status_clear():
    """After a timed-out wait the device still runs the path: a tiny decode
    step matches the oracle and its workspaces report no timeout."""
    from compressed_kv_sparse_gb300 import lib
    ws0 = lib.workspace(256)
    lib.ds4a_wait_selftest(ws0, 1000)
    wl = synth.TINY
    s = wl.layers[0]
    p = 200
    cap = (p + 1) // 4 + 1
    hist = synth.cache_history(wl, 0, p, comp_cap=cap)
    inp = synth.step_inputs(wl, 0, p, 1)
    gc = gpu_cache(s, 1, cap, p + 2, hist, p)
    d = to_dev(inp)
    lib.ds4a_compress_append(gc, p, 1, d)
    k = s.top_k
    topk = torch.empty((1, k), dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, 1, s.index_heads, k))
    lib.ds4a_index_topk(gc, p, 1, d["q_idx"], d["w"], s.index_heads, k, topk, ws)
    out = torch.empty((1, s.n_heads, s.head_dim), device=DEV)
    wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_DECODE, 1, s.n_heads, k))
    lib.ds4a_sparse_attn_decode(gc, p, d["q"][:, 0].contiguous(), s.n_heads, topk, k,
                                1 / np.sqrt(s.head_dim), out, wa)
    torch.cuda.synchronize()
    assert lib.ds4a_workspace_status(ws0) >= 1
    assert lib.ds4a_workspace_status(ws) == 0
    if wa is not None:
        assert lib.ds4a_workspace_status(wa) == 0
    oc = oracle_cache(s, hist, p)
    o_ref, tk_ref = olayer.decode_step(oc, p, to_np(inp), k)
    assert np.array_equal(topk.cpu().numpy(), tk_ref)
    assert rel_l2(np_(out), o_ref) <= TOL["f32"]


def test_tensor_core_calls_leave_status_clear():
    """The tensor-core scorer, certified select and cluster attention at the
    Flash shape: their error words stay zero."""
    from compressed_kv_sparse_gb300 import lib
    shape = synth.LayerShape(ratio=4)
    B, p = 4, 20000
    wl = synth.Workload("st", 80, B, (shape,), p, "decode")
    cap = (p + 1) // 4 + 1
    hist = synth.cache_history(wl, 0, p, comp_cap=cap, device=DEV)
    inp = {n: v.contiguous() for n, v in synth.step_inputs(wl, 0, p, 1, device=DEV).items()}
    gc = gpu_cache(shape, B, cap, p + 2, hist, p)
    lib.ds4a_compress_append(gc, p, 1, inp)
    k = shape.top_k
    topk = torch.empty((B, k), dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, 1, 64, k))
    lib.ds4a_index_topk(gc, p, 1, inp["q_idx"], inp["w"], 64, k, topk, ws)
    out = torch.empty((B, 64, 512), dtype=torch.bfloat16, device=DEV)
    wa = lib.workspace(gc.workspace_bytes(lib.CALL_ATTN_DECODE, 1, 64, k))
    for _ in range(3):
        lib.ds4a_sparse_attn_decode(gc, p, inp["q"][:, 0].contiguous(), 64, topk, k,
                                    1 / np.sqrt(512), out, wa)
    torch.cuda.synchronize()
    assert lib.ds4a_workspace_status(ws) == 0
    assert lib.ds4a_workspace_status(wa) == 0
