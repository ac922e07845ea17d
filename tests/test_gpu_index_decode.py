"""The bf16 decode top-k against the oracle, case by case.

Each case must give the oracle's lists exactly ("【#3】ds4.c を読み解く" §6
indexer): Gaussian rows at the Flash shape at 1, 2, 19 and 32 sequences (the
scorer's CTAs split each sequence's rows 152, 76, 8 and 4 ways), 1/8-grid
ties, every row tied (the selection's full pass), subnormal products, the FP4
QAT query, a row appended by the same step, ragged positions (one sequence
with fewer visible rows than k) and paged rows with a shared prefix."""
import numpy as np
import pytest
import torch

import synth
import test_gpu_full
import test_gpu_paged
import test_gpu_parity
import test_gpu_qat
import test_gpu_ragged
from helpers import gpu_cache, np_, oracle_cache, to_dev
from oracle import layer as olayer
from test_gpu_parity import lib_, run_index

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("B", [1, 2, 19, 32])
def test_flash_shape_gaussian(B):
    """16,384 rows per sequence."""
    run_index(lib_(), synth.LayerShape(ratio=4), B, 65536, 1, seed=50 + B,
              queries=[(b, 0) for b in range(0, B, max(1, B // 4))])


def test_grid_ties():
    run_index(lib_(), synth.LayerShape(ratio=4), 2, 4000, 1, seed=51, grid=True)


def test_all_rows_tied():
    test_gpu_full.test_index_tc_all_rows_tied_fallback()


@pytest.mark.parametrize("q_exp,k_exp", [(-70, -60), (-100, -40)])
def test_tiny_magnitudes(q_exp, k_exp):
    test_gpu_parity.test_index_tc_tiny_magnitudes(q_exp, k_exp)


def test_qat_query():
    test_gpu_qat.test_index_qat_query_exact("bf16", 8, 16383, 1)


def test_qat_boundary_step():
    """Append at p = 8191 (a new indexer row from the same step), then the
    top-k and attention against the oracle."""
    test_gpu_qat.test_qat_decode_step_layer()


def test_ragged_positions():
    test_gpu_ragged.test_ragged_decode_matches_oracle_per_sequence(4)


@pytest.mark.parametrize("case", [c for c in test_gpu_paged.CASES
                                  if c[0] == 4 and c[1] == "bf16" and c[4] == 1])
def test_paged(case):
    test_gpu_paged.test_paged_equals_contiguous(*case)


def test_appended_row_at_boundary():
    """Decode at p = 4i + 3: the append of the same step writes row i, which
    the top-k must see (its tile loads only after the append completes)."""
    lib = lib_()
    shape = synth.LayerShape(ratio=4)
    B, p = 3, 4 * 2047 + 3
    wl = synth.Workload("bnd", 52, B, (shape,), p, "decode")
    cap = (p + 1) // 4 + 1
    hist = synth.cache_history(wl, 0, p, comp_cap=cap)
    inp = synth.step_inputs(wl, 0, p, 1)
    gc = gpu_cache(shape, B, cap, p + 2, hist, p)
    lib.ds4a_compress_append(gc, p, 1, to_dev(inp))
    topk = torch.full((B, 1, shape.top_k), -7, dtype=torch.int32, device=DEV)
    ws = lib.workspace(gc.workspace_bytes(lib.CALL_INDEX_TOPK, 1, 64, shape.top_k))
    lib.ds4a_index_topk(gc, p, 1, inp["q_idx"].to(DEV), inp["w"].to(DEV), 64, shape.top_k, topk,
                        ws)
    torch.cuda.synchronize()
    assert lib.ds4a_workspace_status(ws) == 0
    oc = oracle_cache(shape, hist, p)
    olayer.compress_append(oc, p, {k: np_(v) for k, v in inp.items()}, chunk=False)
    i = (p + 1) // 4 - 1
    oc.index_comp_kv[:, i] = np_(gc.index_comp_kv)[:, i]   # the top-k decides on the GPU's row
    ref = olayer.index_topk(oc, p, np_(inp["q_idx"]), np_(inp["w"]), shape.top_k)
    assert np.array_equal(topk.cpu().numpy(), ref)
