"""GPU parity on the 43-layer Flash decode stack (8 sequences at 131,072
tokens), built and stepped by the benchmark's own runner: the same caches,
inputs, positions and launch configuration (cluster sizes) as the timed step.
Sampled layers of each kind (window-only, c4a with its selection over 32,768
rows per sequence, c128a with 1,024 compressed rows) and sampled sequences
are checked against the oracle: top-k lists exactly, outputs within the bf16
bound ("【#3】ds4.c を読み解く" §1 Flash schedule, §7 mixed attention)."""
import numpy as np
import pytest
import torch

import synth
from helpers import TOL, np_, oracle_cache, rel_l2
from oracle import layer as olayer

pytestmark = pytest.mark.gpu
DEV = "cuda"

# layers checked: both window-only layers' kind, the first and last c4a and
# c128a layers
LAYERS = (0, 2, 3, 41, 42)
SEQS = (0, 5, 7)


@pytest.fixture(scope="module")
def flash_runner():
    import bench
    R = bench.Runner(synth.FLASH_STACK, torch.device(DEV))
    R.step()
    torch.cuda.synchronize()
    yield R
    del R
    torch.cuda.empty_cache()


def test_flash_stack_schedule(flash_runner):
    """The runner's stack follows the page's Flash schedule: 2 window-only,
    21 c4a and 20 c128a layers, and each layer's cache has that ratio."""
    from compressed_kv_sparse_gb300 import lib
    R = flash_runner
    ratios = [L["s"].ratio for L in R.layers]
    assert ratios == [lib.ds4a_layer_compress_ratio(0, il) for il in range(43)]
    assert (ratios.count(0), ratios.count(4), ratios.count(128)) == (2, 21, 20)
    assert all(L["cache"].ratio == L["s"].ratio for L in R.layers)


def test_flash_stack_cluster_sizes(flash_runner):
    """The decode attention of the benchmarked step runs on clusters: the c4a
    layers' bound of 128 + 512 rows is 5 tiles and the c128a layers' 128 +
    1,025 rows (their compressed capacity) 10. The sizes chosen are printed, so
    the layer checks below are known to cover them."""
    from compressed_kv_sparse_gb300 import lib
    R = flash_runner
    got = {}
    for L in R.layers:
        s = L["s"]
        got.setdefault(s.ratio, set()).add(lib.ds4a_decode_cluster_size(L["cache"], s.n_heads,
                                                                        s.top_k))
    print("decode cluster sizes by ratio:", got)
    assert len(got[4]) == 1 and len(got[128]) == 1 and got[0] == {1}
    assert 1 < min(got[4]) <= 5 and 1 < min(got[128]) <= 10


@pytest.mark.parametrize("il", LAYERS)
def test_flash_stack_layer_matches_oracle(flash_runner, il):
    R = flash_runner
    wl = R.wl
    L = R.layers[il]
    s = L["s"]
    p = R.p0
    cap = L["cache"].comp_cap
    # the history the runner loaded (the same seeded draw), per sampled sequence
    hist = synth.cache_history(wl, il, p, comp_cap=cap, device=DEV)
    inp = L["inp"]
    out = L["out"]
    for b in SEQS:
        one = {n: t[b:b + 1].cpu() for n, t in hist.items()}
        oc = oracle_cache(s, one, p)
        ninp = {n: (np_(t[b:b + 1]) if t.dim() > 2 else np_(t)) for n, t in inp.items()}
        o_ref, tk_ref = olayer.decode_step(oc, p, ninp, s.top_k)
        if s.ratio == 4:
            assert np.array_equal(L["topk"][b].cpu().numpy(), tk_ref[0]), (il, b)
        e = rel_l2(np_(out[b]), o_ref[0])
        assert e <= TOL["bf16"], (il, b, e)
    del hist
