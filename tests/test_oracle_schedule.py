"""Pins of oracle.schedule against figures the pages print (tests/golden)."""
import os

from oracle import schedule

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def page_figures():
    out = {}
    for line in open(os.path.join(GOLD, "page_figures.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            out[k] = float(v) if "." in v else int(v)
    return out


def test_schedule_matches_page_table():
    """Every layer 0..60 of both variants against the printed table."""
    rules = []
    for line in open(os.path.join(GOLD, "schedule.txt")):
        line = line.split("#")[0].strip()
        if line:
            rules.append(line.split())
    assert len(rules) == 6
    for variant_name, layers, ratio in rules:
        variant = schedule.FLASH if variant_name == "flash" else schedule.PRO
        if layers == "0-1":
            ils = [0, 1]
        elif layers == "even>=2":
            ils = list(range(2, 61, 2))
        else:
            ils = list(range(3, 61, 2))
        for il in ils:
            assert schedule.layer_compress_ratio(variant, il) == int(ratio), (variant_name, il)


def test_flash_43_layer_counts():
    """The 43-layer Flash stack: 2 uncompressed, 21 c4a, 20 c128a."""
    r = [schedule.layer_compress_ratio(schedule.FLASH, il) for il in range(43)]
    assert (r.count(0), r.count(4), r.count(128)) == (2, 21, 20)
    r = [schedule.layer_compress_ratio(schedule.PRO, il) for il in range(61)]
    assert (r.count(0), r.count(4), r.count(128)) == (0, 30, 31)


def test_raw_capacity_and_chunk_cap():
    f = page_figures()
    assert schedule.raw_capacity(10**6) == f["n_swa"] == f["swa_window"]
    assert schedule.raw_capacity(57) == 57
    assert schedule.prefill_chunk_cap(f["prefill_chunk"] + 1) == f["prefill_chunk"]
    assert schedule.prefill_chunk_cap(f["prefill_chunk"]) == 0


def test_row_counts_page_and_chunk_boundaries():
    f = page_figures()
    assert schedule.n_comp_rows(4, 1_000_000) == f["c4a_rows_per_1m"]
    # the 4096-token chunk that starts at 28,672 and ends at 32,768
    assert schedule.n_comp_rows(4, 28672) == 7168 and schedule.n_comp_rows(4, 32768) == 8192
    assert schedule.n_comp_rows(128, 28672) == 224 and schedule.n_comp_rows(128, 32768) == 256
    assert schedule.n_comp_rows(0, 32768) == 0


def test_kv_bytes_per_million_tokens():
    """vLLM's 9.62 GiB per 1M-token bf16 sequence for the 61-layer Pro stack
    (head dim 512, indexer dim 128); no other combination of the schedule's
    terms lands on it (dropping the indexer rows or the raw window moves it)."""
    f = page_figures()
    ctx = 1 << 20
    b = schedule.stack_kv_bytes(schedule.PRO, 61, 512, 128, ctx, 1, 2)
    assert round(b / 2**30, 2) == f["kv_gib_per_1m_bf16"]
    no_index = schedule.stack_kv_bytes(schedule.PRO, 61, 512, 0, ctx, 1, 2)
    assert round(no_index / 2**30, 2) != f["kv_gib_per_1m_bf16"]
    flash = schedule.stack_kv_bytes(schedule.FLASH, 43, 512, 128, ctx, 1, 2)
    assert round(flash / 2**30, 2) == 6.72
    # one c4a layer: 262,144 rows x (512 + 128) x 2 B = 320 MiB plus the window
    assert schedule.kv_cache_bytes(4, 512, 128, ctx, 1, 2) == 320 * 2**20 + 128 * 512 * 2
