"""bench.py's measurement plumbing without a GPU: the ncu DRAM record
(parsing, per-call division, kernel-name forms, staleness by source hash)
and the step-8 layer flags."""
import json

import pytest

import bench


def _csv(rows):
    head = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"'
    return head + "\n" + "\n".join(
        f'"{i}","{k}","{m}","{u}","{v}"' for i, (k, m, u, v) in enumerate(rows)) + "\n"


def test_write_traffic_sums_a_calls_kernels_per_call(tmp_path, monkeypatch):
    """Read and write bytes of every kernel of a call kind add up; both forms
    ncu prints for the anonymous namespace match; the sum is divided by the
    number of calls; a record for other sources is replaced."""
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"sources_sha256": "other", "entries": {"x": {}}}))
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(path))
    rows = [
        ("void ds4a::(anonymous namespace)::index_qbf_kernel(IndexArgs)", "dram__bytes_read.sum",
         "Kbyte", "1,000"),
        ("void ds4a::<unnamed>::index_score_tc_kernel<1>(CUtensorMap)", "dram__bytes_read.sum",
         "Mbyte", "60"),
        ("void ds4a::<unnamed>::index_score_tc_kernel<1>(CUtensorMap)", "dram__bytes_write.sum",
         "Mbyte", "2"),
        ("void ds4a::<unnamed>::topk_select_tc_kernel<1024>(IndexArgs)", "dram__bytes_read.sum",
         "Mbyte", "4"),
        ("void ds4a::<unnamed>::attn_tc_kernel<1, 0>(CUtensorMap)", "dram__bytes_read.sum",
         "Mbyte", "10"),
        ("void ds4a::<unnamed>::append_step_kernel<bf16>(AppendArgs)", "dram__bytes_write.sum",
         "byte", "512"),
        ("void other_library_kernel()", "dram__bytes_read.sum", "Gbyte", "9"),
    ]
    csv = tmp_path / "t.csv"
    csv.write_text("==PROF== noise line\n" + _csv(rows))
    bench.write_traffic(str(csv), "flash_c4a_layer", "flash_c4a_layer_b8_ctx131072", calls=2)
    rec = json.loads(path.read_text())
    assert rec["sources_sha256"] == bench.sources_hash() and "x" not in rec["entries"]
    ent = rec["entries"][bench.WORKLOADS["flash_c4a_layer"].name]
    assert ent["index_topk"]["bytes_per_call"] == pytest.approx((1e6 + 60e6 + 2e6 + 4e6) / 2)
    assert ent["attn"]["bytes_per_call"] == pytest.approx(10e6 / 2)
    assert ent["append"]["bytes_per_call"] == pytest.approx(256)
    name = bench.WORKLOADS["flash_c4a_layer"].name
    assert bench.recorded_traffic(name, "index_topk") == pytest.approx(33.5e6)
    assert bench.recorded_traffic(name, "attn_r4") == pytest.approx(5e6)   # attention kinds share
    assert bench.recorded_traffic(name, "missing") is None


def test_recorded_traffic_is_null_for_other_sources(tmp_path, monkeypatch):
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"sources_sha256": "0" * 64, "entries": {
        "w": {"index_topk": {"bytes_per_call": 1.0}}}}))
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(path))
    assert bench.recorded_traffic("w", "index_topk") is None


def test_qat_flags_by_layer_kind():
    from compressed_kv_sparse_gb300 import lib
    assert bench.qat_flags(0) == 0
    assert bench.qat_flags(128) == lib.QAT_FP8_ATTN
    assert bench.qat_flags(4) == lib.QAT_FP8_ATTN | lib.QAT_FP4_INDEX


def test_clock_summary_median_max_and_reasons():
    s = bench.ClockSampler(0)
    s.lines = ["2070, 2070, 900.5, Not Active, Not Active, Not Active, Not Active",
               "1980, 2070, 1200.0, Not Active, Not Active, Not Active, Active",
               "2070, 2070, 1300.0, Not Active, Not Active, Not Active, Not Active",
               "[N/A], garbage"]
    out = s.summary()
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}
    s.lines = []
    assert s.summary()["reasons"] == ["unsampled"]


def test_reference_arm_line_keeps_the_contract():
    """The reference arm (the oracle on host cores) prints the contract's keys
    with its own e2e figure and no host-device bytes."""
    line = bench.reference_arm(bench.WORKLOADS["tiny"], 1, 0, 1)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in line, k
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == bench.WORKLOADS["tiny"].name
    ex = line["extrapolation"]         # the step time is scaled from a timed sample
    assert ex["factor"] == pytest.approx(line["ms_per_step"] / ex["timed_ms_per_step"])


def test_oracle_sample_plan_scales_to_a_whole_step():
    """The CPU oracle's sample and its scale factors: on many cores every
    sequence of a layer of each kind runs in parallel and the layers of a
    kind scale it; on one core one (layer, sequence) per kind scales by
    layers x sequences; a prefill chunk samples queries evenly."""
    wl = bench.WORKLOADS["flash43"]
    units, phases, _ = bench.oracle_plan(wl, 16)
    f = dict(phases)
    assert f[("dec", 0)] == 1.0 and f[("dec", 4)] == 10.5 and f[("dec", 128)] == 10.0
    assert sum(1 for u in units if u[:2] == ("dec", 4)) == 16      # 2 layers x 8 sequences
    units, phases, _ = bench.oracle_plan(wl, 1)
    f = dict(phases)
    assert f[("dec", 0)] == 16 and f[("dec", 4)] == 168 and f[("dec", 128)] == 160
    assert len(units) == 3
    wl = bench.WORKLOADS["prefill"]
    units, phases, _ = bench.oracle_plan(wl, 4)
    qs = sorted(t for u in units if u[0] == "qry" for t in u[1])
    assert len(qs) == 16 and qs[0] == 0 and qs[-1] == wl.chunk - 1
    assert dict(phases)[("qry",)] == wl.chunk / 16
