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
