"""Host logic of bench.py that needs no GPU: the committed ncu traffic record
is used only while the kernel source it was taken on is unchanged, scales to
the launch size when it is a ratio, and the bench line's config names the
workload with the keys both arms share."""
import hashlib
import json
import os

import pytest

import bench
import synth


def _fake_root(tmp_path, record, source_text):
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "kernel.cu"
    src.write_text(source_text)
    rec = dict(record, source="kernel.cu")
    rec.setdefault("source_sha256", hashlib.sha256(source_text.encode()).hexdigest())
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"k": rec}))
    return src


def test_traffic_per_launch_while_the_source_matches(tmp_path, monkeypatch):
    _fake_root(tmp_path, {"dram_bytes_per_launch": 1234}, "kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("k") == 1234
    assert bench.ncu_traffic("other") is None


def test_traffic_ratio_scales_to_the_launch(tmp_path, monkeypatch):
    _fake_root(tmp_path, {"dram_bytes_per_algorithmic_byte": 1.5}, "kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("k", 1000.0) == pytest.approx(1500.0)
    assert bench.ncu_traffic("k") is None  # a ratio needs the launch's bytes


def test_traffic_is_null_once_the_source_changes(tmp_path, monkeypatch):
    src = _fake_root(tmp_path, {"dram_bytes_per_launch": 1234}, "kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src.write_text("kernel v2\n")
    assert bench.ncu_traffic("k") is None


def test_committed_traffic_records_name_existing_sources():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    assert "expert_ffn" in recs
    for name, rec in recs.items():
        assert os.path.exists(os.path.join(bench.ROOT, rec["source"])), name
        assert len(rec["source_sha256"]) == 64, name
        assert ("dram_bytes_per_launch" in rec) != ("dram_bytes_per_algorithmic_byte" in rec), name


def test_measured_peaks_fall_back_without_the_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.measured_peaks()
    assert src == "fallback" and peaks["hbm_gbs"] > 0 and peaks["bf16_tflops"] > 0


def test_config_names_the_workload_and_shapes():
    wl = synth.WORKLOADS["decode_2816"]
    c = bench.workload_config(wl, 30, 16, 1)
    assert c["workload"] == "decode_2816" and c["layers"] == 30 and c["cache_slots"] == 16
    assert (c["d_model"], c["experts"], c["top_k"], c["d_ff"], c["d_ff_shared"]) == (2816, 256, 8, 704, 2816)
    assert c["policy"] == "LFU" and c["parallelism"] == "single GPU"
    assert "model" not in c
    assert bench.workload_config(wl, 30, 256, 2, resident=True)["parallelism"] == "replicas"
