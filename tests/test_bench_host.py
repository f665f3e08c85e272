"""Host logic of bench.py that decides reported figures (CPU).

The roofline's `traffic` comes from the committed ncu record only while every
source file of the kernel is unchanged since the capture; the record itself
carries each counter's origin.
"""
import json
import os

import bench


def test_traffic_is_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    kernel = "stream_fwd_tc_kernel"
    rec = tmp_path / "traffic.json"
    good = {"source_sha256": bench.source_digest(kernel), "dram_bytes_per_launch": 123}
    rec.write_text(json.dumps({kernel: {"w": good, "stale": dict(good, source_sha256="0" * 64)}}))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(rec))
    assert bench.kernel_traffic(kernel, "w") == 123
    assert bench.kernel_traffic(kernel, "stale") is None
    assert bench.kernel_traffic(kernel, "missing") is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "absent.json"))
    assert bench.kernel_traffic(kernel, "w") is None


def test_digest_covers_every_listed_source():
    for kernel, files in bench.KERNEL_SOURCES.items():
        for rel in files:
            assert os.path.exists(os.path.join(bench.ROOT, rel)), rel
        assert len(bench.source_digest(kernel)) == 64


def test_committed_traffic_record_is_well_formed():
    with open(bench.PROFILE_TRAFFIC) as f:
        table = json.load(f)
    assert set(table) <= set(bench.KERNEL_SOURCES)
    for kernel, per_workload in table.items():
        for workload, ent in per_workload.items():
            assert ent["dram_bytes_per_launch"] == ent["dram_read_bytes"] + ent["dram_write_bytes"]
            assert len(ent["source_sha256"]) == 64
            cmd = ent["command"]
            assert cmd.startswith("ncu ") and "--clock-control none" in cmd, (kernel, workload)
            assert f"--workload {workload}" in cmd or workload == "inbatch_b128_bf16", (kernel, workload)
