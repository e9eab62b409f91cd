"""bench.py's roofline.traffic: the committed ncu capture's DRAM bytes per PCG
iteration are reported, scaled to a launch, only for the kernel sources and
the workload the capture was taken on."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _record():
    with open(os.path.join(ROOT, "profiles", bench.TRAFFIC_FILE)) as f:
        return json.load(f)


def test_committed_capture_is_consistent():
    rec = _record()
    assert rec["dram_bytes_per_iteration"] == (
        rec["dram_bytes_read_per_launch"] + rec["dram_bytes_write_per_launch"]
    ) / rec["iterations_in_launch"]


def test_traffic_is_scaled_for_the_captured_workload_only(monkeypatch):
    rec = _record()
    per_it = rec["dram_bytes_per_iteration"]
    # as if the kernel sources were the captured ones
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: rec["source_digest"])
    config, contacts = bench.TRAFFIC_WORKLOAD
    assert bench.traffic_per_launch(config, contacts, 500.0) == per_it * 500.0
    assert bench.traffic_per_launch("C4", contacts, 500.0) is None
    assert bench.traffic_per_launch(config, "found", 500.0) is None


def test_traffic_is_dropped_once_the_kernel_sources_change(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "0" * 16)
    config, contacts = bench.TRAFFIC_WORKLOAD
    assert bench.traffic_per_launch(config, contacts, 500.0) is None
