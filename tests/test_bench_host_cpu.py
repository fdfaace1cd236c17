"""Host-side logic of bench.py that needs no GPU."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_committed_traffic_matches_current_sources():
    # the committed ncu traffic belongs to the kernel sources in the tree
    khash = bench.kernel_source_hash()
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    if t["kernel_source_hash"] != khash:
        pytest.skip("kernel sources changed since the committed ncu capture")
    assert bench.profiled_traffic(khash, t["workload"], t["kernels"]) == t["bwd_dram_bytes_per_launch"]


def test_traffic_only_for_its_workload_kernels_and_sources(tmp_path):
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"kernel_source_hash": "abc", "workload": "depth3d", "kernels": "tcgen05",
                                "bwd_dram_bytes_per_launch": 123}))
    assert bench.profiled_traffic("abc", "depth3d", "tcgen05", str(path)) == 123
    assert bench.profiled_traffic("abd", "depth3d", "tcgen05", str(path)) is None
    assert bench.profiled_traffic("abc", "ragged", "tcgen05", str(path)) is None
    assert bench.profiled_traffic("abc", "depth3d", "simt", str(path)) is None
    assert bench.profiled_traffic("abc", "depth3d", "tcgen05", str(tmp_path / "missing.json")) is None
