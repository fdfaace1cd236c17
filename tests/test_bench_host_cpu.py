"""Host-side logic of bench.py that needs no GPU."""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_committed_traffic_matches_current_sources():
    # the committed ncu traffic belongs to the kernel sources in the tree
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    khash = bench.kernel_source_hash(t["kernels"])
    if t["kernel_source_hash"] != khash:
        pytest.skip("kernel sources changed since the committed ncu capture")
    assert bench.profiled_traffic(khash, t["workload"], t["kernels"]) == t["bwd_dram_bytes_per_launch"]


def test_source_hash_covers_the_kernel_unit_and_its_headers():
    # the tcgen05 hash follows swin_tc.cu's includes (tc_ptx.cuh, swin_common.cuh,
    # the public header) and the launch plans; it differs from the SIMT one
    a, b = bench.kernel_source_hash("tcgen05"), bench.kernel_source_hash("simt")
    assert a != b and len(a) == 16 and a == bench.kernel_source_hash("tcgen05")


def test_traffic_only_for_its_workload_kernels_and_sources(tmp_path):
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"kernel_source_hash": "abc", "workload": "depth3d", "kernels": "tcgen05",
                                "bwd_dram_bytes_per_launch": 123}))
    assert bench.profiled_traffic("abc", "depth3d", "tcgen05", str(path)) == 123
    assert bench.profiled_traffic("abd", "depth3d", "tcgen05", str(path)) is None
    assert bench.profiled_traffic("abc", "ragged", "tcgen05", str(path)) is None
    assert bench.profiled_traffic("abc", "depth3d", "simt", str(path)) is None
    assert bench.profiled_traffic("abc", "depth3d", "tcgen05", str(tmp_path / "missing.json")) is None


def test_parity_sample_reads_the_bar():
    # device results stood in by the oracle's own full outputs, rounded to
    # bf16 as the kernels round them: within the bar; one planted error of
    # 0.05 in dK (over the bf16 max-abs bar of 0.02) is caught
    torch = pytest.importorskip("torch")
    import oracle
    from shifted_window_attention_cyclic_gb300 import workloads
    wl = workloads.custom((13, 27), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16", (0.3, 0.3), seed_index=60)
    x = workloads.generate(wl)
    pb = oracle.Problem(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.has_land)
    o, _ = oracle.fwd(pb, x["q"], x["k"], x["v"], x["bias"], x["land"])
    g = oracle.bwd(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"])
    outs = {"o": torch.from_numpy(o).to(torch.bfloat16)}
    outs.update({k: torch.from_numpy(g[k]).to(torch.bfloat16) for k in ("dq", "dk", "dv")})
    res = bench.parity_sample(wl, x, outs, windows=64)
    assert res["within_bar"], res
    assert all(res[k]["max_abs"] < 2e-2 and res[k]["rel_l2"] < 5e-3 for k in ("o", "dq", "dk", "dv"))
    sea = np.argwhere(~x["land"][0].astype(bool))[0]
    outs["dk"][(0,) + tuple(sea)][3] += 0.05
    res = bench.parity_sample(wl, x, outs, windows=10 ** 6)  # every window
    assert not res["within_bar"] and res["dk"]["max_abs"] > 2e-2


def test_counts_of_a_workload_without_bias():
    # beast_w64k: BEAST's [360, 180] windows, no relative-position bias. Its
    # algorithmic bytes carry no bias table, its FLOPs count every pair of
    # real slots of the 8 full windows, and the bench times it with fewer
    # repetitions
    from shifted_window_attention_cyclic_gb300 import workloads
    wl = workloads.WORKLOADS["beast_w64k"]
    assert not wl.bias and wl.head_dim == 128 and int(np.prod(wl.window)) == 64800
    assert "beast_w64k" in bench.EXTRA and bench.EXTRA_REPS["beast_w64k"][0] <= 10
    n = int(np.prod(wl.window))
    win_src = np.arange(8 * n, dtype=np.int32).reshape(8, n)  # 8 full windows (720 x 720 grid)
    f, b, fb, bb, bm = bench.workload_counts(wl, win_src, None)
    assert f == 4.0 * 8 * n * n * wl.channels and b == 2.5 * f
    N, e = wl.tokens, 2
    assert fb == 4 * N * wl.channels * e + 4 * N * wl.heads  # Q, K, V, O + LSE: no bias, no land
    with_bias = workloads.Workload(**{**wl.__dict__, "bias": True})
    rows = int(np.prod([2 * w - 1 for w in wl.window]))
    assert bench.workload_counts(with_bias, win_src, None)[2] == fb + rows * wl.heads * 4
    # its windows are beyond the per-window oracle legs of the bench
    assert n > bench.ORACLE_WINDOW_SLOTS
