"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Routing tables must match bit for bit; outputs and gradients must meet the
fp32 bar (max-abs <= 1e-5) or the bf16 bar (rel-L2 <= 5e-3, max-abs <= 2e-2)
on O, dQ, dK, dV and dBias, for all five workloads (the largest on sampled
windows plus its full dBias) and for seeded small sweeps and edge cases.
"""
import functools

import numpy as np
import pytest

import oracle
from shifted_window_attention_cyclic_gb300 import workloads
from tests.parity_util import (assert_close, gather_windows, host, problem_of, run_gpu, sample_windows)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

IMPLS = ["simt", "auto"]


@functools.lru_cache(maxsize=2)
def _inputs(name):
    wl = workloads.WORKLOADS[name]
    return wl, workloads.generate(wl)


def _check_lse(got, ref, dtype):
    got = np.asarray(got, np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.all(got[~fin] == -np.inf)
    if not fin.any():  # every query on land
        return
    tol = 1e-5 if dtype == "f32" else 2e-3
    assert np.abs(got[fin] - ref[fin]).max() <= tol


def _full_parity(wl, x, impl):
    pb = problem_of(wl)
    res = run_gpu(wl, x, impl=impl, backward=wl.backward)
    o_ref, lse_ref = oracle.fwd(pb, x["q"], x["k"], x["v"], x["bias"], x["land"])
    assert_close("O", host(res["o"]), o_ref, wl.dtype)
    _check_lse(res["lse"].cpu().numpy(), lse_ref, wl.dtype)
    if wl.backward:
        g = oracle.bwd(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"])
        for key in ("dq", "dk", "dv", "dbias"):
            assert_close(key, host(res[key]), g[key], wl.dtype)
    return res


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_tables_bit_exact(name):
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    wl = workloads.WORKLOADS[name]
    desc = C.make_desc(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.dtype,
                       wl.has_land)
    plan = C.swin_attn_plan(desc)
    got = C.swin_attn_plan_tables(plan)
    # the plan keeps the slot-pair table only for windows of up to 2 048 slots
    assert (got[3] is None) == (int(np.prod(wl.window)) > C.RELIDX_MAX_SLOTS)
    want = oracle.tables(problem_of(wl), with_relidx=got[3] is not None)
    for g, w in zip(got, want):
        assert (g is None and w is None) or (g.dtype == w.dtype and np.array_equal(g, w))


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["tiny_fp32", "grid1deg", "ragged", "eddy_ocean"])
def test_workload_full_parity(name, impl):
    wl, x = _inputs(name)
    _full_parity(wl, x, impl)


@pytest.mark.parametrize("impl", IMPLS)
def test_depth3d_sampled_parity_and_full_dbias(impl):
    wl, x = _inputs("depth3d")
    pb = problem_of(wl)
    res = run_gpu(wl, x, impl=impl)
    win_src = oracle.tables(pb)[0]
    ids = sample_windows(pb, 48, seed=5)
    o_ref, lse_ref = oracle.fwd_windows(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], win_ids=ids)
    N, Cc = pb.tokens, pb.channels
    o_got = gather_windows(pb, host(res["o"]).reshape(pb.batch, N, Cc), win_src, ids)
    assert_close("O", o_got, o_ref, wl.dtype)
    lse_got = gather_windows(pb, res["lse"].cpu().numpy().reshape(pb.batch, pb.heads, N).transpose(0, 2, 1),
                             win_src, ids)
    valid = np.stack([win_src[i % pb.nwin] >= 0 for i in ids])
    _check_lse(lse_got[valid], np.transpose(lse_ref, (0, 2, 1))[valid], wl.dtype)
    g = oracle.bwd_windows(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"], win_ids=ids,
                           want=("dq", "dk", "dv"))
    for key in ("dq", "dk", "dv"):
        got = gather_windows(pb, host(res[key]).reshape(pb.batch, N, Cc), win_src, ids)
        assert_close(key, got, g[key], wl.dtype)
    gb = oracle.bwd_windows(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"], want=("dbias",))
    assert_close("dbias", host(res["dbias"]), gb["dbias"], wl.dtype)
    # every token written once: no NaN anywhere, land rows exactly zero
    o_all = host(res["o"])
    assert np.isfinite(o_all).all()
    land = x["land"].astype(bool)
    assert np.all(o_all[land] == 0.0) and np.all(host(res["dq"])[land] == 0.0)
    assert np.all(host(res["dk"])[land] == 0.0) and np.all(host(res["dv"])[land] == 0.0)


SWEEP = [
    # grid, window, shift, periodic, heads, hd, batch, dtype, land
    ((13, 27), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16", (0.3, 0.3)),
    ((17, 19), (5, 6), (2, 3), (1, 1), 3, 16, 2, "bf16", None),
    ((9, 40), (3, 12), (1, 6), (0, 1), 2, 32, 1, "f32", (0.4, 0.4)),
    ((4, 9, 21), (2, 4, 8), (1, 2, 4), (0, 0, 1), 2, 32, 1, "bf16", (0.2, 0.5)),
    ((3, 10, 13), (2, 3, 5), (1, 1, 2), (0, 1, 1), 1, 16, 2, "f32", (0.3, 0.6)),
    ((8, 16), (8, 16), (0, 0), (0, 1), 2, 32, 1, "bf16", None),          # one window = global attention
    ((8, 128), (1, 128), (0, 64), (0, 1), 2, 32, 1, "bf16", None),       # n = 128 along lon only
    ((16, 24), (4, 6), (0, 0), (0, 1), 4, 32, 3, "bf16", (0.3, 0.3)),    # W-MSA, batch 3
    ((7, 7), (8, 8), (0, 0), (0, 0), 2, 32, 1, "bf16", None),            # window larger than grid
    ((11, 11), (8, 8), (4, 4), (0, 0), 2, 16, 1, "f32", None),           # ragged, both dims masked
    # tensor-core path corners: n = 15 < 16 (one key group, no second half),
    # gathered windows whose last row quad is partly past n, batch 2
    ((10, 23), (3, 5), (1, 2), (0, 1), 2, 32, 2, "bf16", (0.3, 0.3)),
    ((9, 30), (3, 7), (2, 3), (1, 1), 3, 32, 1, "bf16", (0.2, 0.2)),     # n = 21
    # w2 = 4 with an odd lon shift: box rows not 4-token aligned (scalar land/LSE loads)
    ((4, 12, 20), (2, 4, 4), (1, 2, 1), (0, 0, 1), 2, 32, 1, "bf16", (0.3, 0.5)),
    # two windows per tensor-core item: 9 windows (the last item holds one),
    # a 3-D case, and n = 60 (second window from tile row 64, 124 rows used)
    ((11, 21), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16", (0.3, 0.3)),
    ((3, 10, 13), (2, 4, 4), (1, 2, 2), (0, 0, 1), 2, 32, 2, "bf16", (0.3, 0.5)),
    ((13, 31), (6, 10), (3, 5), (0, 1), 2, 32, 1, "bf16", (0.3, 0.3)),
    # the largest bias table a 128-token window can have: 7 x 7 x 15 = 735
    # offsets, ragged in all three dimensions; three heads over the CTAs
    ((6, 9, 17), (4, 4, 8), (2, 2, 4), (0, 0, 1), 3, 32, 1, "bf16", (0.3, 0.5)),
    # periodic along depth and lon, ragged in all three dims, unequal shifts;
    # n = 32, so two windows per tensor-core item
    ((5, 6, 11), (2, 4, 4), (1, 2, 3), (1, 0, 1), 2, 32, 1, "bf16", (0.2, 0.4)),
]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("case", SWEEP)
def test_small_sweep(case, impl):
    grid, window, shift, periodic, heads, hd, batch, dtype, land_p = case
    wl = workloads.custom(grid, window, shift, periodic, heads, hd, batch, dtype, land_p,
                          seed_index=300 + SWEEP.index(case))
    _full_parity(wl, workloads.generate(wl), impl)


@pytest.mark.parametrize("grid, window, windows, per_item",
                         [((11, 21), (4, 8), 9, 2), ((13, 31), (6, 10), 12, 2), ((11, 21), (8, 9), 6, 1)])
def test_two_windows_per_item_when_they_fit(grid, window, windows, per_item):
    # the tensor-core plan puts two windows in one 128-row tile when the
    # second can start on a 16-row boundary (round16(n) + n <= 128)
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    attn = SwinWindowAttention(grid, window, (window[0] // 2, window[1] // 2), (0, 1), 2, 32, 1, "bf16")
    info = attn.info
    assert info.impl == 2 and info.windows_per_image == windows
    assert info.work_items == 2 * -(-windows // per_item)


def test_all_land_image_gives_zero_output():
    wl = workloads.custom((9, 16), (3, 8), (1, 4), (0, 1), 2, 32, 1, "bf16", (1.01, 1.01), seed_index=77)
    x = workloads.generate(wl)
    assert x["land"].all()
    res = run_gpu(wl, x)
    assert np.all(host(res["o"]) == 0.0)
    assert np.all(np.isneginf(res["lse"].cpu().numpy()))
    for key in ("dq", "dk", "dv", "dbias"):
        assert np.all(host(res[key]) == 0.0)


def test_dbias_deterministic():
    wl, x = _inputs("ragged")
    a = run_gpu(wl, x)
    b = run_gpu(wl, x)
    for key in ("o", "dq", "dk", "dv", "dbias"):
        assert torch.equal(a[key], b[key]), key


def test_abi_errors_launch_nothing():
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    attn = SwinWindowAttention((16, 32), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16", True)
    dev = torch.device("cuda", 0)
    shape = attn.shape
    q = torch.randn(shape, device=dev).to(torch.bfloat16)
    land = torch.zeros(shape[:-1], dtype=torch.uint8, device=dev)
    o = torch.full(shape, 7.0, device=dev).to(torch.bfloat16)
    lib = C.load_library()
    vp = lambda t: None if t is None else __import__("ctypes").c_void_p(t.data_ptr())
    stream = C._stream(None)
    # land missing while the plan expects it
    assert lib.swin_attn_fwd(attn.plan.handle, vp(q), vp(q), vp(q), None, None, vp(o), None, stream) \
        == C.SWIN_ERR_INVALID_ARG
    # misaligned q
    flat = torch.zeros(q.numel() + 8, dtype=torch.bfloat16, device=dev)
    mis = __import__("ctypes").c_void_p(flat.data_ptr() + 2)
    assert lib.swin_attn_fwd(attn.plan.handle, mis, vp(q), vp(q), None, vp(land), vp(o), None, stream) \
        == C.SWIN_ERR_ALIGNMENT
    # lse off its 16-byte boundary, land off its 4-byte boundary: the kernels
    # read four slots of either with one load
    lse = torch.zeros(attn.lse_shape, device=dev)
    lse_buf = torch.zeros(lse.numel() + 8, device=dev)
    land_buf = torch.zeros(land.numel() + 8, dtype=torch.uint8, device=dev)
    lse_mis = __import__("ctypes").c_void_p(lse_buf.data_ptr() + 4)
    land_mis = __import__("ctypes").c_void_p(land_buf.data_ptr() + 1)
    assert lib.swin_attn_fwd(attn.plan.handle, vp(q), vp(q), vp(q), None, vp(land), vp(o), lse_mis, stream) \
        == C.SWIN_ERR_ALIGNMENT
    assert lib.swin_attn_fwd(attn.plan.handle, vp(q), vp(q), vp(q), None, land_mis, vp(o), vp(lse), stream) \
        == C.SWIN_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert torch.all(o == 7.0)
    assert torch.all(lse == 0.0) and torch.all(lse_buf == 0.0)
    # backward: lse required, workspace checked when dbias is wanted
    dbias = attn.new_bias()
    args = [vp(q)] * 4
    need0 = C.swin_attn_workspace_bytes(attn.plan)
    ws0 = torch.empty(need0, dtype=torch.uint8, device=dev)
    assert lib.swin_attn_bwd(attn.plan.handle, *args, lse_mis, None, vp(land), vp(o), vp(o), vp(o), vp(dbias),
                             vp(ws0), need0, stream) == C.SWIN_ERR_ALIGNMENT
    assert lib.swin_attn_bwd(attn.plan.handle, *args, vp(lse), None, land_mis, vp(o), vp(o), vp(o), vp(dbias),
                             vp(ws0), need0, stream) == C.SWIN_ERR_ALIGNMENT
    assert lib.swin_attn_bwd(attn.plan.handle, *args, None, None, vp(land), vp(o), vp(o), vp(o), None, None, 0,
                             stream) == C.SWIN_ERR_INVALID_ARG
    need = C.swin_attn_workspace_bytes(attn.plan)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    assert lib.swin_attn_bwd(attn.plan.handle, *args, vp(lse), None, vp(land), vp(o), vp(o), vp(o), vp(dbias),
                             vp(ws), need - 256, stream) == C.SWIN_ERR_WORKSPACE
    assert lib.swin_attn_bwd(attn.plan.handle, *args, vp(lse), None, vp(land), vp(o), vp(o), vp(o), vp(dbias),
                             None, need, stream) == C.SWIN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(o == 7.0)
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK


def test_autograd_function_matches_direct_calls():
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention, swin_window_attention
    wl = workloads.custom((13, 27), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16", (0.3, 0.3), seed_index=55)
    x = workloads.generate(wl)
    res = run_gpu(wl, x)
    attn = res["attn"]
    dev = torch.device("cuda", 0)
    q, k, v = (torch.from_numpy(x[n]).to(dev).to(torch.bfloat16).requires_grad_() for n in ("q", "k", "v"))
    bias = torch.from_numpy(x["bias"]).to(dev).requires_grad_()
    land = torch.from_numpy(x["land"]).to(dev)
    o = swin_window_attention(attn, q, k, v, bias, land)
    o.backward(torch.from_numpy(x["dout"]).to(dev).to(torch.bfloat16))
    assert torch.equal(o, res["o"])
    for t, key in ((q, "dq"), (k, "dk"), (v, "dv"), (bias, "dbias")):
        assert torch.equal(t.grad, res[key]), key
