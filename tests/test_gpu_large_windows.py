"""Windows of more than 128 slots with head_dim 128 (the key-tiled tcgen05
kernels) against the oracle, through the C ABI, forward and backward:
TERRA's w = 32 windows (1 024 tokens, 8 key tiles, d/Nh = 128) on a grid
with a periodic seam and land, a ragged 3-D case with partial tiles, a
window of fewer than 128 slots, and a window without a bias whose bias table
would not fit the kernels' column (no dBias there). The backward runs both
ways: delta recomputed as sum_j P dP (swin_attn_bwd) and delta = dout . O
from the forward's output (swin_attn_bwd_o)."""
import numpy as np
import pytest

import oracle
from shifted_window_attention_cyclic_gb300 import workloads
from tests.parity_util import BF16_MAX_ABS, BF16_REL_L2, assert_close, host, problem_of, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = [
    # grid, window, shift, periodic, heads, batch, land, bias
    ((64, 64), (32, 32), (16, 16), (0, 1), 2, 1, (0.3, 0.3), True),         # n = 1024, 8 key tiles
    ((3, 40, 70), (2, 16, 16), (1, 8, 8), (0, 0, 1), 1, 1, (0.2, 0.5), True),  # n = 512, ragged in lat and lon
    ((21, 45), (8, 12), (4, 6), (0, 1), 2, 2, None, True),                    # n = 96: one partial tile
    ((60, 200), (30, 100), (15, 50), (0, 1), 1, 1, None, False),              # n = 3000, no bias (59 x 199 rows)
    ((32, 32), (16, 16), (8, 8), (0, 1), 1, 1, (1.0, 1.0), True),             # n = 256, every token land
]


def _lse_check(got, ref):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    if fin.any():
        assert np.abs(got[fin] - ref[fin]).max() <= 2e-3


@pytest.mark.parametrize("case", CASES)
def test_large_window_forward_matches_the_oracle(case):
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    grid, window, shift, periodic, heads, batch, land_p, with_bias = case
    wl = workloads.custom(grid, window, shift, periodic, heads, 128, batch, "bf16", land_p,
                          seed_index=900 + CASES.index(case))
    x = workloads.generate(wl)
    if not with_bias:
        x["bias"] = np.zeros_like(x["bias"])
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.dtype,
                               wl.has_land)
    assert attn.info.impl == C.SWIN_IMPL_TC
    assert attn.info.work_items == heads * batch * attn.info.windows_per_image * -(-attn.info.slots // 128)
    t = to_device(x, wl, torch.device("cuda", 0))
    o, lse = attn.forward(t["q"], t["k"], t["v"], t["bias"] if with_bias else None, t["land"])
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK
    o_ref, lse_ref = oracle.fwd(problem_of(wl), x["q"], x["k"], x["v"], x["bias"], x["land"])
    assert_close("O", host(o), o_ref, "bf16")
    _lse_check(lse.cpu().numpy().astype(np.float64), lse_ref)
    if x["land"] is not None:
        assert np.all(host(o)[x["land"].astype(bool)] == 0.0)


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("with_o", [False, True], ids=["delta_recomputed", "delta_from_o"])
def test_large_window_backward_matches_the_oracle(case, with_o):
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    grid, window, shift, periodic, heads, batch, land_p, with_bias = case
    wl = workloads.custom(grid, window, shift, periodic, heads, 128, batch, "bf16", land_p,
                          seed_index=900 + CASES.index(case))
    x = workloads.generate(wl)
    if not with_bias:
        x["bias"] = np.zeros_like(x["bias"])
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.dtype,
                               wl.has_land)
    t = to_device(x, wl, torch.device("cuda", 0))
    bias = t["bias"] if with_bias else None
    o, lse = attn.forward(t["q"], t["k"], t["v"], bias, t["land"])
    # with_o: delta = dout . o (o the forward's bf16 output) instead of sum P dP
    dq, dk, dv, dbias = attn.backward(t["q"], t["k"], t["v"], t["dout"], lse, bias, t["land"], want_dbias=with_bias,
                                      o=o if with_o else None)
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK
    g = oracle.bwd(problem_of(wl), x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"])
    for key, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(key, host(got), g[key], "bf16")
    if with_bias and not with_o:
        assert_close("dbias", host(dbias), g["dbias"], "bf16")
    elif with_bias:
        # delta = dout . O carries O's bf16 storage rounding (2^-9 relative per
        # term) into every dS of the query, and dBias adds those dS over every
        # pair of one offset in every window of the head, with one sign: the
        # max-abs bar grows by 2^-8 of the largest |dBias|; relative L2 keeps
        # the bar
        got, ref = host(dbias), g["dbias"]
        rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
        bar = BF16_MAX_ABS + 2.0 ** -8 * np.abs(ref).max()
        assert rel <= BF16_REL_L2 and np.abs(got - ref).max() <= bar, (rel, np.abs(got - ref).max(), bar)
    if x["land"] is not None:
        land = x["land"].astype(bool)
        for got in (dq, dk, dv):
            assert np.all(host(got)[land] == 0.0)
