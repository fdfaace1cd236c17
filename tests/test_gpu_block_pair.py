"""The W-MSA + SW-MSA block pair through the C ABI (two plans, reused): both
layers' outputs and gradients against the oracle called once per layer with
its own shift (0, then floor(w/2) per dim), on a ragged 2-D grid with land
and on a 3-D depth grid; the W-MSA plan's routing has no region bits, and the
two plans agree on every slot pair's bias row."""
import numpy as np
import pytest

import oracle
from shifted_window_attention_cyclic_gb300 import workloads
from tests.parity_util import assert_close, host, problem_of, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = [
    # grid, window, periodic, heads, batch, land
    ((37, 75), (8, 12), (0, 1), 4, 1, (0.3, 0.3)),
    ((5, 21, 43), (2, 8, 8), (0, 0, 1), 2, 1, (0.3, 0.6)),
]


@pytest.mark.parametrize("case", CASES)
def test_block_pair_matches_the_oracle_layer_by_layer(case):
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinBlockPair
    grid, window, periodic, heads, batch, land_p = case
    pair = SwinBlockPair(grid, window, periodic, heads, 32, batch, "bf16", land_p is not None)
    assert pair.shift == tuple(w // 2 for w in window)
    dev = torch.device("cuda", 0)
    layers = []
    for li, shift in enumerate(((0,) * len(grid), pair.shift)):
        wl = workloads.custom(grid, window, shift, periodic, heads, 32, batch, "bf16", land_p, seed_index=810 + li)
        layers.append((wl, workloads.generate(wl)))
    land = layers[0][1]["land"]  # one land mask for both layers (the same grid)
    t = [to_device(x, wl, dev) for wl, x in layers]
    land_d = t[0]["land"]
    first = (t[0]["q"], t[0]["k"], t[0]["v"], t[0]["bias"])
    second = (t[1]["q"], t[1]["k"], t[1]["v"], t[1]["bias"])
    (o1, lse1), (o2, lse2) = pair.forward(first, second, land_d)
    g1, g2 = pair.backward(first, second, t[0]["dout"], t[1]["dout"], lse1, lse2, land_d)
    torch.cuda.synchronize()
    assert C.swin_attn_status(pair.wmsa.plan) == C.SWIN_OK and C.swin_attn_status(pair.swmsa.plan) == C.SWIN_OK
    for (wl, x), o, grads in ((layers[0], o1, g1), (layers[1], o2, g2)):
        pb = problem_of(wl)
        o_ref, _ = oracle.fwd(pb, x["q"], x["k"], x["v"], x["bias"], land)
        assert_close("O", host(o), o_ref, "bf16")
        ref = oracle.bwd(pb, x["q"], x["k"], x["v"], x["bias"], land, x["dout"])
        for key, got in zip(("dq", "dk", "dv", "dbias"), grads):
            assert_close(key, host(got), ref[key], "bf16")
    # W-MSA: no token carries a region bit; both plans share the bias rows
    ws0, reg0, _, rel0 = C.swin_attn_plan_tables(pair.wmsa.plan)
    ws1, reg1, _, rel1 = C.swin_attn_plan_tables(pair.swmsa.plan)
    assert not reg0.any() and reg1.any()
    assert np.array_equal(rel0, rel1)
