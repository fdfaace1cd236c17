"""The key-tiled head_dim-128 kernels on the pages' largest windows, through
the C ABI, against the oracle's sampled-row form (oracle.query_rows,
oracle.key_rows: each output row from its whole window, no n x n matrix):

* TERRA's w = 64 (4 096 tokens) with land, checked at every token;
* TERRA's w = 128 (16 384 tokens) with land and a ragged seam window;
* BEAST's inner windows [180, 30] (5 400 tokens) and outer windows
  [360, 180] (64 800 tokens, 507 key tiles), ragged in latitude.

These windows run without a relative-position bias: the pages put them
through FlashAttention / cuDNN attention, which has none (and the kernels
hold at most 4 096 bias rows). O, LSE and dQ are compared at sampled query
tokens of every window and region; dK and dV at sampled key tokens of the
windows listed per case (the oracle needs the LSE of every query of a key's
region, O(n_r^2 hd)). The backward runs both ways (delta recomputed; delta =
dout . O)."""
import numpy as np
import pytest

import oracle
from shifted_window_attention_cyclic_gb300 import workloads
from tests.parity_util import assert_close, host, problem_of, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CASES = {
    # grid, window, shift, periodic, heads, land, queries per group, key groups (lat window, lon window,
    # region or None for all), keys per group; None: every token
    "terra_w64": ((128, 200), (64, 64), (32, 32), (0, 1), 2, 0.3, None, None, None),
    # lat window 1 splits at lat 192 (two regions of 8 192 slots); lon window 4 is 28 wide and wraps the seam
    "terra_w128": ((256, 540), (128, 128), (64, 64), (0, 1), 1, 0.3, 12, [(1, 0, None), (0, 4, None)], 24),
    # lat window 0 splits at lat 110 (3 300 + 2 100 slots); lat window 1 holds 20 of its 180 rows
    "beast_inner": ((200, 90), (180, 30), (90, 15), (0, 1), 2, None, 8, [(0, 1, None), (1, 2, None)], 16),
    # lat window 0 splits at lat 220 (39 600 + 25 200 slots); lat window 1 holds 40 of its 360 rows
    "beast_outer": ((400, 360), (360, 180), (180, 90), (0, 1), 1, None, 8, [(0, 0, 1), (1, 1, None)], 16),
}


def _sample(pb, tok, live, per_group, rng, groups=None):
    """Tokens of each (window, region) group (all groups, or those listed as
    (lat window, lon window, region or None)): the group's first and last
    live slots in window order (its first and last key tiles) plus random
    ones."""
    gid, slot, reg = oracle.route(pb, tok)
    nw1 = pb.windows_per_dim[1]
    out = []
    for g in np.unique(gid):
        wlat, wlon = divmod(int(g), nw1)
        for r in np.unique(reg[gid == g]):
            if groups is not None and (wlat, wlon, None) not in groups and (wlat, wlon, int(r)) not in groups:
                continue
            sel = np.flatnonzero((gid == g) & (reg == r) & live)
            if sel.size == 0:
                continue
            order = sel[np.argsort(slot[sel])]
            pick = {int(order[0]), int(order[-1])}
            pick.update(int(x) for x in rng.choice(sel, size=min(per_group, sel.size), replace=False))
            out.extend(sorted(pick))
    return np.array(out, np.int64)


@pytest.mark.parametrize("name", list(CASES))
def test_large_window_rows_match_the_oracle(name):
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    grid, window, shift, periodic, heads, land_p, per_q, key_groups, per_k = CASES[name]
    wl = workloads.custom(grid, window, shift, periodic, heads, 128, 1, "bf16",
                          None if land_p is None else (land_p, land_p), seed_index=950 + list(CASES).index(name))
    x = workloads.generate(wl)
    x["bias"] = np.zeros_like(x["bias"])
    pb = problem_of(wl)
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.dtype,
                               wl.has_land)
    assert attn.info.impl == C.SWIN_IMPL_TC and attn.info.slots == int(np.prod(window))
    t = to_device(x, wl, torch.device("cuda", 0))
    o, lse = attn.forward(t["q"], t["k"], t["v"], None, t["land"])
    grads = {}
    for mode in ("delta_recomputed", "delta_from_o"):
        grads[mode] = attn.backward(t["q"], t["k"], t["v"], t["dout"], lse, None, t["land"], want_dbias=False,
                                    o=o if mode == "delta_from_o" else None)
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK

    N, Cc = pb.tokens, pb.channels
    tok = np.arange(N, dtype=np.int64)
    live = np.ones(N, bool) if x["land"] is None else x["land"].reshape(-1) == 0
    rng = np.random.default_rng(7)
    q_tok = tok if per_q is None else _sample(pb, tok, np.ones(N, bool), per_q, rng)
    k_tok = tok if per_k is None else _sample(pb, tok, live, per_k, rng, key_groups)
    assert q_tok.size and k_tok.size

    o_ref, lse_ref, dq_ref = oracle.query_rows(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], q_tok, x["dout"])
    dk_ref, dv_ref = oracle.key_rows(pb, x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"], k_tok)

    flat = lambda a: host(a).reshape(N, Cc)
    assert_close("O", flat(o)[q_tok], o_ref, "bf16")
    lse_got = lse.cpu().numpy().astype(np.float64).reshape(heads, N)[:, q_tok].T
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_got), fin)
    assert np.abs(lse_got[fin] - lse_ref[fin]).max() <= 2e-3
    for mode, (dq, dk, dv, _) in grads.items():
        assert_close("dq " + mode, flat(dq)[q_tok], dq_ref, "bf16")
        assert_close("dk " + mode, flat(dk)[k_tok], dk_ref, "bf16")
        assert_close("dv " + mode, flat(dv)[k_tok], dv_ref, "bf16")
        if x["land"] is not None:
            for got in (dq, dk, dv):
                assert np.all(flat(got)[~live] == 0.0)
    if x["land"] is not None:
        assert np.all(flat(o)[~live] == 0.0)
