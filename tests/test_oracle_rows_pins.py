"""Pins of the oracle's sampled-row entry points (oracle.route, query_rows,
key_rows), which check windows too large for the per-window form: against
the per-window oracle (itself pinned in test_oracle_pins.py) on every token
of small grids, against the token-pair brute force, and against the
definition's invariants (a query's probabilities sum to one, so the dV of a
region's keys add up to the dout of its queries, and the dS of a query sum to
zero, so the dK of a region's keys add up to zero)."""
import numpy as np
import pytest

import oracle
from oracle import Problem, bruteforce

CASES = [
    # grid, window, shift, periodic, heads, head_dim, batch, land
    ((6, 10), (3, 5), (1, 2), (0, 1), 2, 8, 1, True),       # periodic lon, land
    ((7, 9), (3, 4), (1, 2), (1, 0), 1, 4, 2, False),       # ragged both dims, batch 2
    ((3, 5, 8), (2, 3, 4), (1, 1, 2), (0, 0, 1), 2, 8, 1, True),  # 3-D, ragged depth and lat
    ((4, 6), (4, 6), (0, 0), (0, 0), 1, 8, 1, False),       # one window, no shift (plain attention)
]


def _inputs(pb, seed):
    rng = np.random.default_rng(seed)
    shape = (pb.batch,) + tuple(pb.grid) + (pb.channels,)
    q, k, v, dout = (rng.standard_normal(shape).astype(np.float32) for _ in range(4))
    bias = (0.5 * rng.standard_normal((pb.bias_rows, pb.heads))).astype(np.float32)
    land = (rng.random((pb.batch,) + tuple(pb.grid)) < 0.3).astype(np.uint8) if pb.has_land else None
    return q, k, v, bias, dout, land


def _pb(case):
    grid, window, shift, periodic, heads, hd, batch, land = case
    return Problem(grid=grid, window=window, shift=shift, periodic=periodic, heads=heads, head_dim=hd, batch=batch,
                   has_land=land)


@pytest.mark.parametrize("case", CASES)
def test_route_matches_the_window_tables(oracle_mod, case):
    pb = _pb(case)
    win_src, region, _, _ = oracle.tables(pb)
    tok = np.arange(pb.batch * pb.tokens)
    gid, slot, reg = oracle.route(pb, tok)
    b, t = np.divmod(tok, pb.tokens)
    assert np.array_equal(gid // pb.nwin, b)
    w = gid % pb.nwin
    assert np.array_equal(win_src[w, slot], t)
    assert np.array_equal(region[w, slot], reg)


@pytest.mark.parametrize("case", CASES)
def test_query_rows_match_the_window_oracle(oracle_mod, case):
    pb = _pb(case)
    q, k, v, bias, dout, land = _inputs(pb, 11 + CASES.index(case))
    o_ref, lse_ref = oracle.fwd(pb, q, k, v, bias, land)
    g = oracle.bwd(pb, q, k, v, bias, land, dout)
    tok = np.random.default_rng(1).permutation(pb.batch * pb.tokens)  # every token, in a scrambled order
    o, lse, dq = oracle.query_rows(pb, q, k, v, bias, land, tok, dout)
    b, t = np.divmod(tok, pb.tokens)
    np.testing.assert_allclose(o, o_ref.reshape(pb.batch, pb.tokens, -1)[b, t], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, g["dq"].reshape(pb.batch, pb.tokens, -1)[b, t], rtol=0, atol=1e-12)
    lr = lse_ref.reshape(pb.batch, pb.heads, pb.tokens)[b, :, t]
    assert np.array_equal(np.isfinite(lse), np.isfinite(lr))
    np.testing.assert_allclose(lse[np.isfinite(lse)], lr[np.isfinite(lr)], rtol=0, atol=1e-12)
    _, lse_only, none = oracle.query_rows(pb, q, k, v, bias, land, tok[:5])
    assert none is None and np.array_equal(lse_only, lse[:5])


@pytest.mark.parametrize("case", CASES)
def test_key_rows_match_the_window_oracle(oracle_mod, case):
    pb = _pb(case)
    q, k, v, bias, dout, land = _inputs(pb, 21 + CASES.index(case))
    g = oracle.bwd(pb, q, k, v, bias, land, dout)
    tok = np.random.default_rng(2).permutation(pb.batch * pb.tokens)
    dk, dv = oracle.key_rows(pb, q, k, v, bias, land, dout, tok)
    b, t = np.divmod(tok, pb.tokens)
    np.testing.assert_allclose(dk, g["dk"].reshape(pb.batch, pb.tokens, -1)[b, t], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, g["dv"].reshape(pb.batch, pb.tokens, -1)[b, t], rtol=0, atol=1e-12)


def test_query_rows_match_the_token_pair_brute_force(oracle_mod):
    pb = Problem(grid=(5, 9), window=(2, 4), shift=(1, 2), periodic=(0, 1), heads=2, head_dim=4, batch=1,
                 has_land=True)
    q, k, v, bias, _, land = _inputs(pb, 31)
    o_bf, lse_bf = bruteforce.fwd(pb, q, k, v, bias, land)
    tok = np.arange(pb.tokens)
    o, lse, _ = oracle.query_rows(pb, q, k, v, bias, land, tok)
    np.testing.assert_allclose(o, o_bf.reshape(pb.tokens, -1), rtol=0, atol=1e-12)
    lb = lse_bf.reshape(pb.heads, pb.tokens).T
    assert np.array_equal(np.isfinite(lse), np.isfinite(lb))
    np.testing.assert_allclose(lse[np.isfinite(lse)], lb[np.isfinite(lb)], rtol=0, atol=1e-12)


def test_key_rows_satisfy_the_region_sums(oracle_mod):
    # every live query's probabilities sum to one over the keys it sees (its
    # region's live keys), so sum_j dV_j over a region = sum_i dout_i over the
    # region's live queries; sum_j dS_ij = 0 for every query, so sum_j dK_j = 0
    pb = Problem(grid=(9, 16), window=(4, 8), shift=(2, 4), periodic=(0, 1), heads=2, head_dim=8, batch=1,
                 has_land=True)
    q, k, v, bias, dout, land = _inputs(pb, 41)
    tok = np.arange(pb.tokens)
    dk, dv = oracle.key_rows(pb, q, k, v, bias, land, dout, tok)
    gid, _, reg = oracle.route(pb, tok)
    live = land.reshape(-1) == 0
    do = dout.reshape(pb.tokens, -1).astype(np.float64)
    groups = 0
    for g_ in np.unique(gid):
        for r in np.unique(reg[gid == g_]):
            sel = (gid == g_) & (reg == r) & live
            if not sel.any():
                continue
            groups += 1
            np.testing.assert_allclose(dv[sel].sum(0), do[sel].sum(0), rtol=0, atol=1e-12)
            np.testing.assert_allclose(dk[sel].sum(0), 0.0, rtol=0, atol=1e-12)
    assert groups == 8  # 6 windows; the two that straddle lat 7 | 8 hold both regions
    assert np.all(dk[~live] == 0) and np.all(dv[~live] == 0)


def test_rows_reject_bad_tokens(oracle_mod):
    pb = Problem(grid=(4, 6), window=(2, 3), shift=(1, 1), periodic=(0, 1), heads=1, head_dim=4)
    q, k, v, bias, dout, land = _inputs(pb, 51)
    for bad in ([-1], [pb.tokens]):
        with pytest.raises(ValueError):
            oracle.query_rows(pb, q, k, v, bias, land, bad)
        with pytest.raises(ValueError):
            oracle.key_rows(pb, q, k, v, bias, land, dout, bad)


def _random_cases():
    from tests.test_oracle_pins import _random_problems
    return _random_problems(24, 4711)


@pytest.mark.parametrize("pb", _random_cases(), ids=lambda pb: "g%s_w%s_s%s_p%s" % (
    "x".join(map(str, pb.grid)), "x".join(map(str, pb.window)), "".join(map(str, pb.shift)),
    "".join(map(str, pb.periodic))))
def test_rows_match_the_token_pair_form_on_random_geometries(oracle_mod, pb):
    # every token of seeded tiny geometries over the whole descriptor space
    # (2-D and 3-D, windows that do not divide or exceed the grid, every shift
    # and periodic combination, land, batch 2): O and LSE against the
    # token-pair brute force, dQ, dK and dV against torch autograd through the
    # same token-pair form; neither forms a window table
    from tests.test_oracle_pins import _bruteforce_grads
    q, k, v, bias, dout, land = _inputs(pb, 61)
    tok = np.arange(pb.batch * pb.tokens)
    o, lse, dq = oracle.query_rows(pb, q, k, v, bias, land, tok, dout)
    dk, dv = oracle.key_rows(pb, q, k, v, bias, land, dout, tok)
    o_bf, lse_bf = bruteforce.fwd(pb, q, k, v, bias, land)
    g = _bruteforce_grads(pb, q, k, v, bias, land, dout)
    flat = lambda a: np.asarray(a).reshape(pb.batch * pb.tokens, -1)
    np.testing.assert_allclose(o, flat(o_bf), rtol=0, atol=1e-12)
    lb = np.transpose(np.asarray(lse_bf).reshape(pb.batch, pb.heads, pb.tokens), (0, 2, 1)).reshape(-1, pb.heads)
    assert np.array_equal(np.isfinite(lse), np.isfinite(lb))
    np.testing.assert_allclose(lse[np.isfinite(lse)], lb[np.isfinite(lb)], rtol=0, atol=1e-12)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(got, flat(g[name]), rtol=0, atol=1e-11, err_msg=name)
