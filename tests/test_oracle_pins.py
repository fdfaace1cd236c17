"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle (oracle/swin_oracle.c) against a fact that the
pages or the mathematics fix: a hand-derived routing table, the slot-side
closed form of the route, a token-pair brute force that never forms a window
table, library attention (torch SDPA, float64) on the special cases that reduce
to it, closed forms, invariants, and central finite differences.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import Problem, bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(pb, seed, land_p=None, bf16=True):
    rng = np.random.default_rng(seed)
    shape = (pb.batch,) + tuple(pb.grid) + (pb.channels,)

    def nrm(s, std=1.0):
        x = (rng.standard_normal(s) * std).astype(np.float32)
        if bf16:  # coarse mantissa keeps finite-difference steps exact in float32
            x = (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
        return x

    q, k, v, dout = nrm(shape), nrm(shape), nrm(shape), nrm(shape)
    bias = nrm((pb.bias_rows, pb.heads), 0.5)
    land = None
    if pb.has_land:
        land = (rng.random((pb.batch,) + tuple(pb.grid)) < (land_p or 0.3)).astype(np.uint8)
    return q, k, v, bias, dout, land


# ---------------------------------------------------------------- routing ---

def _read_golden():
    rows = {}
    with open(os.path.join(GOLDEN, "routing_4x6_w2x4_s1x2.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":")
            rows[key.strip()] = [int(x) for x in vals.split()]
    return rows


def test_golden_routing_table(oracle_mod):
    pb = Problem(grid=(4, 6), window=(2, 4), shift=(1, 2), periodic=(0, 1), heads=1, head_dim=4)
    g = _read_golden()
    win_src, region, tok_dst, relidx = oracle.tables(pb)
    for w in range(4):
        assert list(win_src[w]) == g["win_src %d" % w]
        assert list(region[w]) == g["region %d" % w]
    assert list(tok_dst) == g["tok_dst"]
    for key in [k for k in g if k.startswith("relidx")]:
        _, i, j = key.split()
        assert relidx[int(i), int(j)] == g[key][0]


def _slot_side_tables(pb):
    """win_src and region from the slot side: u_d = (w_d*W_d + s_d + S_d) mod G_d."""
    nwd = pb.windows_per_dim
    win_src = np.full((pb.nwin, pb.slots), -1, np.int64)
    region = np.zeros((pb.nwin, pb.slots), np.uint8)
    for wf in range(pb.nwin):
        wc = np.unravel_index(wf, nwd)
        for sf in range(pb.slots):
            sc = np.unravel_index(sf, pb.window)
            p = [wc[a] * pb.window[a] + sc[a] for a in range(pb.ndim)]
            if any(p[a] >= pb.grid[a] for a in range(pb.ndim)):
                continue
            u = [(p[a] + pb.shift[a]) % pb.grid[a] for a in range(pb.ndim)]
            win_src[wf, sf] = np.ravel_multi_index(u, pb.grid)
            r = 0
            for a in range(pb.ndim):
                if not pb.periodic[a] and pb.shift[a] > 0 and p[a] >= pb.grid[a] - pb.shift[a]:
                    r |= 1 << a
            region[wf, sf] = r
    return win_src, region


ROUTING_CASES = [
    ((4, 6), (2, 4), (1, 2), (0, 1)),
    ((16, 32), (4, 8), (2, 4), (0, 0)),
    ((13, 21), (4, 8), (2, 4), (0, 1)),
    ((13, 21), (4, 8), (3, 7), (1, 0)),
    ((9, 10), (9, 10), (0, 0), (0, 1)),
    ((7, 11), (3, 5), (0, 0), (0, 1)),
    ((5, 9, 14), (2, 4, 4), (1, 2, 2), (0, 0, 1)),
    ((3, 7, 10), (2, 3, 4), (1, 1, 3), (0, 1, 1)),
    ((181, 362), (8, 8), (4, 4), (0, 1)),
]


@pytest.mark.parametrize("grid,window,shift,periodic", ROUTING_CASES)
def test_tables_match_slot_side_closed_form(oracle_mod, grid, window, shift, periodic):
    pb = Problem(grid=grid, window=window, shift=shift, periodic=periodic, heads=1, head_dim=4)
    win_src, region, tok_dst, relidx = oracle.tables(pb)
    ws2, reg2 = _slot_side_tables(pb)
    np.testing.assert_array_equal(win_src, ws2)
    np.testing.assert_array_equal(region, reg2)
    # bijection: every token fills exactly one slot, and the inverse route returns it
    flat = win_src.reshape(-1)
    real = flat[flat >= 0]
    assert np.array_equal(np.sort(real), np.arange(pb.tokens))
    assert np.array_equal(flat[tok_dst], np.arange(pb.tokens))
    # shift then unshift is the identity on a random field
    x = np.random.default_rng(0).standard_normal(pb.tokens)
    windowed = np.where(flat >= 0, x[np.maximum(flat, 0)], np.nan)
    assert np.array_equal(windowed[tok_dst], x)


def test_relidx_structure(oracle_mod):
    pb = Problem(grid=(5, 9, 14), window=(2, 4, 4), shift=(1, 2, 2), periodic=(0, 0, 1), heads=1, head_dim=4)
    relidx = oracle.tables(pb)[3]
    n, rows = pb.slots, pb.bias_rows
    center = int(np.ravel_multi_index([w - 1 for w in pb.window], [2 * w - 1 for w in pb.window]))
    assert np.all(np.diag(relidx) == center)
    assert np.all(relidx + relidx.T == 2 * center)
    assert relidx.min() == 0 and relidx.max() == rows - 1
    assert len(np.unique(relidx)) == rows
    # relative offsets: equal offsets share a row, different offsets do not
    offs = np.array([np.unravel_index(s, pb.window) for s in range(n)])
    for i in range(0, n, 7):
        for j in range(0, n, 5):
            d = tuple(offs[i] - offs[j] + np.array(pb.window) - 1)
            assert relidx[i, j] == np.ravel_multi_index(d, [2 * w - 1 for w in pb.window])


# ---------------------------------------------------------------- forward ---

FWD_CASES = [
    # grid, window, shift, periodic, heads, hd, batch, land
    ((8, 16), (4, 8), (2, 4), (0, 0), 2, 8, 1, False),
    ((13, 21), (4, 8), (2, 4), (0, 1), 2, 8, 2, True),
    ((9, 10), (3, 5), (1, 2), (1, 1), 1, 16, 1, True),
    ((11, 9), (4, 4), (3, 1), (0, 1), 3, 4, 1, False),
    ((4, 7, 10), (2, 4, 4), (1, 2, 2), (0, 0, 1), 2, 8, 1, True),
    ((3, 5, 9), (2, 3, 4), (0, 0, 0), (0, 0, 1), 1, 8, 2, False),
    # periodic along depth and lon, ragged in all three dims, unequal shifts
    ((5, 6, 11), (2, 4, 4), (1, 2, 3), (1, 0, 1), 2, 8, 1, True),
]


@pytest.mark.parametrize("case", FWD_CASES)
def test_fwd_matches_token_pair_bruteforce(oracle_mod, case):
    grid, window, shift, periodic, heads, hd, batch, land = case
    pb = Problem(grid=grid, window=window, shift=shift, periodic=periodic, heads=heads, head_dim=hd,
                 batch=batch, has_land=land)
    q, k, v, bias, _, landm = _inputs(pb, 11)
    o, lse = oracle.fwd(pb, q, k, v, bias, landm)
    o2, lse2 = bruteforce.fwd(pb, q, k, v, bias, landm)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)


def _sdpa(qw, kw, vw, mask_add):
    """Library attention, float64 CPU: [H, L, hd] x3 with an additive [H, L, L] mask."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qw), torch.from_numpy(kw), torch.from_numpy(vw),
        attn_mask=torch.from_numpy(mask_add)).numpy()


def _window_slices(pb):
    import itertools
    ranges = [range(0, g, w) for g, w in zip(pb.grid, pb.window)]
    for start in itertools.product(*ranges):
        yield tuple(slice(s, min(s + w, g)) for s, w, g in zip(start, pb.window, pb.grid))


@pytest.mark.parametrize("grid,window,periodic,land", [((12, 20), (4, 8), (0, 1), False),
                                                        ((13, 21), (4, 8), (0, 1), True),
                                                        ((5, 9, 14), (2, 4, 4), (0, 0, 1), True)])
def test_shift0_equals_independent_window_attention(oracle_mod, grid, window, periodic, land):
    """shift = 0: W-MSA, i.e. plain attention inside each window slice."""
    pb = Problem(grid=grid, window=window, shift=(0,) * len(grid), periodic=periodic, heads=2, head_dim=8,
                 has_land=land)
    q, k, v, bias, _, landm = _inputs(pb, 3)
    o, _ = oracle.fwd(pb, q, k, v, bias, landm)
    H, hd = pb.heads, pb.head_dim
    for sl in _window_slices(pb):
        full = (0,) + sl
        qs, ks, vs = (np.asarray(x[full], np.float64).reshape(-1, H, hd).transpose(1, 0, 2) for x in (q, k, v))
        shp = [s.stop - s.start for s in sl]
        offs = np.array(np.unravel_index(np.arange(int(np.prod(shp))), shp)).T
        rows = np.zeros((len(offs), len(offs)), np.int64)
        for a, w in enumerate(pb.window):
            rows = rows * (2 * w - 1) + (offs[:, None, a] - offs[None, :, a] + w - 1)
        mask = np.transpose(np.asarray(bias, np.float64)[rows], (2, 0, 1)).copy()
        lnd = np.zeros(len(offs), bool) if landm is None else landm[full].reshape(-1).astype(bool)
        if lnd.all():
            continue
        mask[:, :, lnd] = -np.inf
        ref = _sdpa(qs, ks, vs, mask).transpose(1, 0, 2).reshape(shp + [pb.channels])
        ref[lnd.reshape(shp)] = 0.0
        np.testing.assert_allclose(o[full], ref, rtol=0, atol=1e-12)


def test_single_window_equals_global_attention(oracle_mod):
    pb = Problem(grid=(7, 12), window=(7, 12), shift=(0, 0), periodic=(0, 1), heads=2, head_dim=8)
    q, k, v, bias, _, _ = _inputs(pb, 5)
    o, _ = oracle.fwd(pb, q, k, v, bias)
    H, hd, N = pb.heads, pb.head_dim, pb.tokens
    qs, ks, vs = (np.asarray(x, np.float64).reshape(N, H, hd).transpose(1, 0, 2) for x in (q, k, v))
    relidx = oracle.tables(pb)[3]
    mask = np.transpose(np.asarray(bias, np.float64)[relidx], (2, 0, 1)).copy()
    ref = _sdpa(qs, ks, vs, mask).transpose(1, 0, 2).reshape(o.shape)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", FWD_CASES)
def test_rows_sum_to_one_and_masked_keys_have_zero_weight(oracle_mod, case):
    grid, window, shift, periodic, heads, hd, batch, land = case
    pb = Problem(grid=grid, window=window, shift=shift, periodic=periodic, heads=heads, head_dim=hd,
                 batch=batch, has_land=land)
    q, k, v, bias, _, landm = _inputs(pb, 7)
    ones = np.ones_like(v)
    o1, _ = oracle.fwd(pb, q, k, ones, bias, landm)
    ocean = np.ones(o1.shape[:-1], bool) if landm is None else ~landm.astype(bool)
    np.testing.assert_allclose(o1[ocean], 1.0, rtol=0, atol=1e-12)
    if landm is not None:
        assert np.all(o1[~ocean] == 0.0)
        # land keys: arbitrary K and V on land tokens leave every output bit-identical
        o, lse = oracle.fwd(pb, q, k, v, bias, landm)
        k2, v2 = k.copy(), v.copy()
        k2[~ocean] = 1e3
        v2[~ocean] = -7e3
        o2, lse2 = oracle.fwd(pb, q, k2, v2, bias, landm)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_region_mask_blocks_wrapped_tokens(oracle_mod):
    """A token that wrapped across the non-periodic lat edge must not see the
    non-wrapped tokens of its window, and vice versa."""
    pb = Problem(grid=(8, 8), window=(4, 4), shift=(2, 0), periodic=(0, 1), heads=1, head_dim=4)
    q, k, v, bias, _, _ = _inputs(pb, 9)
    o, _ = oracle.fwd(pb, q, k, v, bias)
    # rows 0,1 wrapped into the last lat window together with rows 6,7
    k2, v2 = k.copy(), v.copy()
    k2[0, 0:2] = 50.0
    v2[0, 0:2] = 1e4
    o2, _ = oracle.fwd(pb, q, k2, v2, bias)
    assert np.array_equal(o[0, 6:8], o2[0, 6:8])
    assert not np.allclose(o[0, 0:2], o2[0, 0:2])


def test_zero_query_gives_mean_of_visible_values(oracle_mod):
    pb = Problem(grid=(12, 20), window=(4, 5), shift=(0, 0), periodic=(0, 1), heads=2, head_dim=4, has_land=True)
    _, k, v, _, _, landm = _inputs(pb, 13)
    q = np.zeros_like(k)
    bias = np.zeros((pb.bias_rows, pb.heads), np.float32)
    o, _ = oracle.fwd(pb, q, k, v, bias, landm)
    for sl in _window_slices(pb):
        full = (0,) + sl
        lnd = landm[full].astype(bool)
        if lnd.all():
            continue
        mean = np.asarray(v[full], np.float64)[~lnd].mean(0)
        np.testing.assert_allclose(o[full][~lnd], np.broadcast_to(mean, o[full][~lnd].shape), rtol=0, atol=1e-12)


def test_lon_roll_equivariance(oracle_mod):
    """With W divisible by w_lon, rolling inputs and land along the periodic lon
    axis by a multiple of w_lon rolls the outputs by the same amount."""
    for s_lon in (0, 3, 5):
        pb = Problem(grid=(9, 24), window=(3, 6), shift=(1, s_lon), periodic=(0, 1), heads=2, head_dim=4,
                     has_land=True)
        q, k, v, bias, _, landm = _inputs(pb, 17)
        o, _ = oracle.fwd(pb, q, k, v, bias, landm)
        r = 12
        rq, rk, rv = (np.roll(x, r, axis=2) for x in (q, k, v))
        o2, _ = oracle.fwd(pb, rq, rk, rv, bias, np.roll(landm, r, axis=2))
        np.testing.assert_allclose(o2, np.roll(o, r, axis=2), rtol=0, atol=1e-13)


# --------------------------------------------------------------- backward ---

def _loss(pb, q, k, v, bias, land, dout):
    o, _ = oracle.fwd(pb, q, k, v, bias, land)
    return float(np.sum(o * np.asarray(dout, np.float64)))


@pytest.mark.parametrize("case", [FWD_CASES[1], FWD_CASES[4], ((16, 32), (4, 8), (2, 4), (0, 0), 2, 16, 1, False)])
def test_bwd_matches_central_differences(oracle_mod, case):
    grid, window, shift, periodic, heads, hd, batch, land = case
    pb = Problem(grid=grid, window=window, shift=shift, periodic=periodic, heads=heads, head_dim=hd,
                 batch=batch, has_land=land)
    q, k, v, bias, dout, landm = _inputs(pb, 21)
    g = oracle.bwd(pb, q, k, v, bias, landm, dout)
    rng = np.random.default_rng(1)
    eps = 2.0 ** -10  # exact in float32 for bf16-grained inputs
    for name, x in (("dq", q), ("dk", k), ("dv", v), ("dbias", bias)):
        flat = x.reshape(-1)
        picks = rng.choice(flat.size, size=12, replace=False)
        for p in picks:
            xp, xm = x.copy(), x.copy()
            xp.reshape(-1)[p] += eps
            xm.reshape(-1)[p] -= eps
            args = {"q": q, "k": k, "v": v, "bias": bias}
            key = name[1:]
            args[key] = xp
            lp = _loss(pb, args["q"], args["k"], args["v"], args["bias"], landm, dout)
            args[key] = xm
            lm = _loss(pb, args["q"], args["k"], args["v"], args["bias"], landm, dout)
            fd = (lp - lm) / (2 * eps)
            an = g[name].reshape(-1)[p]
            assert abs(fd - an) <= 2e-6 + 1e-5 * abs(an), (name, p, fd, an)


def test_bwd_matches_library_autograd_on_w_msa(oracle_mod):
    """shift = 0, no land: each window is plain attention, so torch autograd
    through float64 SDPA gives dQ, dK, dV and the per-window bias gradient."""
    pb = Problem(grid=(8, 12), window=(4, 6), shift=(0, 0), periodic=(0, 1), heads=2, head_dim=8)
    q, k, v, bias, dout, _ = _inputs(pb, 23)
    g = oracle.bwd(pb, q, k, v, bias, None, dout)
    H, hd = pb.heads, pb.head_dim
    relidx = oracle.tables(pb)[3]
    btab = torch.tensor(bias, dtype=torch.float64, requires_grad=True)
    total = 0.0
    grads = {n: np.zeros(q.shape) for n in ("dq", "dk", "dv")}
    for sl in _window_slices(pb):
        full = (0,) + sl
        t = [torch.tensor(np.asarray(x[full], np.float64).reshape(-1, H, hd).transpose(1, 0, 2).copy(),
                          requires_grad=True) for x in (q, k, v)]
        mask = btab[torch.from_numpy(relidx.astype(np.int64))].permute(2, 0, 1)
        o = torch.nn.functional.scaled_dot_product_attention(t[0], t[1], t[2], attn_mask=mask)
        go = torch.from_numpy(np.asarray(dout[full], np.float64).reshape(-1, H, hd).transpose(1, 0, 2).copy())
        total = total + (o * go).sum()
        o.backward(go, retain_graph=False)
        for n, tt in zip(("dq", "dk", "dv"), t):
            grads[n][full] = tt.grad.numpy().transpose(1, 0, 2).reshape(grads[n][full].shape)
    for n in ("dq", "dk", "dv"):
        np.testing.assert_allclose(g[n], grads[n], rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dbias"], btab.grad.numpy(), rtol=0, atol=1e-12)


def test_bwd_window_subset_matches_full(oracle_mod):
    pb = Problem(grid=(13, 21), window=(4, 8), shift=(2, 4), periodic=(0, 1), heads=2, head_dim=8, batch=2,
                 has_land=True)
    q, k, v, bias, dout, landm = _inputs(pb, 29)
    full = oracle.bwd_windows(pb, q, k, v, bias, landm, dout)
    ids = np.array([3, 0, pb.nwin + 5, 2 * pb.nwin - 1])
    sub = oracle.bwd_windows(pb, q, k, v, bias, landm, dout, win_ids=ids)
    for n in ("dq", "dk", "dv"):
        np.testing.assert_array_equal(sub[n], full[n][ids])
    o_full, l_full = oracle.fwd_windows(pb, q, k, v, bias, landm)
    o_sub, l_sub = oracle.fwd_windows(pb, q, k, v, bias, landm, win_ids=ids)
    np.testing.assert_array_equal(o_sub, o_full[ids])
    np.testing.assert_array_equal(l_sub, l_full[ids])


@pytest.mark.parametrize("case", [FWD_CASES[1], FWD_CASES[4], ((9, 20), (3, 8), (1, 4), (1, 1), 2, 8, 2, True)])
def test_bwd_softmax_gradient_sums(oracle_mod, case):
    """Every softmax row sums to one, so its gradient row dS sums to zero.
    Summed over all tokens (the route is a bijection): dBias sums to zero per
    head, dK sums to zero per channel, and dV sums to the sum of dO over the
    tokens whose output is not forced to zero (sea tokens). Using P or dS
    untransposed for dK or dV breaks these sums, since column sums are not one
    or zero."""
    grid, window, shift, periodic, heads, hd, batch, land = case
    pb = Problem(grid=grid, window=window, shift=shift, periodic=periodic, heads=heads, head_dim=hd,
                 batch=batch, has_land=land)
    q, k, v, bias, dout, landm = _inputs(pb, 31, land_p=0.3)
    g = oracle.bwd(pb, q, k, v, bias, landm, dout)
    C = pb.channels
    scale = np.abs(g["dk"]).max() + np.abs(g["dbias"]).max()
    np.testing.assert_allclose(g["dbias"].sum(axis=0), 0.0, atol=1e-12 * scale * g["dbias"].size)
    np.testing.assert_allclose(g["dk"].reshape(-1, C).sum(axis=0), 0.0, atol=1e-12 * scale * g["dk"].size)
    sea = np.ones(g["dv"].shape[:-1], bool) if landm is None else ~landm.astype(bool)
    want = np.asarray(dout, np.float64)[sea].sum(axis=0)
    np.testing.assert_allclose(g["dv"].reshape(-1, C).sum(axis=0), want, rtol=0, atol=1e-10)
    if landm is not None:
        for key in ("dq", "dk", "dv"):
            assert np.all(g[key][~sea] == 0.0)


# ------------------------------------------------- random tiny geometries ---

def _random_problems(count, seed):
    """Seeded descriptors over the whole valid space at tiny sizes: 2-D and
    3-D, windows that do not divide (or exceed) the grid, every shift and
    periodic combination, batch and heads 1-2, with and without land."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        nd = int(rng.integers(2, 4))
        grid = tuple(int(rng.integers(1, 10 if nd == 2 else 7)) for _ in range(nd))
        window = tuple(int(rng.integers(1, min(g + 2, 6) + 1)) for g in grid)
        if int(np.prod(window)) > 128:
            continue
        shift = tuple(int(rng.integers(0, w)) for w in window)
        shift = tuple(s if s < g else 0 for s, g in zip(shift, grid))
        periodic = tuple(int(rng.integers(0, 2)) for _ in range(nd))
        out.append(Problem(grid=grid, window=window, shift=shift, periodic=periodic,
                           heads=int(rng.integers(1, 3)), head_dim=int(rng.choice([4, 8])),
                           batch=int(rng.integers(1, 3)), has_land=bool(rng.integers(0, 2))))
    return out


RANDOM = _random_problems(40, 2026)


def _bruteforce_grads(pb, q, k, v, bias, land, dout):
    """dQ, dK, dV, dBias by torch autograd (float64) through the token-pair
    form: full N x N visibility from the definition, no window table. Land
    queries have O = 0, so they pass no gradient."""
    win, off, region = bruteforce._token_geometry(pb.grid, pb.window, pb.shift, pb.periodic)
    rows = torch.from_numpy(bruteforce._pair_rows(off, pb.window))
    shape = (pb.batch, pb.tokens, pb.heads, pb.head_dim)
    t = [torch.tensor(np.asarray(x, np.float64).reshape(shape), requires_grad=True) for x in (q, k, v)]
    btab = torch.tensor(np.asarray(bias, np.float64), requires_grad=True)
    go = torch.from_numpy(np.asarray(dout, np.float64).reshape(shape))
    total = 0.0
    for b in range(pb.batch):
        land_b = None if land is None else np.asarray(land).reshape(pb.batch, pb.tokens)[b].astype(bool)
        vis = torch.from_numpy(bruteforce.visibility(pb.grid, pb.window, pb.shift, pb.periodic, land_b))
        sea = torch.ones(pb.tokens, dtype=torch.float64) if land_b is None else torch.from_numpy(~land_b).double()
        empty = ~vis.any(1)
        for h in range(pb.heads):
            s = t[0][b, :, h] @ t[1][b, :, h].T / np.sqrt(pb.head_dim) + btab[rows, h]
            s = s.masked_fill(~vis, float("-inf")).masked_fill(empty[:, None], 0.0)
            o = torch.softmax(s, 1) @ t[2][b, :, h] * sea[:, None]
            total = total + (o * go[b, :, h]).sum()
    total.backward()
    g = {n: x.grad.numpy().reshape((pb.batch,) + tuple(pb.grid) + (pb.channels,))
         for n, x in zip(("dq", "dk", "dv"), t)}
    g["dbias"] = btab.grad.numpy()
    return g


@pytest.mark.parametrize("pb", RANDOM, ids=lambda pb: "g%s_w%s_s%s_p%s" % (
    "x".join(map(str, pb.grid)), "x".join(map(str, pb.window)), "".join(map(str, pb.shift)),
    "".join(map(str, pb.periodic))))
def test_random_geometry_matches_bruteforce(oracle_mod, pb):
    win_src, region, tok_dst, _ = oracle.tables(pb)
    ws2, reg2 = _slot_side_tables(pb)
    np.testing.assert_array_equal(win_src, ws2)
    np.testing.assert_array_equal(region, reg2)
    flat = win_src.reshape(-1)
    assert np.array_equal(np.sort(flat[flat >= 0]), np.arange(pb.tokens))
    assert np.array_equal(flat[tok_dst], np.arange(pb.tokens))
    q, k, v, bias, dout, landm = _inputs(pb, 41, land_p=0.35)
    o, lse = oracle.fwd(pb, q, k, v, bias, landm)
    o2, lse2 = bruteforce.fwd(pb, q, k, v, bias, landm)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)
    g = oracle.bwd(pb, q, k, v, bias, landm, dout)
    g2 = _bruteforce_grads(pb, q, k, v, bias, landm, dout)
    for key in ("dq", "dk", "dv", "dbias"):
        np.testing.assert_allclose(g[key], g2[key], rtol=0, atol=1e-11, err_msg=key)
