"""Pin of the shift mask against the standard Swin mask (CPU).

The oracle decides key visibility with a two-label rule per non-periodic
dimension: a token's region bit is set when its rolled position wrapped
across the edge (p >= G - s). The Swin Transformer instead labels every
rolled position with one of three slices per masked dimension, [0, G - w),
[G - w, G - s) and [G - s, G), and lets a query see only keys of its own
window with the same combined label (BEAST page, "Model Architecture": the
domain is rolled by floor(w/2) between layers and attention runs in
Swin-style windows; the tiny 16x32 configuration asks for that standard
mask). Where the window divides the grid, the first two slices never share
a window, so the two rules must give the same visibility; these tests build
the three-slice labels the way Swin does (slicing an image of labels in the
rolled frame, then cutting it into windows) and compare them with the
oracle's visibility, from its routing tables and from its token-pair brute
force. On a ragged grid the two rules differ, and the oracle keeps physical
neighbours together (its stated reading); the last test records that.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import Problem, bruteforce


def swin_three_slice_labels(grid, window, shift, periodic):
    """Label image in the rolled frame: each masked dimension (periodic 0,
    shift > 0) is cut into the slices [0, G - w), [G - w, G - s), [G - s, G),
    and the label counts the slice combinations in order."""
    img = np.zeros(grid, np.int64)
    per_dim = []
    for G, w, s, per in zip(grid, window, shift, periodic):
        if per or s == 0:
            per_dim.append([slice(0, G)])
        else:
            per_dim.append([slice(0, G - w), slice(G - w, G - s), slice(G - s, G)])
    for cnt, sl in enumerate(itertools.product(*per_dim)):
        img[sl] = cnt
    return img


def swin_visibility(grid, window, shift, periodic):
    """N x N visibility (tokens in grid order) under the three-slice mask: a
    rolled position p belongs to window p // w; a query sees the keys of its
    window that carry its label."""
    labels = swin_three_slice_labels(grid, window, shift, periodic)
    G, w, s = (np.asarray(a) for a in (grid, window, shift))
    coords = np.stack(np.meshgrid(*[np.arange(g) for g in grid], indexing="ij"), -1).reshape(-1, len(grid))
    p = np.mod(coords - s, G)  # rolled position of every grid token
    win = p // w
    lab = labels[tuple(p.T)]
    return np.all(win[:, None] == win[None, :], -1) & (lab[:, None] == lab[None, :])


def oracle_table_visibility(pb):
    """N x N visibility from the oracle's routing tables: same window, same region bits."""
    win_src, region, _, _ = oracle.tables(pb)
    win = np.full(pb.tokens, -1)
    reg = np.full(pb.tokens, -1)
    for w in range(pb.nwin):
        ok = win_src[w] >= 0
        win[win_src[w][ok]] = w
        reg[win_src[w][ok]] = region[w][ok]
    assert (win >= 0).all()
    return (win[:, None] == win[None, :]) & (reg[:, None] == reg[None, :])


DIVISIBLE = [
    ((16, 32), (4, 8), (2, 4), (0, 0)),          # the tiny configuration: both dims masked
    ((16, 32), (4, 8), (2, 4), (0, 1)),          # longitude periodic (no slices there)
    ((12, 24), (6, 12), (3, 6), (0, 1)),         # the 1-degree stage's window and shift on a small grid
    ((16, 16), (8, 8), (4, 4), (0, 0)),
    ((16, 24), (8, 12), (4, 6), (0, 0)),         # the eddy stage's window and shift
    ((4, 16, 32), (2, 8, 8), (1, 4, 4), (0, 0, 0)),  # depth-level windows, every dim masked
    ((4, 16, 32), (2, 8, 8), (1, 4, 4), (0, 0, 1)),
    ((6, 8, 12), (2, 4, 4), (1, 1, 3), (0, 0, 0)),   # shifts other than w/2
]


@pytest.mark.parametrize("grid,window,shift,periodic", DIVISIBLE)
def test_two_label_rule_equals_swin_three_slice_mask_on_divisible_grids(oracle_mod, grid, window, shift, periodic):
    pb = Problem(grid, window, shift, periodic, heads=1, head_dim=4)
    swin = swin_visibility(grid, window, shift, periodic)
    assert np.array_equal(bruteforce.visibility(grid, window, shift, periodic), swin)
    assert np.array_equal(oracle_table_visibility(pb), swin)
    # the masks are not trivial: some window holds two or more labels
    assert (swin.sum(1) < int(np.prod(window))).any() == any(s > 0 and not p for s, p in zip(shift, periodic))


def test_two_label_rule_keeps_ragged_neighbours_that_three_slices_split(oracle_mod):
    # G = 13, w = 4, s = 2: windows of rolled rows [8, 12) and the short [12, 13);
    # the three-slice cut at G - w = 9 falls inside the window [8, 12) and
    # separates rows 8 and 9, which are physical neighbours that neither wrapped.
    grid, window, shift, periodic = (13, 4), (4, 4), (2, 0), (0, 0)
    swin = swin_visibility(grid, window, shift, periodic)
    ours = bruteforce.visibility(grid, window, shift, periodic)
    assert not np.array_equal(ours, swin)
    tok = lambda p0, c: ((p0 + 2) % 13) * 4 + c  # token at rolled row p0, column c
    assert ours[tok(8, 0), tok(9, 0)] and not swin[tok(8, 0), tok(9, 0)]
