"""Token-pair brute force for tiny grids (test infrastructure only).

Builds the full N x N visibility matrix straight from the definition, token by
token, and never forms a window table:

1. rolled position p = (u - s) mod G (roll by -s; BEAST page, "Model
   Architecture": the domain is rolled between attention layers);
2. window coordinate floor(p / w), in-window offset p mod w (TERRA,
   Sec. IV.D "Differentiable Token Routes");
3. region bit per non-periodic dimension with s > 0: p >= G - s;
4. key u' is visible to query u iff same window, same region bits and u' is
   not land;
5. logits hd^-1/2 q.k + bias[row(offset_u, offset_u')], softmax over visible
   keys, O = P V; land queries give O = 0 and LSE = -inf.

Everything is fp64 numpy on [N, N] matrices, so keep N to a few thousand.
"""
from __future__ import annotations

import numpy as np


def _token_geometry(grid, window, shift, periodic):
    G = np.asarray(grid)
    w = np.asarray(window)
    s = np.asarray(shift)
    per = np.asarray(periodic, dtype=bool)
    coords = np.stack(np.meshgrid(*[np.arange(g) for g in grid], indexing="ij"), -1).reshape(-1, len(grid))
    p = np.mod(coords - s, G)
    win = p // w
    off = p % w
    region = (~per) & (s > 0) & (p >= G - s)
    return win, off, region


def _pair_rows(off, window):
    """Bias row of every (query, key) pair from the in-window offsets."""
    row = np.zeros((off.shape[0], off.shape[0]), np.int64)
    for a, w in enumerate(window):
        row = row * (2 * w - 1) + (off[:, None, a] - off[None, :, a] + w - 1)
    return row


def visibility(grid, window, shift, periodic, land_img=None):
    win, off, region = _token_geometry(grid, window, shift, periodic)
    vis = np.all(win[:, None, :] == win[None, :, :], -1) & np.all(region[:, None, :] == region[None, :, :], -1)
    if land_img is not None:
        vis &= ~land_img.reshape(-1).astype(bool)[None, :]
    return vis


def fwd(pb, q, k, v, bias, land=None):
    """O [B, *grid, C] and LSE [B, heads, *grid], fp64."""
    q = np.asarray(q, np.float64).reshape(pb.batch, pb.tokens, pb.heads, pb.head_dim)
    k = np.asarray(k, np.float64).reshape(pb.batch, pb.tokens, pb.heads, pb.head_dim)
    v = np.asarray(v, np.float64).reshape(pb.batch, pb.tokens, pb.heads, pb.head_dim)
    bias = np.asarray(bias, np.float64)
    win, off, region = _token_geometry(pb.grid, pb.window, pb.shift, pb.periodic)
    rows = _pair_rows(off, pb.window)
    o = np.zeros((pb.batch, pb.tokens, pb.heads, pb.head_dim))
    lse = np.zeros((pb.batch, pb.heads, pb.tokens))
    scale = 1.0 / np.sqrt(pb.head_dim)
    for b in range(pb.batch):
        land_b = None
        if pb.has_land and land is not None:
            land_b = np.asarray(land).reshape(pb.batch, pb.tokens)[b].astype(bool)
        vis = visibility(pb.grid, pb.window, pb.shift, pb.periodic, land_b)
        for h in range(pb.heads):
            s = scale * q[b, :, h] @ k[b, :, h].T + bias[rows, h]
            s = np.where(vis, s, -np.inf)
            m = s.max(1, keepdims=True)
            e = np.where(vis, np.exp(s - np.where(np.isfinite(m), m, 0.0)), 0.0)
            l = e.sum(1, keepdims=True)
            p = e / np.where(l > 0, l, 1.0)
            o[b, :, h] = p @ v[b, :, h]
            with np.errstate(divide="ignore"):  # a row with no visible key: log 0 = -inf
                lse[b, h] = (m + np.log(l))[:, 0]
            if land_b is not None:
                o[b, land_b, h] = 0.0
                lse[b, h, land_b] = -np.inf
    return (o.reshape((pb.batch,) + tuple(pb.grid) + (pb.channels,)),
            lse.reshape((pb.batch, pb.heads) + tuple(pb.grid)))
