"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
on seeded workload inputs and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np

import oracle
from oracle import Problem

# Tolerances (the bar of the task): fp32 path max-abs <= 1e-5; bf16 path
# relative L2 <= 5e-3 and max-abs <= 2e-2, for O, dQ, dK, dV and dBias.
F32_MAX_ABS = 1e-5
BF16_REL_L2 = 5e-3
BF16_MAX_ABS = 2e-2


def problem_of(wl):
    return Problem(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.has_land)


def errors(got, ref, mask=None):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    diff = got - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    return max_abs, rel


def assert_close(name, got, ref, dtype, mask=None):
    max_abs, rel = errors(got, ref, mask)
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, "%s: max-abs %.3e > %.1e" % (name, max_abs, F32_MAX_ABS)
    else:
        assert max_abs <= BF16_MAX_ABS and rel <= BF16_REL_L2, \
            "%s: max-abs %.3e (<= %.0e), rel-L2 %.3e (<= %.0e)" % (name, max_abs, BF16_MAX_ABS, rel, BF16_REL_L2)
    return max_abs, rel


def to_device(x, wl, dev):
    import torch
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    out = {}
    for key in ("q", "k", "v", "dout"):
        out[key] = None if x[key] is None else torch.from_numpy(x[key]).to(dev).to(tdt)
    out["bias"] = torch.from_numpy(x["bias"]).to(dev)
    out["land"] = None if x["land"] is None else torch.from_numpy(x["land"]).to(dev)
    return out


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(wl, x, impl="auto", backward=True, dev=None):
    """Forward (and backward) through the C ABI; returns numpy float64 results."""
    import torch
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    dev = dev or torch.device("cuda", 0)
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch,
                               wl.dtype, wl.has_land, impl)
    t = to_device(x, wl, dev)
    o, lse = attn.forward(t["q"], t["k"], t["v"], t["bias"], t["land"])
    res = {"attn": attn, "o": o, "lse": lse}
    if backward:
        dq, dk, dv, dbias = attn.backward(t["q"], t["k"], t["v"], t["dout"], lse, t["bias"], t["land"])
        res.update(dq=dq, dk=dk, dv=dv, dbias=dbias)
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == 0
    return res


def sample_windows(pb, count, seed=0):
    """Window ids that include the grid corners, seam and ragged edges plus random ones."""
    nwd = pb.windows_per_dim
    import itertools
    corner = []
    for wc in itertools.product(*[sorted({0, 1, n // 2, n - 2, n - 1} & set(range(n))) for n in nwd]):
        corner.append(int(np.ravel_multi_index(wc, nwd)))
    rng = np.random.default_rng(seed)
    rand = rng.choice(pb.nwin, size=min(count, pb.nwin), replace=False).tolist()
    ids = []
    for b in range(pb.batch):
        ids += [b * pb.nwin + w for w in sorted(set(corner + rand))]
    return np.array(ids, np.int64)


def gather_windows(pb, grid_arr, win_src, ids):
    """grid_arr [B, N, X] -> per-window slot rows [ids, n, X] (pad rows 0)."""
    out = np.zeros((len(ids), pb.slots) + grid_arr.shape[2:], grid_arr.dtype)
    for x, gid in enumerate(ids):
        b, w = divmod(int(gid), pb.nwin)
        src = win_src[w]
        ok = src >= 0
        out[x][ok] = grid_arr[b, src[ok]]
    return out
