"""Plain fp64 CPU oracle for shifted-window multi-head self-attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers. Nothing in the product
package imports this module, and this module imports nothing from the product
package (it shares no code with the CUDA path).

Two independent implementations of one definition live here:

* ``swin_oracle.c`` (loaded through ctypes): window-by-window, built on routing
  tables derived from each token's own coordinates (TERRA, Sec. IV.D
  "Differentiable Token Routes"; BEAST page, "Model Architecture"), exact
  fp64 softmax attention per window and head, exact backward.
* ``bruteforce``: token-pair form on tiny grids; builds the full N x N
  visibility matrix from the definition and never forms a window table.

See ``swin_oracle.c`` for the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swin_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_swin.so")


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, OpenMP, -O2) next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Desc(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int32), ("pad0", ctypes.c_int32), ("batch", ctypes.c_int64),
                ("grid", ctypes.c_int32 * 3), ("window", ctypes.c_int32 * 3),
                ("shift", ctypes.c_int32 * 3), ("periodic", ctypes.c_int32 * 3),
                ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("has_land", ctypes.c_int32), ("pad1", ctypes.c_int32)]


@dataclass(frozen=True)
class Problem:
    """Geometry of one SW-MSA call. Dimensions are outermost first:
    (lat, lon) or (depth, lat, lon)."""
    grid: tuple
    window: tuple
    shift: tuple
    periodic: tuple
    heads: int
    head_dim: int
    batch: int = 1
    has_land: bool = False

    @property
    def ndim(self):
        return len(self.grid)

    @property
    def channels(self):
        return self.heads * self.head_dim

    @property
    def windows_per_dim(self):
        return tuple(-(-g // w) for g, w in zip(self.grid, self.window))

    @property
    def nwin(self):
        return int(np.prod(self.windows_per_dim))

    @property
    def slots(self):
        return int(np.prod(self.window))

    @property
    def tokens(self):
        return int(np.prod(self.grid))

    @property
    def bias_rows(self):
        return int(np.prod([2 * w - 1 for w in self.window]))

    def _c(self):
        d = _Desc()
        d.ndim = self.ndim
        d.batch = self.batch
        for a in range(self.ndim):
            d.grid[a] = self.grid[a]
            d.window[a] = self.window[a]
            d.shift[a] = self.shift[a]
            d.periodic[a] = int(bool(self.periodic[a]))
        d.heads = self.heads
        d.head_dim = self.head_dim
        d.has_land = int(bool(self.has_land))
        return d


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        lib.oracle_tables.argtypes = [P(_Desc), ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_fwd.argtypes = [P(_Desc)] + [ctypes.c_void_p] * 6 + [ctypes.c_int64,
                                                                        ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_bwd.argtypes = [P(_Desc)] + [ctypes.c_void_p] * 7 + [ctypes.c_int64] + [ctypes.c_void_p] * 4
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_route.argtypes = [P(_Desc), ctypes.c_void_p, ctypes.c_int64] + [ctypes.c_void_p] * 3
        lib.oracle_query_rows.argtypes = [P(_Desc)] + [ctypes.c_void_p] * 7 + [ctypes.c_int64] + [ctypes.c_void_p] * 3
        lib.oracle_key_rows.argtypes = [P(_Desc)] + [ctypes.c_void_p] * 7 + [ctypes.c_int64] + [ctypes.c_void_p] * 2
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().oracle_num_threads()


def tables(pb: Problem, with_relidx: bool = True):
    """Routing tables of one image: (win_src [nwin, n] int32 with -1 pads,
    region [nwin, n] uint8, tok_dst [N] int32, relidx [n, n] int32, or None
    when with_relidx is false: n x n entries are too many for large windows)."""
    lib = _load()
    win_src = np.empty((pb.nwin, pb.slots), np.int32)
    region = np.empty((pb.nwin, pb.slots), np.uint8)
    tok_dst = np.empty((pb.tokens,), np.int32)
    relidx = np.empty((pb.slots, pb.slots), np.int32) if with_relidx else None
    d = pb._c()
    rc = lib.oracle_tables(ctypes.byref(d), _ptr(win_src), _ptr(region), _ptr(tok_dst), _ptr(relidx))
    if rc:
        raise ValueError("oracle_tables failed: %d" % rc)
    return win_src, region, tok_dst, relidx


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _land(pb, land):
    if not pb.has_land:
        return None
    return np.ascontiguousarray(land, dtype=np.uint8)


def fwd_windows(pb: Problem, q, k, v, bias, land=None, win_ids=None):
    """Forward on a list of global window ids (b*nwin + w); None = all.
    Returns (o_win [ids, n, C] f64, lse_win [ids, heads, n] f64)."""
    lib = _load()
    ids = None if win_ids is None else np.ascontiguousarray(win_ids, dtype=np.int64)
    m = pb.batch * pb.nwin if ids is None else len(ids)
    o = np.zeros((m, pb.slots, pb.channels), np.float64)
    lse = np.zeros((m, pb.heads, pb.slots), np.float64)
    q, k, v, bias = _f32(q), _f32(k), _f32(v), _f32(bias)
    landa = _land(pb, land)
    d = pb._c()
    rc = lib.oracle_fwd(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(landa),
                        _ptr(ids), m, _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("oracle_fwd failed: %d" % rc)
    return o, lse


def bwd_windows(pb: Problem, q, k, v, bias, land, dout, win_ids=None, want=("dq", "dk", "dv", "dbias")):
    """Backward on a list of global window ids; None = all (dbias is then the
    full gradient). Returns dict with dq/dk/dv [ids, n, C] and dbias [rows, heads]."""
    lib = _load()
    ids = None if win_ids is None else np.ascontiguousarray(win_ids, dtype=np.int64)
    m = pb.batch * pb.nwin if ids is None else len(ids)
    out = {}
    for key in ("dq", "dk", "dv"):
        out[key] = np.zeros((m, pb.slots, pb.channels), np.float64) if key in want else None
    out["dbias"] = np.zeros((pb.bias_rows, pb.heads), np.float64) if "dbias" in want else None
    q, k, v, bias, dout = _f32(q), _f32(k), _f32(v), _f32(bias), _f32(dout)
    landa = _land(pb, land)
    d = pb._c()
    rc = lib.oracle_bwd(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(landa), _ptr(dout),
                        _ptr(ids), m, _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dbias"]))
    if rc:
        raise ValueError("oracle_bwd failed: %d" % rc)
    return {k_: v_ for k_, v_ in out.items() if v_ is not None}


def scatter_windows(pb: Problem, win_rows, win_src, win_ids=None, fill=0.0):
    """Place per-window slot rows [ids, n, X] back on the grid [B, N, X]
    using the oracle's own win_src table (pad slots are dropped)."""
    m = win_rows.shape[0]
    ids = np.arange(pb.batch * pb.nwin) if win_ids is None else np.asarray(win_ids)
    out = np.full((pb.batch, pb.tokens) + win_rows.shape[2:], fill, dtype=win_rows.dtype)
    for x in range(m):
        b, w = divmod(int(ids[x]), pb.nwin)
        src = win_src[w]
        ok = src >= 0
        out[b, src[ok]] = win_rows[x][ok]
    return out


def fwd(pb: Problem, q, k, v, bias, land=None):
    """Full forward on the grid: O [B, *grid, C] f64 and LSE [B, heads, *grid] f64."""
    win_src = tables(pb)[0]
    o_win, lse_win = fwd_windows(pb, q, k, v, bias, land)
    o = scatter_windows(pb, o_win, win_src)
    lse = scatter_windows(pb, np.transpose(lse_win, (0, 2, 1)), win_src, fill=np.nan)
    return (o.reshape((pb.batch,) + tuple(pb.grid) + (pb.channels,)),
            np.transpose(lse, (0, 2, 1)).reshape((pb.batch, pb.heads) + tuple(pb.grid)))


def bwd(pb: Problem, q, k, v, bias, land, dout):
    """Full backward on the grid: dict of dq/dk/dv [B, *grid, C] and dbias [rows, heads]."""
    win_src = tables(pb)[0]
    g = bwd_windows(pb, q, k, v, bias, land, dout)
    shape = (pb.batch,) + tuple(pb.grid) + (pb.channels,)
    return {"dq": scatter_windows(pb, g["dq"], win_src).reshape(shape),
            "dk": scatter_windows(pb, g["dk"], win_src).reshape(shape),
            "dv": scatter_windows(pb, g["dv"], win_src).reshape(shape),
            "dbias": g["dbias"]}


# ---- sampled rows: windows too large for the per-window form ----------------

def _tokens(pb, tokens):
    t = np.ascontiguousarray(tokens, dtype=np.int64).reshape(-1)
    if t.size and (t.min() < 0 or t.max() >= pb.batch * pb.tokens):
        raise ValueError("token index out of range")
    return t


def route(pb: Problem, tokens):
    """Window (global id b*nwin + w), slot and region bits of flat tokens b*N + t."""
    t = _tokens(pb, tokens)
    gid = np.empty(t.size, np.int64)
    slot = np.empty(t.size, np.int32)
    reg = np.empty(t.size, np.int32)
    d = pb._c()
    rc = _load().oracle_route(ctypes.byref(d), _ptr(t), t.size, _ptr(gid), _ptr(slot), _ptr(reg))
    if rc:
        raise ValueError("oracle_route failed: %d" % rc)
    return gid, slot, reg


def query_rows(pb: Problem, q, k, v, bias, land, tokens, dout=None):
    """O [m, C], LSE [m, heads] and, given dout, dQ [m, C] (fp64) of the query
    tokens listed by flat index b*N + t, each from its whole window; no n x n
    matrix is formed. Returns (o, lse, dq or None)."""
    t = _tokens(pb, tokens)
    o = np.zeros((t.size, pb.channels), np.float64)
    lse = np.zeros((t.size, pb.heads), np.float64)
    dq = np.zeros((t.size, pb.channels), np.float64) if dout is not None else None
    q, k, v, bias, dout = _f32(q), _f32(k), _f32(v), _f32(bias), _f32(dout)
    d = pb._c()
    rc = _load().oracle_query_rows(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(_land(pb, land)),
                                   _ptr(dout), _ptr(t), t.size, _ptr(o), _ptr(lse), _ptr(dq))
    if rc:
        raise ValueError("oracle_query_rows failed: %d" % rc)
    return o, lse, dq


def key_rows(pb: Problem, q, k, v, bias, land, dout, tokens):
    """dK [m, C] and dV [m, C] (fp64) of the tokens listed by flat index as
    keys. Costs O(n_r^2 hd) per (window, head), n_r the queries of the listed
    keys' regions in that window."""
    t = _tokens(pb, tokens)
    dk = np.zeros((t.size, pb.channels), np.float64)
    dv = np.zeros((t.size, pb.channels), np.float64)
    q, k, v, bias, dout = _f32(q), _f32(k), _f32(v), _f32(bias), _f32(dout)
    d = pb._c()
    rc = _load().oracle_key_rows(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(_land(pb, land)),
                                 _ptr(dout), _ptr(t), t.size, _ptr(dk), _ptr(dv))
    if rc:
        raise ValueError("oracle_key_rows failed: %d" % rc)
    return dk, dv
