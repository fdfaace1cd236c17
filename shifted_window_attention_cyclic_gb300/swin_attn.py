"""Thin ctypes binding of the C ABI in include/swin_attn.h.

Argument marshalling only: every step of the attention runs in the CUDA
library libswin_attn.so that sits next to this file. There is no fallback;
if the library is missing or cannot load, every call raises.

Function names match the C entry points. Tensors are torch CUDA tensors
(PyTorch supplies device memory and streams); the binding passes their data
pointers and the current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
# SWIN_ATTN_CHECK_BOUNDS=1 selects the bounds-checked testing build of the
# same sources (every kernel-addressed global access range-checked).
CHECK_BOUNDS = os.environ.get("SWIN_ATTN_CHECK_BOUNDS", "0") == "1"
LIB_PATH = os.path.join(HERE, "libswin_attn_bounds.so" if CHECK_BOUNDS else "libswin_attn.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "swin_attn.h")

SWIN_OK = 0
SWIN_ERR_INVALID_ARG = -1
SWIN_ERR_UNSUPPORTED = -2
SWIN_ERR_ALIGNMENT = -3
SWIN_ERR_WORKSPACE = -4
SWIN_ERR_CUDA = -5
SWIN_ERR_TIMEOUT = -6
SWIN_ERR_DEVICE = -7

SWIN_F32 = 0
SWIN_BF16 = 1
SWIN_IMPL_AUTO = 0
SWIN_IMPL_SIMT = 1
SWIN_IMPL_TC = 2


class SwinAttnError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("%s: %s (%d)" % (what, strerror(code), code))
        self.code = code


class swin_attn_desc(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int32), ("impl", ctypes.c_int32), ("batch", ctypes.c_int64),
                ("grid", ctypes.c_int32 * 3), ("window", ctypes.c_int32 * 3),
                ("shift", ctypes.c_int32 * 3), ("periodic", ctypes.c_int32 * 3),
                ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("has_land", ctypes.c_int32)]


class swin_attn_plan_info(ctypes.Structure):
    _fields_ = [("windows_per_image", ctypes.c_int64), ("tokens_per_image", ctypes.c_int64),
                ("slots", ctypes.c_int32), ("bias_rows", ctypes.c_int32), ("impl", ctypes.c_int32),
                ("fwd_ctas", ctypes.c_int32), ("bwd_ctas", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("work_items", ctypes.c_int64), ("dbias_slots", ctypes.c_int64)]


_lib = None


def load_library():
    """Load libswin_attn.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("%s is not built (run __graft_entry__.build()); "
                           "this package has no CPU fallback" % os.path.basename(LIB_PATH))
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.swin_attn_plan.argtypes = [ctypes.POINTER(swin_attn_desc), ctypes.POINTER(vp)]
    lib.swin_attn_plan.restype = ctypes.c_int
    lib.swin_attn_plan_get_info.argtypes = [vp, ctypes.POINTER(swin_attn_plan_info)]
    lib.swin_attn_plan_get_info.restype = ctypes.c_int
    lib.swin_attn_plan_tables.argtypes = [vp, vp, vp, vp, vp]
    lib.swin_attn_plan_tables.restype = ctypes.c_int
    lib.swin_attn_workspace_bytes.argtypes = [vp]
    lib.swin_attn_workspace_bytes.restype = sz
    lib.swin_attn_fwd.argtypes = [vp] * 9
    lib.swin_attn_fwd.restype = ctypes.c_int
    lib.swin_attn_bwd.argtypes = [vp] * 13 + [sz, vp]
    lib.swin_attn_bwd.restype = ctypes.c_int
    lib.swin_attn_bwd_o.argtypes = [vp] * 14 + [sz, vp]
    lib.swin_attn_bwd_o.restype = ctypes.c_int
    lib.swin_attn_bwd_noalloc.argtypes = [vp] * 13
    lib.swin_attn_bwd_noalloc.restype = ctypes.c_int
    lib.swin_attn_block_fwd.argtypes = [vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.swin_attn_block_fwd.restype = ctypes.c_int
    lib.swin_attn_plan_set_debug.argtypes = [vp, ctypes.c_uint64, ctypes.c_int]
    lib.swin_attn_plan_set_debug.restype = ctypes.c_int
    lib.swin_attn_status.argtypes = [vp, vp]
    lib.swin_attn_status.restype = ctypes.c_int
    lib.swin_attn_plan_destroy.argtypes = [vp]
    lib.swin_attn_plan_destroy.restype = None
    lib.swin_attn_strerror.argtypes = [ctypes.c_int]
    lib.swin_attn_strerror.restype = ctypes.c_char_p
    lib.swin_attn_window_range.argtypes = [i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.swin_attn_window_range.restype = ctypes.c_int
    lib.swin_attn_fixed_padded_extent.argtypes = [i64, i64, i64, i64, ctypes.POINTER(i64)]
    lib.swin_attn_fixed_padded_extent.restype = ctypes.c_int
    _lib = lib
    return lib


def declared_symbols():
    """Entry points declared in include/swin_attn.h."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(swin_attn_\w+)\s*\(", text, re.M)))


def strerror(code: int) -> str:
    return load_library().swin_attn_strerror(int(code)).decode()


def _check(code, what):
    if code != SWIN_OK:
        raise SwinAttnError(code, what)


def make_desc(grid, window, shift, periodic, heads, head_dim, batch=1, dtype="bf16", has_land=False,
              impl="auto") -> swin_attn_desc:
    d = swin_attn_desc()
    d.ndim = len(grid)
    d.impl = {"auto": SWIN_IMPL_AUTO, "simt": SWIN_IMPL_SIMT, "tc": SWIN_IMPL_TC}[impl]
    d.batch = batch
    for a in range(len(grid)):
        d.grid[a] = grid[a]
        d.window[a] = window[a]
        d.shift[a] = shift[a]
        d.periodic[a] = int(periodic[a])
    d.heads = heads
    d.head_dim = head_dim
    d.dtype = {"f32": SWIN_F32, "bf16": SWIN_BF16}[dtype] if isinstance(dtype, str) else int(dtype)
    d.has_land = int(bool(has_land))
    return d


class Plan:
    """Owns a swin_attn_plan_t; destroyed with the object."""

    def __init__(self, handle, desc):
        self.handle = handle
        self.desc = desc
        info = swin_attn_plan_info()
        _check(load_library().swin_attn_plan_get_info(handle, ctypes.byref(info)), "swin_attn_plan_get_info")
        self.info = info

    def close(self):
        if self.handle:
            load_library().swin_attn_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def dtype(self):
        return "bf16" if self.desc.dtype == SWIN_BF16 else "f32"

    @property
    def grid(self):
        return tuple(self.desc.grid[a] for a in range(self.desc.ndim))

    @property
    def channels(self):
        return self.desc.heads * self.desc.head_dim


def swin_attn_plan(desc: swin_attn_desc) -> Plan:
    lib = load_library()
    h = ctypes.c_void_p()
    _check(lib.swin_attn_plan(ctypes.byref(desc), ctypes.byref(h)), "swin_attn_plan")
    return Plan(h, desc)


RELIDX_MAX_SLOTS = 2048  # the plan keeps the [n][n] bias-row table for windows up to this size


def swin_attn_plan_tables(plan: Plan):
    """(win_src [nwin, n] int32, region [nwin, n] uint8, tok_dst [N] int32, relidx [n, n] int32, or None
    for windows of more than RELIDX_MAX_SLOTS slots)."""
    nwin, n, N = plan.info.windows_per_image, plan.info.slots, plan.info.tokens_per_image
    win_src = np.empty((nwin, n), np.int32)
    region = np.empty((nwin, n), np.uint8)
    tok_dst = np.empty((N,), np.int32)
    relidx = np.empty((n, n), np.int32) if n <= RELIDX_MAX_SLOTS else None
    p = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    _check(load_library().swin_attn_plan_tables(plan.handle, p(win_src), p(region), p(tok_dst), p(relidx)),
           "swin_attn_plan_tables")
    return win_src, region, tok_dst, relidx


def swin_attn_workspace_bytes(plan: Plan) -> int:
    return int(load_library().swin_attn_workspace_bytes(plan.handle))


def _ptr(t, align=1, what=""):
    """Raw device address of a tensor (None passes NULL). `align` is the
    alignment the library reads it with: 16 bytes for the activations and
    lse (the tensor-core kernels read four LSE values in one load), 4 for
    land (four land bytes in one load), bias and dbias."""
    if t is None:
        return None
    p = t.data_ptr()
    if p % align:
        raise SwinAttnError(SWIN_ERR_ALIGNMENT, "%s not %d-byte aligned" % (what, align))
    return ctypes.c_void_p(p)


def _acts(*named):
    return [_ptr(t, 16, n) for n, t in named]


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def swin_attn_fwd(plan: Plan, q, k, v, bias, land, o, lse, stream=None) -> None:
    pq, pk, pv, po, plse = _acts(("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse))
    _check(load_library().swin_attn_fwd(plan.handle, pq, pk, pv, _ptr(bias, 4, "bias"), _ptr(land, 4, "land"), po,
                                        plse, _stream(stream)), "swin_attn_fwd")


def swin_attn_bwd(plan: Plan, q, k, v, dout, lse, bias, land, dq, dk, dv, dbias, workspace, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    pq, pk, pv, pdo, plse, pdq, pdk, pdv = _acts(("q", q), ("k", k), ("v", v), ("dout", dout), ("lse", lse),
                                                 ("dq", dq), ("dk", dk), ("dv", dv))
    _check(load_library().swin_attn_bwd(plan.handle, pq, pk, pv, pdo, plse, _ptr(bias, 4, "bias"),
                                        _ptr(land, 4, "land"), pdq, pdk, pdv, _ptr(dbias, 4, "dbias"),
                                        _ptr(workspace, 256, "workspace"), ws_bytes, _stream(stream)),
           "swin_attn_bwd")


def swin_attn_bwd_o(plan: Plan, q, k, v, o, dout, lse, bias, land, dq, dk, dv, dbias, workspace,
                    stream=None) -> None:
    """Backward given the forward's output o (head_dim 128: delta from dout . o)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    pq, pk, pv, po, pdo, plse, pdq, pdk, pdv = _acts(("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout),
                                                     ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))
    _check(load_library().swin_attn_bwd_o(plan.handle, pq, pk, pv, po, pdo, plse, _ptr(bias, 4, "bias"),
                                          _ptr(land, 4, "land"), pdq, pdk, pdv, _ptr(dbias, 4, "dbias"),
                                          _ptr(workspace, 256, "workspace"), ws_bytes, _stream(stream)),
           "swin_attn_bwd_o")


def swin_attn_bwd_noalloc(plan: Plan, q, k, v, dout, lse, bias, land, dq, dk, dv, dbias, stream=None) -> None:
    """Backward without a workspace argument: the partial dBias tables live in
    a fixed array inside the library, so the call allocates nothing."""
    pq, pk, pv, pdo, plse, pdq, pdk, pdv = _acts(("q", q), ("k", k), ("v", v), ("dout", dout), ("lse", lse),
                                                 ("dq", dq), ("dk", dk), ("dv", dv))
    _check(load_library().swin_attn_bwd_noalloc(plan.handle, pq, pk, pv, pdo, plse, _ptr(bias, 4, "bias"),
                                                _ptr(land, 4, "land"), pdq, pdk, pdv, _ptr(dbias, 4, "dbias"),
                                                _stream(stream)), "swin_attn_bwd_noalloc")


def swin_attn_block_fwd(plan: Plan, x, ln_gamma, ln_beta, ln_eps, w_qkv, b_qkv, w_o, b_o, bias, land, y,
                        stream=None) -> None:
    """LayerNorm + QKV projection, SW-MSA, out-projection + residual in one
    launch (see include/swin_attn.h); y must not overlap x."""
    px, py, pwq, pwo = _acts(("x", x), ("y", y), ("w_qkv", w_qkv), ("w_o", w_o))
    _check(load_library().swin_attn_block_fwd(plan.handle, px, _ptr(ln_gamma, 4, "ln_gamma"),
                                              _ptr(ln_beta, 4, "ln_beta"), float(ln_eps), pwq,
                                              _ptr(b_qkv, 4, "b_qkv"), pwo, _ptr(b_o, 4, "b_o"),
                                              _ptr(bias, 4, "bias"), _ptr(land, 4, "land"), py, _stream(stream)),
           "swin_attn_block_fwd")


def swin_attn_status(plan: Plan, stream=None) -> int:
    return int(load_library().swin_attn_status(plan.handle, _stream(stream)))


def swin_attn_plan_set_debug(plan: Plan, wait_limit_ns: int, force_timeout: int) -> None:
    _check(load_library().swin_attn_plan_set_debug(plan.handle, int(wait_limit_ns), int(force_timeout)),
           "swin_attn_plan_set_debug")


def swin_attn_plan_destroy(plan: Plan) -> None:
    plan.close()


def swin_attn_window_range(M: int, P: int, r: int):
    L, R = ctypes.c_int64(), ctypes.c_int64()
    _check(load_library().swin_attn_window_range(M, P, r, ctypes.byref(L), ctypes.byref(R)),
           "swin_attn_window_range")
    return L.value, R.value


def swin_attn_fixed_padded_extent(extent: int, stride: int, window: int, ranks: int) -> int:
    padded = ctypes.c_int64()
    _check(load_library().swin_attn_fixed_padded_extent(extent, stride, window, ranks, ctypes.byref(padded)),
           "swin_attn_fixed_padded_extent")
    return padded.value


def swin_attn_strerror(code: int) -> str:
    return strerror(code)
