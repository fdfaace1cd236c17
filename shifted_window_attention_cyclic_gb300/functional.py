"""Torch-facing wrapper: a reusable plan + workspace and an autograd Function.

PyTorch only allocates device memory and provides the stream; both passes are
single calls into the CUDA library (swin_attn_fwd, swin_attn_bwd).
"""
from __future__ import annotations

import torch

from . import swin_attn as C

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def check_tensor(name, t, shape, dtype, device):
    """Raise ValueError unless `t` is a contiguous `dtype` tensor of exactly
    `shape` on `device` whose data starts on a 16-byte boundary. The library
    reads and writes every tensor through a raw pointer and cannot check any
    of this itself; a wrong shape or dtype would read or write past the
    caller's buffers."""
    if not isinstance(t, torch.Tensor):
        raise ValueError("%s: expected a torch.Tensor, got %s" % (name, type(t).__name__))
    if t.device != device:
        raise ValueError("%s: on %s, expected %s" % (name, t.device, device))
    if t.dtype != dtype:
        raise ValueError("%s: dtype %s, expected %s" % (name, t.dtype, dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s: shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if not t.is_contiguous():
        raise ValueError("%s: not contiguous" % name)
    if t.data_ptr() % 16:
        raise ValueError("%s: data not 16-byte aligned" % name)


def check_call(tensors, shape, lse_shape, bias_shape, dtype, device, has_land):
    """Check every tensor of one forward or backward call (None = not passed).
    Activations and their gradients are `dtype` [B, *grid, C]; lse is fp32
    [B, heads, *grid]; bias and dbias are fp32 [rows, heads]; land is uint8
    [B, *grid] and required exactly when the plan was made with a land mask."""
    for name, t in tensors.items():
        if t is None:
            if name == "land" and has_land:
                raise ValueError("land: the plan was made with a land mask; pass uint8 %s" % (tuple(shape[:-1]),))
            continue
        if name in ("bias", "dbias"):
            check_tensor(name, t, bias_shape, torch.float32, device)
        elif name == "lse":
            check_tensor(name, t, lse_shape, torch.float32, device)
        elif name == "land":
            if has_land:
                check_tensor(name, t, shape[:-1], torch.uint8, device)
        else:
            check_tensor(name, t, shape, dtype, device)


class SwinWindowAttention:
    """Shifted-window multi-head self-attention over a [B, *grid, C] tensor.

    grid/window/shift/periodic are per dimension, outermost first
    ((lat, lon) or (depth, lat, lon)); land masks are uint8 [B, *grid].
    """

    def __init__(self, grid, window, shift, periodic, heads, head_dim, batch=1, dtype="bf16", has_land=False,
                 impl="auto", device=None):
        if device is not None:
            torch.cuda.set_device(device)
        self.desc = C.make_desc(grid, window, shift, periodic, heads, head_dim, batch, dtype, has_land, impl)
        self.plan = C.swin_attn_plan(self.desc)
        self.dtype = dtype
        self.torch_dtype = _TORCH_DTYPE[dtype]
        self.shape = (batch,) + tuple(grid) + (heads * head_dim,)
        self.lse_shape = (batch, heads) + tuple(grid)
        self.heads = heads
        self.has_land = has_land
        self.bias_shape = (self.plan.info.bias_rows, heads)
        self.device = torch.device("cuda", torch.cuda.current_device())
        self._ws = None

    def _check(self, **tensors):
        check_call(tensors, self.shape, self.lse_shape, self.bias_shape, self.torch_dtype, self.device,
                   self.has_land)

    @property
    def info(self):
        return self.plan.info

    def workspace(self):
        nbytes = C.swin_attn_workspace_bytes(self.plan)
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def new_bias(self):
        return torch.zeros((self.info.bias_rows, self.heads), dtype=torch.float32, device=self.device)

    def forward(self, q, k, v, bias=None, land=None, o=None, lse=None, need_lse=True, stream=None):
        self._check(q=q, k=k, v=v, bias=bias, land=land, o=o, lse=lse)
        if o is None:
            o = torch.empty(self.shape, dtype=self.torch_dtype, device=self.device)
        if lse is None and need_lse:
            lse = torch.empty(self.lse_shape, dtype=torch.float32, device=self.device)
        C.swin_attn_fwd(self.plan, q, k, v, bias, land if self.has_land else None, o, lse, stream)
        return o, lse

    def backward(self, q, k, v, dout, lse, bias=None, land=None, dq=None, dk=None, dv=None, dbias=None,
                 want_dbias=True, stream=None, o=None):
        """Gradients (dq, dk, dv, dbias). With the forward's output `o`, head_dim
        128 takes delta = dout . o instead of recomputing it (one key sweep less)."""
        if lse is None:
            raise ValueError("lse: the backward needs the forward's log-sum-exp")
        self._check(q=q, k=k, v=v, dout=dout, lse=lse, bias=bias, land=land, dq=dq, dk=dk, dv=dv, dbias=dbias,
                    o=o)
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        if dbias is None and want_dbias:
            dbias = self.new_bias()
        ws = self.workspace()  # dBias partial tables; for head_dim 128 also delta
        if o is None:
            C.swin_attn_bwd(self.plan, q, k, v, dout, lse, bias, land if self.has_land else None, dq, dk, dv, dbias,
                            ws, stream)
        else:
            C.swin_attn_bwd_o(self.plan, q, k, v, o, dout, lse, bias, land if self.has_land else None, dq, dk, dv,
                              dbias, ws, stream)
        return dq, dk, dv, dbias


    def block_forward(self, x, ln_gamma, ln_beta, w_qkv, b_qkv, w_o, b_o, bias=None, land=None, ln_eps=1e-5,
                      y=None, stream=None):
        """The attention half of a Swin block in one launch: y = x + SW-MSA(
        LayerNorm(x) W_qkv^T + b_qkv) W_o^T + b_o (bf16 x, y, W_qkv [3C, C],
        W_o [C, C]; float32 LayerNorm and bias vectors). Forward only."""
        self._check(x=x, bias=bias, land=land, y=y)
        c = self.shape[-1]
        for name, t, shape, dt in (("ln_gamma", ln_gamma, (c,), torch.float32), ("ln_beta", ln_beta, (c,), torch.float32),
                                   ("w_qkv", w_qkv, (3 * c, c), torch.bfloat16), ("b_qkv", b_qkv, (3 * c,), torch.float32),
                                   ("w_o", w_o, (c, c), torch.bfloat16), ("b_o", b_o, (c,), torch.float32)):
            if tuple(t.shape) != shape or t.dtype != dt or t.device != self.device or not t.is_contiguous():
                raise ValueError("%s: want a contiguous %s %s on %s" % (name, dt, shape, self.device))
        if y is None:
            y = torch.empty(self.shape, dtype=self.torch_dtype, device=self.device)
        C.swin_attn_block_fwd(self.plan, x, ln_gamma, ln_beta, ln_eps, w_qkv, b_qkv, w_o, b_o, bias,
                              land if self.has_land else None, y, stream)
        return y


class _SwinAttnFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, attn, q, k, v, bias, land):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o, lse = attn.forward(q, k, v, bias, land)
        ctx.attn = attn
        ctx.save_for_backward(q, k, v, bias, land, lse, o)
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, bias, land, lse, o = ctx.saved_tensors
        want_dbias = bias is not None and ctx.needs_input_grad[4]
        dq, dk, dv, dbias = ctx.attn.backward(q, k, v, dout.contiguous(), lse, bias, land, want_dbias=want_dbias,
                                              o=o)
        return None, dq, dk, dv, dbias, None


def swin_window_attention(attn: SwinWindowAttention, q, k, v, bias=None, land=None):
    """Autograd-aware SW-MSA: returns O; gradients flow to q, k, v and bias."""
    return _SwinAttnFn.apply(attn, q, k, v, bias, land)


class SwinBlockPair:
    """The attention of one Swin block pair over a [B, *grid, C] tensor: W-MSA
    (no shift) in the first block, SW-MSA (the grid rolled by floor(w/2) per
    dim) in the second, as TERRA's Fig. 4 stacks them and as the BEAST page
    rolls the domain by half a window between attention layers.

    Two plans, built once and reused for every step: the shift changes the
    routing tables (window sources, region bits and inverse route); the bias
    row of a slot pair does not depend on it. Each call is one C-ABI call per
    layer; the layers' own projections and MLP sit outside this op.
    """

    def __init__(self, grid, window, periodic, heads, head_dim, batch=1, dtype="bf16", has_land=False,
                 impl="auto", device=None):
        shift = tuple(w // 2 if g > w // 2 else 0 for g, w in zip(grid, window))
        self.shift = shift
        self.wmsa = SwinWindowAttention(grid, window, (0,) * len(grid), periodic, heads, head_dim, batch, dtype,
                                        has_land, impl, device)
        self.swmsa = SwinWindowAttention(grid, window, shift, periodic, heads, head_dim, batch, dtype, has_land,
                                         impl, device)

    def forward(self, first, second, land=None):
        """first, second: (q, k, v, bias) of the W-MSA and the SW-MSA layer.
        Returns ((O, lse) of the first, (O, lse) of the second)."""
        return self.wmsa.forward(*first, land=land), self.swmsa.forward(*second, land=land)

    def backward(self, first, second, dout_first, dout_second, lse_first, lse_second, land=None):
        """Gradients (dq, dk, dv, dbias) of both layers, second layer first
        (the order a training step runs them)."""
        g2 = self.swmsa.backward(*second[:3], dout_second, lse_second, second[3], land)
        g1 = self.wmsa.backward(*first[:3], dout_first, lse_first, first[3], land)
        return g1, g2
