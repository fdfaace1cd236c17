"""Torch-facing wrapper: a reusable plan + workspace and an autograd Function.

PyTorch only allocates device memory and provides the stream; both passes are
single calls into the CUDA library (swin_attn_fwd, swin_attn_bwd).
"""
from __future__ import annotations

import torch

from . import swin_attn as C

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


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
        self.device = torch.device("cuda", torch.cuda.current_device())
        self._ws = None

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
        if o is None:
            o = torch.empty(self.shape, dtype=self.torch_dtype, device=self.device)
        if lse is None and need_lse:
            lse = torch.empty(self.lse_shape, dtype=torch.float32, device=self.device)
        C.swin_attn_fwd(self.plan, q, k, v, bias, land if self.has_land else None, o, lse, stream)
        return o, lse

    def backward(self, q, k, v, dout, lse, bias=None, land=None, dq=None, dk=None, dv=None, dbias=None,
                 want_dbias=True, stream=None):
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        if dbias is None and want_dbias:
            dbias = self.new_bias()
        ws = self.workspace() if dbias is not None else None
        C.swin_attn_bwd(self.plan, q, k, v, dout, lse, bias, land if self.has_land else None, dq, dk, dv, dbias,
                        ws, stream)
        return dq, dk, dv, dbias


class _SwinAttnFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, attn, q, k, v, bias, land):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o, lse = attn.forward(q, k, v, bias, land)
        ctx.attn = attn
        ctx.save_for_backward(q, k, v, bias, land, lse)
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, bias, land, lse = ctx.saved_tensors
        want_dbias = bias is not None and ctx.needs_input_grad[4]
        dq, dk, dv, dbias = ctx.attn.backward(q, k, v, dout.contiguous(), lse, bias, land, want_dbias=want_dbias)
        return None, dq, dk, dv, dbias, None


def swin_window_attention(attn: SwinWindowAttention, q, k, v, bias=None, land=None):
    """Autograd-aware SW-MSA: returns O; gradients flow to q, k, v and bias."""
    return _SwinAttnFn.apply(attn, q, k, v, bias, land)
