"""Plain fp64 oracle of the Swin attention block's forward with its neighbours:
LayerNorm, the QKV projection, shifted-window attention, the out-projection
and the residual add.

TEST INFRASTRUCTURE ONLY (same callers as the rest of ``oracle``); it imports
nothing from the product package.

What it follows:
* TERRA, Fig. 4 (the Swin block: "Layernorm", then window attention, then
  the MLP) and Sec. III (Swin blocks of W-MSA and SW-MSA); the BEAST page,
  "Model Architecture" (Swin blocks). The pages name the block's parts but
  not their formulas; the plainest reading, taken here, is the usual pre-norm
  Swin block's attention half:
      Xn = LayerNorm(X) = (X - mean) / sqrt(var + eps) * gamma + beta
           (mean and biased variance over the C channels of each token),
      [Q | K | V] = Xn W_qkv^T + b_qkv     (W_qkv [3C, C]: rows 0..C-1 give Q,
           C..2C-1 give K, 2C..3C-1 give V; head h owns channels h*hd..h*hd+hd-1
           of each),
      O = SW-MSA(Q, K, V; bias, masks)     (the existing oracle, ``oracle.fwd``),
      Y = X + O W_o^T + b_o                (W_o [C, C], rows = output channel).
* Precision: the attention's inputs are bf16 (BEAST runs its attention in
  bf16), so Q, K and V are rounded to bf16 before the attention, and so is
  its output O before the out-projection, and Xn before the QKV projection
  (the projections are bf16 tensor-core products with fp32 accumulation).
  Each rounding is to nearest, ties to even, of the value first rounded to
  float32 (the kernel rounds its float32 results the same way). Everything
  else is fp64.

Pins (tests/test_oracle_block_pins.py): LayerNorm against a hand-computed row and
against torch's layer_norm in fp64; the block with W_o = 0 and b_o = 0 gives
Y = X exactly; the whole block against an independent composition (torch
fp64 layer_norm and linear around the token-pair brute force) on tiny grids.
"""
from __future__ import annotations

import numpy as np

from . import Problem, fwd


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 (ties to even), returned as float64."""
    f = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def layer_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis (Ba, Kiros and Hinton's layer normalisation):
    mean and biased variance of each token's channels, fp64."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x - mean) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def qkv_projection(xn: np.ndarray, w_qkv: np.ndarray, b_qkv: np.ndarray):
    """[Q | K | V] = Xn W_qkv^T + b_qkv, split into three [..., C] arrays (fp64)."""
    y = np.asarray(xn, np.float64) @ np.asarray(w_qkv, np.float64).T + np.asarray(b_qkv, np.float64)
    c = y.shape[-1] // 3
    return y[..., :c], y[..., c:2 * c], y[..., 2 * c:]


def block_fwd(pb: Problem, x, gamma, beta, eps, w_qkv, b_qkv, w_o, b_o, bias, land=None):
    """Y [B, *grid, C] fp64 of the attention half of a Swin block (see the
    module docstring), plus the intermediates as a dict (xn, q, k, v, o)."""
    x = np.asarray(x, np.float64)
    xn = round_bf16(layer_norm(x, gamma, beta, eps))
    q, k, v = qkv_projection(xn, round_bf16(w_qkv), b_qkv)
    q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
    o, _ = fwd(pb, q, k, v, bias, land)
    ob = round_bf16(o)
    y = x + ob @ round_bf16(w_o).T.astype(np.float64) + np.asarray(b_o, np.float64)
    return y, {"xn": xn, "q": q, "k": k, "v": v, "o": o}
