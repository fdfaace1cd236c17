"""Pins of the block oracle (oracle/block.py: LayerNorm, QKV projection,
shifted-window attention, out-projection, residual) against things other than
itself: a hand-computed LayerNorm row, torch's layer_norm and bfloat16
conversion, an exact special case, and an independent composition of torch
float64 layer_norm / linear around the token-pair brute force."""
import numpy as np
import pytest
import torch

from oracle import Problem, block, bruteforce


def test_layer_norm_hand_row():
    # [1, 2, 3, 4]: mean 2.5, biased variance 1.25, so (x - 2.5) / sqrt(1.25)
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    gamma = np.array([1.0, 2.0, 3.0, 4.0])
    beta = np.array([0.5, -0.5, 0.0, 1.0])
    s = np.sqrt(1.25)
    want = np.array([-1.5 / s * 1.0 + 0.5, -0.5 / s * 2.0 - 0.5, 0.5 / s * 3.0, 1.5 / s * 4.0 + 1.0])
    np.testing.assert_allclose(block.layer_norm(x, gamma, beta, 0.0)[0], want, rtol=0, atol=1e-15)


def test_layer_norm_matches_torch_and_standardises():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 7, 96)) * 3.0 + 1.5
    gamma, beta = rng.standard_normal(96), rng.standard_normal(96)
    got = block.layer_norm(x, gamma, beta, 1e-5)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(gamma),
                                         torch.from_numpy(beta), 1e-5).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    z = block.layer_norm(x, np.ones(96), np.zeros(96), 0.0)
    np.testing.assert_allclose(z.mean(-1), 0.0, atol=1e-13)
    np.testing.assert_allclose((z ** 2).mean(-1), 1.0, atol=1e-12)


def test_round_bf16_ties_to_even_and_matches_torch():
    one = 1.0
    assert block.round_bf16(np.array([one]))[0] == 1.0
    assert block.round_bf16(np.array([one + 2.0 ** -8]))[0] == 1.0                 # tie, even stays
    assert block.round_bf16(np.array([one + 3 * 2.0 ** -8]))[0] == one + 2.0 ** -6  # tie, odd rounds up
    assert block.round_bf16(np.array([-(one + 2.0 ** -7 + 2.0 ** -12)]))[0] == -(one + 2.0 ** -7)
    x = np.random.default_rng(4).standard_normal(4096) * 10.0
    ref = torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(block.round_bf16(x), ref)


def _block_inputs(pb, seed):
    rng = np.random.default_rng(seed)
    c = pb.channels
    x = rng.standard_normal((pb.batch,) + tuple(pb.grid) + (c,)).astype(np.float32)
    x = block.round_bf16(x)
    gamma = 1.0 + 0.1 * rng.standard_normal(c)
    beta = 0.1 * rng.standard_normal(c)
    w_qkv = rng.standard_normal((3 * c, c)) / np.sqrt(c)
    b_qkv = 0.1 * rng.standard_normal(3 * c)
    w_o = rng.standard_normal((c, c)) / np.sqrt(c)
    b_o = 0.1 * rng.standard_normal(c)
    bias = 0.5 * rng.standard_normal((pb.bias_rows, pb.heads))
    land = None
    if pb.has_land:
        land = (rng.random((pb.batch,) + tuple(pb.grid)) < 0.3).astype(np.uint8)
    return x, gamma, beta, w_qkv, b_qkv, w_o, b_o, bias, land


def test_zero_out_projection_gives_the_residual():
    pb = Problem(grid=(6, 10), window=(3, 5), shift=(1, 2), periodic=(0, 1), heads=2, head_dim=8, batch=1,
                 has_land=True)
    x, gamma, beta, w_qkv, b_qkv, w_o, b_o, bias, land = _block_inputs(pb, 5)
    y, _ = block.block_fwd(pb, x, gamma, beta, 1e-5, w_qkv, b_qkv, np.zeros_like(w_o), np.zeros_like(b_o),
                           bias, land)
    np.testing.assert_array_equal(y, x)


def _bf16_t(t):
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)


BLOCK_CASES = [
    ((6, 10), (3, 5), (1, 2), (0, 1), 2, 8, 1, True),
    ((5, 9), (2, 4), (1, 2), (1, 1), 3, 4, 2, False),
    ((3, 5, 8), (2, 3, 4), (1, 1, 2), (0, 0, 1), 2, 8, 1, True),
]


@pytest.mark.parametrize("case", BLOCK_CASES)
def test_block_matches_independent_composition(case):
    grid, window, shift, periodic, heads, hd, batch, land = case
    pb = Problem(grid=grid, window=window, shift=shift, periodic=periodic, heads=heads, head_dim=hd,
                 batch=batch, has_land=land)
    x, gamma, beta, w_qkv, b_qkv, w_o, b_o, bias, landm = _block_inputs(pb, 6)
    y, _ = block.block_fwd(pb, x, gamma, beta, 1e-5, w_qkv, b_qkv, w_o, b_o, bias, landm)
    c = pb.channels
    xt = torch.from_numpy(x)
    xn = _bf16_t(torch.nn.functional.layer_norm(xt, (c,), torch.from_numpy(gamma), torch.from_numpy(beta), 1e-5))
    qkv = torch.nn.functional.linear(xn, _bf16_t(torch.from_numpy(w_qkv)), torch.from_numpy(b_qkv))
    q, k, v = (_bf16_t(t).numpy() for t in qkv.split(c, dim=-1))
    o, _ = bruteforce.fwd(pb, q, k, v, bias, landm)
    o = _bf16_t(torch.from_numpy(o.reshape(x.shape)))
    ref = xt + torch.nn.functional.linear(o, _bf16_t(torch.from_numpy(w_o)), torch.from_numpy(b_o))
    np.testing.assert_allclose(y, ref.numpy(), rtol=0, atol=1e-10)
