"""The attention half of a Swin block in one launch (swin_attn_block_fwd:
LayerNorm + QKV projection, SW-MSA, out-projection + residual) against the
block oracle (oracle/block.py) element by element, on 2-D and 3-D grids with
ragged windows, land, W-MSA (shift 0), C = 64 .. 256, and on the 1-degree
grid of the configs (2 x 180 x 360, C = 256) in full.

Tolerance: the bar of the attention outputs (bf16: relative L2 <= 5e-3,
max-abs <= 2e-2) plus the bf16 storage of y itself. The oracle's y is not
rounded; the kernel's is, which adds up to half a bf16 ulp of |y| (2^-9
relative), and a value that lands next to a rounding boundary may round the
other way, which makes it one ulp (2^-8 relative): max-abs <= 2e-2 +
2^-8 |y_ref|. The rest (fp32 against fp64 LayerNorm and products, P in bf16
for the PV product) is the attention's own error, propagated through W_o."""
import numpy as np
import pytest

from oracle import block as oblock
from shifted_window_attention_cyclic_gb300 import workloads
from tests.parity_util import BF16_MAX_ABS, BF16_REL_L2, problem_of

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EPS = 1e-5

CASES = [
    # grid, window, shift, periodic, heads, batch, land
    ((12, 20), (4, 8), (2, 4), (0, 1), 2, 2, (0.3, 0.3)),
    ((13, 23), (6, 12), (3, 6), (0, 1), 4, 1, None),
    ((4, 16, 32), (2, 8, 8), (1, 4, 4), (0, 0, 1), 8, 1, (0.3, 0.6)),
    ((15, 22), (7, 7), (0, 0), (0, 0), 6, 1, (0.2, 0.2)),
    ((9, 40), (8, 16), (4, 8), (1, 1), 8, 1, None),
    # every token land: attention contributes nothing, y = x + b_o
    ((8, 16), (4, 8), (2, 4), (0, 1), 2, 1, (1.0, 1.0)),
    # windows of 8 slots: the second softmax warpgroup has no keys
    ((6, 12), (2, 4), (1, 2), (0, 1), 4, 2, (0.3, 0.3)),
]


def _run(wl, x):
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    dev = torch.device("cuda", 0)
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, 32, wl.batch, "bf16",
                               wl.has_land)
    t = lambda a, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(dt)
    land = None if x["land"] is None else torch.from_numpy(x["land"]).to(dev)
    y = attn.block_forward(t(x["x"], torch.bfloat16), t(x["gamma"]), t(x["beta"]), t(x["w_qkv"], torch.bfloat16),
                           t(x["b_qkv"]), t(x["w_o"], torch.bfloat16), t(x["b_o"]), t(x["bias"]), land, EPS)
    torch.cuda.synchronize()
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    assert C.swin_attn_status(attn.plan) == 0
    return y.float().cpu().numpy().astype(np.float64)


def _compare(wl, x):
    y = _run(wl, x)
    ref, _ = oblock.block_fwd(problem_of(wl), x["x"], x["gamma"], x["beta"], EPS, x["w_qkv"], x["b_qkv"],
                              x["w_o"], x["b_o"], x["bias"], x["land"])
    assert np.isfinite(y).all()
    diff = np.abs(y - ref)
    excess = float((diff - (BF16_MAX_ABS + 2.0 ** -8 * np.abs(ref))).max())
    rel = float(np.linalg.norm(y - ref) / np.linalg.norm(ref))
    assert excess <= 0.0, "max-abs over the bar by %.3e (max-abs %.3e)" % (excess, diff.max())
    assert rel <= BF16_REL_L2, "relative L2 %.3e" % rel
    return float(diff.max()), rel


@pytest.mark.parametrize("case", CASES)
def test_block_matches_the_oracle(case):
    grid, window, shift, periodic, heads, batch, land_p = case
    wl = workloads.custom(grid, window, shift, periodic, heads, 32, batch, "bf16", land_p, seed_index=900)
    _compare(wl, workloads.generate_block(wl))


def test_block_on_the_one_degree_grid():
    wl = workloads.WORKLOADS["grid1deg"]
    _compare(wl, workloads.generate_block(wl))


def test_block_rejects_what_it_does_not_support():
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    dev = torch.device("cuda", 0)
    # 12 heads of 32: C = 384 is over the 256 channels the kernel holds
    attn = SwinWindowAttention((8, 16), (4, 8), (2, 4), (0, 1), 12, 32, 1, "bf16", False)
    c = 384
    x = torch.zeros((1, 8, 16, c), dtype=torch.bfloat16, device=dev)
    f = lambda *s: torch.zeros(s, dtype=torch.float32, device=dev)
    w = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device=dev)
    with pytest.raises(C.SwinAttnError) as e:
        attn.block_forward(x, f(c), f(c), w(3 * c, c), f(3 * c), w(c, c), f(c))
    assert e.value.code == C.SWIN_ERR_UNSUPPORTED
    # y overlapping x
    attn2 = SwinWindowAttention((8, 16), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16", False)
    c = 64
    x = torch.zeros((1, 8, 16, c), dtype=torch.bfloat16, device=dev)
    with pytest.raises(C.SwinAttnError) as e:
        attn2.block_forward(x, f(c), f(c), w(3 * c, c), f(3 * c), w(c, c), f(c), y=x)
    assert e.value.code == C.SWIN_ERR_INVALID_ARG
