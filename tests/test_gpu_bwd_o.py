"""swin_attn_bwd_o on the kernels that recompute delta in the pass that needs
it (head_dim 32 on tcgen05, fp32 on SIMT): the forward's output is ignored
there, so the gradients equal swin_attn_bwd's bit for bit (dBias of these
kernels is deterministic)."""
import pytest

from shifted_window_attention_cyclic_gb300 import workloads
from tests.parity_util import to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_fp32", "ragged"])
def test_bwd_o_equals_bwd_where_delta_is_recomputed(name):
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    wl = workloads.WORKLOADS[name]
    x = workloads.generate(wl)
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch, wl.dtype,
                               wl.has_land)
    t = to_device(x, wl, torch.device("cuda", 0))
    o, lse = attn.forward(t["q"], t["k"], t["v"], t["bias"], t["land"])
    g1 = attn.backward(t["q"], t["k"], t["v"], t["dout"], lse, t["bias"], t["land"])
    g2 = attn.backward(t["q"], t["k"], t["v"], t["dout"], lse, t["bias"], t["land"], o=o)
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
