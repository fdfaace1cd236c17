"""swin_attn_bwd_noalloc: the backward for callers that cannot allocate
device memory (no device allocator of their own, or a memory pool they may
not touch while stepping). Its partial dBias tables live in a fixed array
inside the library instead of a caller workspace.

Checked through the C ABI against the workspace entry point swin_attn_bwd and
against the CPU oracle, on two calls in a row that follow a call on other
inputs (so the array holds another call's tables when each compared call
starts), with the same tolerances as the other parity tests; neither torch's
allocator nor the device's free memory moves across those calls. This file
is collected last."""
import numpy as np
import pytest

import oracle
from shifted_window_attention_cyclic_gb300 import workloads
from tests.parity_util import assert_close, host, problem_of, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _grads_via(attn, t, lse, noalloc, dout=None):
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    dq, dk, dv = (torch.full_like(t["q"], float("nan")) for _ in range(3))
    dbias = torch.full((attn.info.bias_rows, attn.heads), float("nan"), device=t["q"].device)
    dout = t["dout"] if dout is None else dout
    if noalloc:
        C.swin_attn_bwd_noalloc(attn.plan, t["q"], t["k"], t["v"], dout, lse, t["bias"], t["land"], dq, dk, dv,
                                dbias)
    else:
        C.swin_attn_bwd(attn.plan, t["q"], t["k"], t["v"], dout, lse, t["bias"], t["land"], dq, dk, dv, dbias,
                        attn.workspace())
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK
    return {"dq": dq, "dk": dk, "dv": dv, "dbias": dbias}


def _noalloc_into(attn, t, lse, out):
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    C.swin_attn_bwd_noalloc(attn.plan, t["q"], t["k"], t["v"], t["dout"], lse, t["bias"], t["land"], out["dq"],
                            out["dk"], out["dv"], out["dbias"])
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK


@pytest.mark.parametrize("case", [
    ((181, 362), (8, 8), (4, 4), (0, 1), 12, 32, 1, "bf16", None),          # ragged grid, tensor-core path
    ((4, 9, 21), (2, 4, 8), (1, 2, 4), (0, 0, 1), 3, 32, 2, "bf16", (0.2, 0.5)),
    ((16, 32), (4, 8), (2, 4), (0, 0), 2, 16, 1, "f32", None),              # fp32 path
])
def test_noalloc_matches_workspace_entry_point_twice(case):
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    grid, window, shift, periodic, heads, hd, batch, dtype, land_p = case
    wl = workloads.custom(grid, window, shift, periodic, heads, hd, batch, dtype, land_p, seed_index=700)
    x = workloads.generate(wl)
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch,
                               wl.dtype, wl.has_land)
    t = to_device(x, wl, torch.device("cuda", 0))
    _, lse = attn.forward(t["q"], t["k"], t["v"], t["bias"], t["land"])
    ref = _grads_via(attn, t, lse, noalloc=False)
    g = oracle.bwd(problem_of(wl), x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"])
    # a call on another upstream gradient leaves other partial tables in the array
    other = _grads_via(attn, t, lse, noalloc=True, dout=torch.flip(t["dout"], dims=[1]))
    assert np.isfinite(host(other["dbias"])).all()
    outs = [{k_: torch.full_like(v_, float("nan")) for k_, v_ in ref.items()} for _ in range(2)]
    torch.cuda.synchronize()
    used, free = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for out in outs:
        _noalloc_into(attn, t, lse, out)
    assert torch.cuda.memory_allocated() == used
    assert torch.cuda.mem_get_info()[0] == free
    for out in outs:
        for key in ("dq", "dk", "dv", "dbias"):
            got = host(out[key])
            assert np.isfinite(got).all()
            assert_close(key, got, host(ref[key]), wl.dtype)
            assert_close(key, got, g[key], wl.dtype)


def test_noalloc_rejects_plans_beyond_its_array():
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    # 2048 heads on a 2x8x8 window: (CTAs + heads) partial tables of 675 rows exceed 4 MiB
    attn = SwinWindowAttention((2, 8, 8), (2, 8, 8), (1, 4, 4), (0, 0, 1), 2048, 32)
    need = C.swin_attn_workspace_bytes(attn.plan)
    assert need > 4 << 20
    dev = torch.device("cuda", 0)
    q = torch.zeros(attn.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(attn.lse_shape, device=dev)
    dbias = attn.new_bias()
    with pytest.raises(C.SwinAttnError) as err:
        C.swin_attn_bwd_noalloc(attn.plan, q, q, q, q, lse, None, None, q, q, q, dbias)
    assert err.value.code == C.SWIN_ERR_WORKSPACE
    # without dbias the array is not needed, so the same plan is accepted
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    C.swin_attn_bwd_noalloc(attn.plan, q, q, q, q, lse, None, None, dq, dk, dv, None)
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK
    for d in (dq, dk, dv):
        assert torch.isfinite(d).all()
