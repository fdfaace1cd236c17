"""Failure path of the tensor-core kernels, without any GPU fault.

The plan's testing hook makes one role of the next launch wait on an mbarrier
that nothing arrives at. The bounded wait gives up after a short limit, the
CTA drains its copies and MMAs, frees TMEM and exits; the host reads
SWIN_ERR_TIMEOUT from the device status word. The same plan then runs
normally again and matches the oracle, so the context stayed usable."""
import numpy as np
import pytest

import oracle
from shifted_window_attention_cyclic_gb300 import workloads
from tests.parity_util import assert_close, host, problem_of, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_forced_wait_timeout_is_reported_and_recoverable():
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    wl = workloads.custom((13, 27), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16", (0.3, 0.3), seed_index=91)
    x = workloads.generate(wl)
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch,
                               wl.dtype, wl.has_land, "tc")
    assert attn.info.impl == C.SWIN_IMPL_TC
    t = to_device(x, wl, torch.device("cuda", 0))
    C.swin_attn_plan_set_debug(attn.plan, 5_000_000, 1)  # 5 ms limit, forced wait
    attn.forward(t["q"], t["k"], t["v"], t["bias"], t["land"])
    assert C.swin_attn_status(attn.plan) == C.SWIN_ERR_TIMEOUT
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK  # status word was cleared
    C.swin_attn_plan_set_debug(attn.plan, 1_000_000_000, 0)
    o, _ = attn.forward(t["q"], t["k"], t["v"], t["bias"], t["land"])
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK
    o_ref, _ = oracle.fwd(problem_of(wl), x["q"], x["k"], x["v"], x["bias"], x["land"])
    assert_close("O", host(o), o_ref, wl.dtype)


def test_forced_wait_timeout_in_backward_is_reported_and_recoverable():
    """The same failure path in the backward kernel: its softmax warps wait on
    the barrier nothing arrives at; the gather, MMA and epilogue roles see the
    abort flag and leave, copies and MMAs in flight drain, TMEM is freed. The
    plan then runs the backward normally and meets the oracle."""
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    wl = workloads.custom((13, 27), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16", (0.3, 0.3), seed_index=92)
    x = workloads.generate(wl)
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch,
                               wl.dtype, wl.has_land, "tc")
    assert attn.info.impl == C.SWIN_IMPL_TC
    t = to_device(x, wl, torch.device("cuda", 0))
    _, lse = attn.forward(t["q"], t["k"], t["v"], t["bias"], t["land"])
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK
    C.swin_attn_plan_set_debug(attn.plan, 5_000_000, 1)  # 5 ms limit, forced wait
    attn.backward(t["q"], t["k"], t["v"], t["dout"], lse, t["bias"], t["land"])
    assert C.swin_attn_status(attn.plan) == C.SWIN_ERR_TIMEOUT
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK  # status word was cleared
    C.swin_attn_plan_set_debug(attn.plan, 1_000_000_000, 0)
    dq, dk, dv, dbias = attn.backward(t["q"], t["k"], t["v"], t["dout"], lse, t["bias"], t["land"])
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK
    g = oracle.bwd(problem_of(wl), x["q"], x["k"], x["v"], x["bias"], x["land"], x["dout"])
    for key, got in (("dq", dq), ("dk", dk), ("dv", dv), ("dbias", dbias)):
        assert_close(key, host(got), g[key], wl.dtype)


def test_debug_hook_rejects_bad_arguments():
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    attn = SwinWindowAttention((8, 16), (4, 8), (2, 4), (0, 1), 2, 32)
    lib = C.load_library()
    assert lib.swin_attn_plan_set_debug(attn.plan.handle, 0, 0) == C.SWIN_ERR_INVALID_ARG
    assert lib.swin_attn_plan_set_debug(attn.plan.handle, 10, 2) == C.SWIN_ERR_INVALID_ARG
    assert lib.swin_attn_plan_set_debug(None, 10, 0) == C.SWIN_ERR_INVALID_ARG


def test_forced_wait_timeout_in_fused_block_is_reported_and_recoverable():
    """The fused block kernel (LayerNorm + QKV, SW-MSA, out-projection): every
    thread waits on the barrier nothing arrives at, the CTA agrees on the
    failure, drains the weight copies in flight, frees TMEM and exits; the
    plan then runs the block normally and meets the block oracle."""
    from oracle import block as oblock
    from shifted_window_attention_cyclic_gb300 import swin_attn as C
    from shifted_window_attention_cyclic_gb300.functional import SwinWindowAttention
    wl = workloads.custom((13, 27), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16", (0.3, 0.3), seed_index=93)
    xb = workloads.generate_block(wl)
    attn = SwinWindowAttention(wl.grid, wl.window, wl.shift, wl.periodic, wl.heads, wl.head_dim, wl.batch,
                               wl.dtype, wl.has_land, "tc")
    dev = torch.device("cuda", 0)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf = lambda a: f32(a).to(torch.bfloat16)
    args = (bf(xb["x"]), f32(xb["gamma"]), f32(xb["beta"]), bf(xb["w_qkv"]), f32(xb["b_qkv"]), bf(xb["w_o"]),
            f32(xb["b_o"]), f32(xb["bias"]), f32(xb["land"]))
    C.swin_attn_plan_set_debug(attn.plan, 5_000_000, 1)  # 5 ms limit, forced wait
    attn.block_forward(*args)
    assert C.swin_attn_status(attn.plan) == C.SWIN_ERR_TIMEOUT
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK  # status word was cleared
    C.swin_attn_plan_set_debug(attn.plan, 1_000_000_000, 0)
    y = attn.block_forward(*args)
    torch.cuda.synchronize()
    assert C.swin_attn_status(attn.plan) == C.SWIN_OK
    ref, _ = oblock.block_fwd(problem_of(wl), xb["x"], xb["gamma"], xb["beta"], 1e-5, xb["w_qkv"], xb["b_qkv"],
                              xb["w_o"], xb["b_o"], xb["bias"], xb["land"])
    got = host(y)
    assert np.isfinite(got).all()
    assert (np.abs(got - ref) <= 2e-2 + 2.0 ** -8 * np.abs(ref)).all()
