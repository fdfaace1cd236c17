"""Argument checks of the torch wrapper, on the CPU: the tensors the parity
tests and smoke() build pass them, and each kind of caller mistake that would
make the library read or write past a buffer is refused before any call."""
import pytest

torch = pytest.importorskip("torch")

from oracle import Problem  # noqa: E402
from shifted_window_attention_cyclic_gb300 import workloads  # noqa: E402
from shifted_window_attention_cyclic_gb300.functional import check_call, check_tensor  # noqa: E402
from tests.parity_util import to_device  # noqa: E402
from tests.test_gpu_parity import SWEEP  # noqa: E402

CPU = torch.device("cpu")
TDT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _shapes(wl):
    pb = Problem(grid=wl.grid, window=wl.window, shift=wl.shift, periodic=wl.periodic, heads=wl.heads,
                 head_dim=wl.head_dim, batch=wl.batch, has_land=wl.has_land)
    shape = (wl.batch,) + tuple(wl.grid) + (wl.heads * wl.head_dim,)
    return shape, (wl.batch, wl.heads) + tuple(wl.grid), (pb.bias_rows, wl.heads)


def _cases():
    yield workloads.WORKLOADS["tiny_fp32"]
    for i, c in enumerate(SWEEP):
        grid, window, shift, periodic, heads, hd, batch, dtype, land_p = c
        yield workloads.custom(grid, window, shift, periodic, heads, hd, batch, dtype, land_p, seed_index=300 + i)


@pytest.mark.parametrize("wl", list(_cases()), ids=lambda wl: "x".join(map(str, wl.grid)))
def test_test_inputs_pass_the_checks(wl):
    t = to_device(workloads.generate(wl), wl, CPU)
    shape, lse_shape, bias_shape = _shapes(wl)
    lse = torch.zeros(lse_shape, dtype=torch.float32)
    dbias = torch.zeros(bias_shape, dtype=torch.float32)
    outs = {n: torch.empty(shape, dtype=TDT[wl.dtype]) for n in ("o", "dq", "dk", "dv")}
    fwd = dict(q=t["q"], k=t["k"], v=t["v"], bias=t["bias"], land=t["land"], o=outs["o"], lse=lse)
    check_call(fwd, shape, lse_shape, bias_shape, TDT[wl.dtype], CPU, wl.has_land)
    bwd = dict(q=t["q"], k=t["k"], v=t["v"], dout=t["dout"], lse=lse, bias=t["bias"], land=t["land"],
               dq=outs["dq"], dk=outs["dk"], dv=outs["dv"], dbias=dbias)
    check_call(bwd, shape, lse_shape, bias_shape, TDT[wl.dtype], CPU, wl.has_land)


def test_each_mistake_is_refused():
    shape, lse_shape, bias_shape = (1, 8, 16, 64), (1, 2, 8, 16), (105, 2)
    good = dict(q=torch.zeros(shape, dtype=torch.bfloat16), bias=torch.zeros(bias_shape),
                lse=torch.zeros(lse_shape), land=torch.zeros(shape[:-1], dtype=torch.uint8))

    def refused(match, **change):
        args = dict(good, **change)
        with pytest.raises(ValueError, match=match):
            check_call(args, shape, lse_shape, bias_shape, torch.bfloat16, CPU, True)

    check_call(good, shape, lse_shape, bias_shape, torch.bfloat16, CPU, True)
    refused("dtype", q=torch.zeros(shape, dtype=torch.float32))
    refused("shape", q=torch.zeros((1, 8, 16, 32), dtype=torch.bfloat16))
    refused("contiguous", q=torch.zeros((1, 16, 8, 64), dtype=torch.bfloat16).transpose(1, 2))
    flat = torch.zeros(1 + 8 * 16 * 64, dtype=torch.bfloat16)
    refused("aligned", q=flat[1:].view(shape))
    refused("dtype", bias=torch.zeros(bias_shape, dtype=torch.float64))
    refused("shape", bias=torch.zeros((104, 2)))
    refused("shape", lse=torch.zeros((1, 8, 16)))
    refused("dtype", land=torch.zeros(shape[:-1], dtype=torch.bool))
    refused("land mask", land=None)
    refused("torch.Tensor", q=[0.0])
    with pytest.raises(ValueError, match="on cpu"):
        check_tensor("q", good["q"], shape, torch.bfloat16, torch.device("cuda", 0))
    # a plan without land ignores a land argument
    check_call(dict(good, land=torch.zeros(3)), shape, lse_shape, bias_shape, torch.bfloat16, CPU, False)
