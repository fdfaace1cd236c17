"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/swin_attn.h, rejects bad descriptors before touching CUDA,
and its TERRA Eq. (4) window split and Eq. (3) padding match the pages'
worked examples."""
import ctypes
import os

import pytest

from shifted_window_attention_cyclic_gb300 import swin_attn as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return C.load_library()


def test_exports_every_declared_symbol(lib):
    names = C.declared_symbols()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), name


def test_strerror_covers_codes(lib):
    for code in range(0, -8, -1):
        assert C.strerror(code) != "unknown status"
    assert C.strerror(-99) == "unknown status"


def test_eq4_window_ranges_match_worked_examples(lib):
    with open(os.path.join(GOLDEN, "window_ranges_eq4.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, vals = line.split(":")
            M, P = (int(x) for x in head.split())
            want = [int(x) for x in vals.split()]
            got = []
            for r in range(P):
                got += list(C.swin_attn_window_range(M, P, r))
            assert got == want
    # ten windows on four ranks: two ranks get three, two get two (TERRA Sec. V.B)
    sizes = sorted(R - L for L, R in (C.swin_attn_window_range(10, 4, r) for r in range(4)))
    assert sizes == [2, 2, 3, 3]


def test_eq4_ranges_partition_and_balance(lib):
    for M, P in [(0, 3), (1, 5), (45, 4), (73728, 152), (1000003, 304)]:
        prev = 0
        sizes = []
        for r in range(P):
            L, R = C.swin_attn_window_range(M, P, r)
            assert L == prev
            prev = R
            sizes.append(R - L)
        assert prev == M and max(sizes) - min(sizes) <= 1


def test_window_range_rejects_bad_arguments(lib):
    L, R = ctypes.c_int64(), ctypes.c_int64()
    for args in [(-1, 4, 0), (10, 0, 0), (10, 4, 4), (10, 4, -1)]:
        assert lib.swin_attn_window_range(*args, ctypes.byref(L), ctypes.byref(R)) == C.SWIN_ERR_INVALID_ARG


BAD_DESCS = [
    (dict(grid=(16, 32), window=(4, 8), shift=(4, 0), periodic=(0, 1), heads=2, head_dim=16), C.SWIN_ERR_INVALID_ARG),
    (dict(grid=(16, 32), window=(4, 8), shift=(-1, 0), periodic=(0, 1), heads=2, head_dim=16), C.SWIN_ERR_INVALID_ARG),
    (dict(grid=(16, 32), window=(0, 8), shift=(0, 0), periodic=(0, 1), heads=2, head_dim=16), C.SWIN_ERR_INVALID_ARG),
    (dict(grid=(2, 32), window=(4, 8), shift=(3, 0), periodic=(0, 1), heads=2, head_dim=16), C.SWIN_ERR_INVALID_ARG),
    (dict(grid=(16, 32), window=(4, 8), shift=(2, 4), periodic=(0, 2), heads=2, head_dim=16), C.SWIN_ERR_INVALID_ARG),
    (dict(grid=(16, 32), window=(4, 8), shift=(2, 4), periodic=(0, 1), heads=0, head_dim=16), C.SWIN_ERR_INVALID_ARG),
    (dict(grid=(16, 32), window=(16, 16), shift=(2, 4), periodic=(0, 1), heads=2, head_dim=16), C.SWIN_ERR_UNSUPPORTED),
    (dict(grid=(16, 32), window=(4, 8), shift=(2, 4), periodic=(0, 1), heads=2, head_dim=64), C.SWIN_ERR_UNSUPPORTED),
    (dict(grid=(16, 32), window=(4, 8), shift=(2, 4), periodic=(0, 1), heads=2, head_dim=24), C.SWIN_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("kw,code", BAD_DESCS)
def test_plan_rejects_bad_descriptor_without_cuda(lib, kw, code):
    d = C.make_desc(**kw)
    h = ctypes.c_void_p()
    assert lib.swin_attn_plan(ctypes.byref(d), ctypes.byref(h)) == code
    assert not h.value


def test_plan_rejects_bad_dtype_impl_batch_ndim(lib):
    h = ctypes.c_void_p()
    base = dict(grid=(16, 32), window=(4, 8), shift=(2, 4), periodic=(0, 1), heads=2, head_dim=16)
    d = C.make_desc(**base)
    d.dtype = 7
    assert lib.swin_attn_plan(ctypes.byref(d), ctypes.byref(h)) == C.SWIN_ERR_UNSUPPORTED
    d = C.make_desc(**base)
    d.impl = 9
    assert lib.swin_attn_plan(ctypes.byref(d), ctypes.byref(h)) == C.SWIN_ERR_INVALID_ARG
    d = C.make_desc(**base)
    d.batch = 0
    assert lib.swin_attn_plan(ctypes.byref(d), ctypes.byref(h)) == C.SWIN_ERR_INVALID_ARG
    d = C.make_desc(**base)
    d.ndim = 4
    assert lib.swin_attn_plan(ctypes.byref(d), ctypes.byref(h)) == C.SWIN_ERR_INVALID_ARG
    # the kernels address the [B*T, C] row view with 32-bit row numbers and
    # keep the batch in an int: B*T >= 2^31 (or B > INT32_MAX) is refused at plan time
    d = C.make_desc(grid=(32768, 32768), window=(4, 8), shift=(2, 4), periodic=(0, 1), heads=1, head_dim=16,
                    batch=2)
    assert lib.swin_attn_plan(ctypes.byref(d), ctypes.byref(h)) == C.SWIN_ERR_UNSUPPORTED
    d = C.make_desc(**base)
    d.batch = 2 ** 31
    assert lib.swin_attn_plan(ctypes.byref(d), ctypes.byref(h)) == C.SWIN_ERR_UNSUPPORTED
    assert not h.value
    assert lib.swin_attn_plan(None, ctypes.byref(h)) == C.SWIN_ERR_INVALID_ARG
    assert lib.swin_attn_plan(ctypes.byref(d), None) == C.SWIN_ERR_INVALID_ARG


def test_null_plan_is_rejected(lib):
    assert lib.swin_attn_fwd(None, *([None] * 8)) == C.SWIN_ERR_INVALID_ARG
    assert lib.swin_attn_bwd(None, *([None] * 12), 0, None) == C.SWIN_ERR_INVALID_ARG
    assert lib.swin_attn_status(None, None) == C.SWIN_ERR_INVALID_ARG
    assert lib.swin_attn_workspace_bytes(None) == 0
    lib.swin_attn_plan_destroy(None)


def test_eq3_padding_matches_worked_example(lib):
    with open(os.path.join(GOLDEN, "padding_eq3.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, vals = line.split(":")
            H, W, stride, w, m, n = (int(x) for x in head.split())
            mh, mw, pct = vals.split()
            Hp = C.swin_attn_fixed_padded_extent(H, stride, w, m)
            Wp = C.swin_attn_fixed_padded_extent(W, stride, w, n)
            assert (Hp // (stride * w), Wp // (stride * w)) == (int(mh), int(mw))
            assert Hp % (stride * w * m) == 0 and Wp % (stride * w * n) == 0
            assert round(100.0 * (Hp * Wp / (H * W) - 1.0), 1) == float(pct)


def test_eq3_padding_is_the_least_multiple(lib):
    # Fig. 6 of TERRA Sec. V.A: a 9 x 5 window grid on a 2 x 2 mesh pads to
    # 10 x 6 windows (extents counted in windows: stride = window = 1)
    assert C.swin_attn_fixed_padded_extent(9, 1, 1, 2) == 10
    assert C.swin_attn_fixed_padded_extent(5, 1, 1, 2) == 6
    for extent in (1, 7, 8, 9, 255, 256, 257, 4320):
        for stride, w, r in ((1, 1, 1), (8, 8, 1), (8, 128, 4), (4, 12, 3)):
            q = stride * w * r
            got = C.swin_attn_fixed_padded_extent(extent, stride, w, r)
            assert got % q == 0 and extent <= got < extent + q


def test_eq3_padding_rejects_bad_arguments(lib):
    bad = [(0, 8, 8, 1), (10, 0, 8, 1), (10, 8, 0, 1), (10, 8, 8, 0), (-1, 8, 8, 1),
           (2 ** 62, 2 ** 31, 2 ** 31, 2), (2 ** 63 - 1, 1, 1, 2)]
    out = ctypes.c_int64(-7)
    for args in bad:
        assert lib.swin_attn_fixed_padded_extent(*args, ctypes.byref(out)) == C.SWIN_ERR_INVALID_ARG
        assert out.value == -7
    assert lib.swin_attn_fixed_padded_extent(10, 8, 8, 1, None) == C.SWIN_ERR_INVALID_ARG


def test_missing_library_raises_no_fallback(monkeypatch):
    # without the CUDA library every entry point raises; nothing falls back
    monkeypatch.setattr(C, "_lib", None)
    monkeypatch.setattr(C, "LIB_PATH", os.path.join(GOLDEN, "no_such_libswin_attn.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        C.load_library()
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        C.swin_attn_window_range(10, 4, 0)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        C.swin_attn_plan(C.make_desc((8, 16), (4, 8), (2, 4), (0, 1), 2, 32, 1, "bf16"))


def test_binding_refuses_misaligned_lse_land_and_activations(lib):
    # the tensor-core kernels read four LSE values (16 bytes) and four land
    # bytes with one load each; the binding refuses pointers off those
    # boundaries before the call (CPU tensors: nothing reaches a device)
    import types
    torch = pytest.importorskip("torch")
    plan = types.SimpleNamespace(handle=None)
    f32 = torch.zeros(64, dtype=torch.float32)
    u8 = torch.zeros(64, dtype=torch.uint8)
    good = f32[:16]
    with pytest.raises(C.SwinAttnError, match="lse not 16-byte aligned"):
        C.swin_attn_fwd(plan, good, good, good, None, None, good, f32[1:17])
    with pytest.raises(C.SwinAttnError, match="land not 4-byte aligned"):
        C.swin_attn_fwd(plan, good, good, good, None, u8[1:], good, good)
    with pytest.raises(C.SwinAttnError, match="q not 16-byte aligned"):
        C.swin_attn_bwd(plan, f32[2:18], good, good, good, good, None, None, good, good, good, None, None)
    with pytest.raises(C.SwinAttnError, match="land not 4-byte aligned"):
        C.swin_attn_bwd(plan, good, good, good, good, good, None, u8[2:], good, good, good, None, None)
    with pytest.raises(C.SwinAttnError, match="lse not 16-byte aligned"):
        C.swin_attn_bwd_noalloc(plan, good, good, good, good, f32[3:19], None, None, good, good, good, None)
