"""Host-side tests of the C ABI that need no GPU: the library builds and loads,
exports every entry point include/moe_mxfp4.h declares, plans workspaces
consistently, and rejects bad arguments with the documented status codes before
touching a device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_mxfp4_gb300 import build

    build.build()
    import mixture_experts_mxfp4_gb300 as moe

    return moe.load_library()


def _declared_symbols():
    syms = set()
    inc = os.path.join(ROOT, "include")
    for name in os.listdir(inc):
        if not name.endswith(".h"):
            continue
        text = open(os.path.join(inc, name)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(moe_mxfp4_\w+)\s*\(", text):
            syms.add(m.group(1))
    return sorted(syms)


def test_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert "moe_mxfp4_forward" in declared
    for s in declared:
        assert hasattr(lib, s), f"{s} declared in include/ but not exported"
    import mixture_experts_mxfp4_gb300 as moe

    assert sorted(moe.EXPORTS) == sorted(declared)


def test_status_strings(lib):
    import mixture_experts_mxfp4_gb300 as moe

    for code in moe.STATUS:
        assert lib.moe_mxfp4_status_string(code)
    assert b"sm_103a" in lib.moe_mxfp4_version()


@pytest.mark.parametrize("shape", [(16, 256, 128, 9, 3), (16, 7168, 256, 257, 9),
                                   (128, 7168, 256, 257, 9), (512, 7168, 2048, 33, 9),
                                   (4096, 7168, 256, 257, 9), (1, 128, 128, 1, 1)])
def test_plan_layout(lib, shape):
    import mixture_experts_mxfp4_gb300 as moe
    import oracle

    T, D, I, E, K = shape
    pl = moe.get_plan(*shape)
    assert pl.block_m == 16
    assert pl.cap == oracle.route_capacity(T, K, E, 16)
    assert pl.tile_rows % 16 == 0 and 16 <= pl.tile_rows <= 128
    assert pl.a1s_stride % 16 == 0 and pl.a1s_stride >= D // 32
    assert pl.a2s_stride % 16 == 0 and pl.a2s_stride >= I // 32
    R = T * K
    expect = {"sorted_ids": pl.cap * 4, "sorted_w": pl.cap * 4, "route_pos": R * 4,
              "a1q": pl.cap * D // 2, "a2q": pl.cap * I // 2, "P": R * D * 4,
              "seg_start": (E + 1) * 4}
    prev_end = 0
    for i, name in enumerate(moe.REGIONS):
        off, nb = pl.region(name)
        assert off % 256 == 0
        assert off >= prev_end
        prev_end = off + nb
        if name in expect:
            assert nb == expect[name], name
    assert pl.workspace_bytes >= prev_end
    assert moe.workspace_size(*shape) == pl.workspace_bytes


def test_validation_codes_without_device(lib):
    import mixture_experts_mxfp4_gb300 as moe

    good = 1 << 20  # a fake, 16-byte aligned address; never dereferenced on these paths
    args = [good] * 8

    def call(T=16, D=256, I=128, E=9, K=3, ptrs=None):
        p = ptrs or args
        return moe.forward_ptr(*p, T, D, I, E, K, 0)

    assert call(T=-1) == 1
    assert call(E=0) == 1
    assert call(E=1025) == 1
    assert call(K=0) == 1
    assert call(K=17) == 1
    assert call(D=0) == 1
    assert call(D=320) == 2      # d_model not a multiple of 128
    assert call(I=96) == 2       # d_inter not a multiple of 64
    assert call(D=1000) == 2
    assert call(T=0) == 0        # empty input: nothing to do
    nulls = list(args)
    nulls[3] = 0
    assert call(ptrs=nulls) == 1
    mis = list(args)
    mis[0] = good + 8
    assert call(ptrs=mis) == 3
    assert moe.workspace_size(16, 320, 128, 9, 3) == 0
    with pytest.raises(moe.MoeError):
        moe.get_plan(16, 256, 100, 9, 3)
    # workspace registration checks alignment before any device call
    assert lib.moe_mxfp4_set_workspace(ctypes.c_void_p(good + 64), 1024) == 3


def test_padded_validation_codes_without_device(lib):
    import mixture_experts_mxfp4_gb300 as moe

    good = 1 << 20
    args = [good] * 8

    def call(T=16, D=224, I=96, Dp=256, Ip=128, E=9, K=3):
        return moe.forward_padded_ptr(*args, T, D, I, Dp, Ip, E, K, 0)

    assert call(D=200) == 2       # logical size not a multiple of 32
    assert call(I=16) == 2        # below one scale block
    assert call(D=288) == 1       # logical size above the stored one
    assert call(Ip=192) == 2      # padded stored size not 128, 256 or a multiple of 512
    assert call(Ip=160) == 2      # stored size not a multiple of 64
    assert call(T=0) == 0
    assert moe.call_launches(16, 255, 128, 9, 3) == -1


@pytest.mark.parametrize("shape,run", [((16, 2944, 384, 16, 4), (3072, 512)),
                                       ((200, 1152, 768, 8, 3), (1536, 1024)),
                                       ((16, 384, 192, 9, 3), (512, 256)),
                                       ((8, 128, 64, 4, 2), (128, 128)),
                                       ((16, 7168, 256, 257, 9), (7168, 256))])
def test_run_widths_in_the_plan(lib, shape, run):
    """Widths that are not 128, 256 or a multiple of 512 run at the next such width:
    the activation regions use it, and the weight scales get a region of rows of
    the run widths' scale bytes (none for widths run as they are)."""
    import mixture_experts_mxfp4_gb300 as moe

    T, D, I, E, K = shape
    Dr, Ir = run
    pl = moe.get_plan(*shape)
    assert (pl.d_model_run, pl.d_inter_run) == (Dr, Ir)
    assert pl.region("a1q")[1] == pl.cap * Dr // 2 and pl.region("a2q")[1] == pl.cap * Ir // 2
    assert pl.region("P")[1] == T * K * Dr * 4
    assert pl.a1s_stride >= Dr // 32 and pl.a2s_stride >= Ir // 32
    w13s = E * 2 * I * (Dr // 32)
    expect = 0 if (Dr, Ir) == (D, I) else (w13s + 255) // 256 * 256 + E * D * (Ir // 32)
    assert pl.region("wscale")[1] == expect
    assert moe.workspace_size(*shape) == pl.workspace_bytes
    c = moe.gemm_config(*shape)
    assert Dr % c.stage1_k == 0 and Ir % c.stage2_k == 0
    # the bf16-activation forward takes only widths it runs as they are
    if (Dr, Ir) != (D, I):
        with pytest.raises(moe.MoeError):
            moe.get_plan_w4a16(*shape)
        assert moe.load_library().moe_mxfp4_workspace_size_w4a16(*shape) == 0


def test_topk_sum_validation_without_device(lib):
    import mixture_experts_mxfp4_gb300 as moe

    good = 1 << 20
    assert moe.topk_sum_ptr(good, good, good, 16, 256, 0) == 1      # topk 0
    assert moe.topk_sum_ptr(good, good, good, 16, 256, 17) == 1     # topk above 16
    assert moe.topk_sum_ptr(good, good, good, -1, 256, 3) == 1      # T < 0
    assert moe.topk_sum_ptr(good, good, good, 16, 200, 3) == 2      # d_model not a multiple of 128
    assert moe.topk_sum_ptr(good, good, good, 0, 256, 3) == 0       # empty: nothing enqueued
    assert moe.topk_sum_ptr(good, 0, good, 16, 256, 3) == 1         # null pointer
    assert moe.topk_sum_ptr(good + 4, good, good, 16, 256, 3) == 3  # misaligned


def test_w4a16_entry_and_plan_without_device(lib):
    import mixture_experts_mxfp4_gb300 as moe

    good = 1 << 20
    args = [good] * 8
    assert moe.forward_w4a16_ptr(*args, 16, 384, 128, 9, 3, 0) == 2   # unsupported d_model
    assert moe.forward_w4a16_ptr(*args, 0, 256, 128, 9, 3, 0) == 0    # empty batch
    pl = moe.get_plan_w4a16(16, 7168, 256, 257, 9)
    ref = moe.get_plan(16, 7168, 256, 257, 9)
    assert pl.bf16_act == 1 and ref.bf16_act == 0
    assert pl.region("a1b")[1] == pl.cap * 7168 * 2 and pl.region("a2b")[1] == pl.cap * 256 * 2
    assert pl.region("a1q")[1] == 0 and ref.region("a1b")[1] == 0
    assert moe.load_library().moe_mxfp4_workspace_size_w4a16(16, 7168, 256, 257, 9) == pl.workspace_bytes


def test_pointer_kind_without_device(lib):
    """Null and ordinary host memory are never usable as forward buffers; with no
    GPU present every query answers -1 (and leaves no error behind)."""
    assert lib.moe_mxfp4_pointer_kind(None) == -1
    buf = ctypes.create_string_buffer(64)
    assert lib.moe_mxfp4_pointer_kind(ctypes.cast(buf, ctypes.c_void_p)) == -1
    assert lib.moe_mxfp4_pointer_kind(ctypes.cast(buf, ctypes.c_void_p)) == -1


@pytest.mark.parametrize("shape,rows", [
    ((16, 7168, 256, 257, 9), 16),    # decode: 0.56 routes per expert
    ((128, 7168, 256, 257, 9), 16),   # decode batch: 4.5
    ((64, 256, 128, 9, 3), 32),       # 21.3
    ((64, 256, 128, 5, 3), 64),       # 38.4
    ((512, 7168, 2048, 33, 9), 128),  # dense shard: 140
    ((4096, 7168, 256, 257, 9), 128), # prefill: 143 on average
])
def test_route_tile_width_rule(lib, shape, rows):
    """Route-tile width: the smallest of 16/32/64/128 rows above the expected
    routes per expert (T*topk/E <= 8, 24, 48, else 128)."""
    import mixture_experts_mxfp4_gb300 as moe

    assert moe.get_plan(*shape).tile_rows == rows


def test_tuning_override_without_device(lib):
    """The tuning override forces the route-tile width of the plan (the workspace
    size does not change) and rejects values outside the documented set."""
    import mixture_experts_mxfp4_gb300 as moe

    shape = (128, 7168, 256, 257, 9)
    size = moe.workspace_size(*shape)
    try:
        for rows in (16, 32, 64, 128):
            for copies in (0, 1, 2, 3, 4):
                moe.set_tuning(rows, copies)
                assert moe.get_plan(*shape).tile_rows == rows
                assert moe.workspace_size(*shape) == size
        for bad in ((8, 0), (48, 0), (256, 0), (-1, 0), (0, 5), (0, -1)):
            assert lib.moe_mxfp4_set_tuning(*bad) == 1
    finally:
        moe.set_tuning(0, 0)
    assert moe.get_plan(*shape).tile_rows == 16


def test_nvtx_switch_without_device(lib):
    """The NVTX switch takes 0 and 1 and rejects anything else (no device needed:
    the ranges are host-side)."""
    import mixture_experts_mxfp4_gb300 as moe

    try:
        moe.set_nvtx(True)
        moe.set_nvtx(False)
        for bad in (-1, 2, 7):
            assert lib.moe_mxfp4_set_nvtx(bad) == 1
    finally:
        moe.set_nvtx(False)


def test_checked_build_without_device(lib):
    """The bounds-checked variant builds from the same sources with MOE_CHECKED=1,
    loads without a GPU, exports every declared entry point and says what it is."""
    from mixture_experts_mxfp4_gb300 import build

    path = build.build(checked=True)
    clib = ctypes.CDLL(path)
    for s in _declared_symbols():
        assert hasattr(clib, s), s
    clib.moe_mxfp4_version.restype = ctypes.c_char_p
    assert b"bounds-checked" in clib.moe_mxfp4_version()
    assert b"bounds-checked" not in lib.moe_mxfp4_version()
