"""GPU parity: the CUDA library (called through the C ABI) against the CPU oracle.

Bars (from the method's acceptance criteria):
  * routing arrays, tile list and the quantised hidden rows: bit-exact;
  * requantised intermediate (a2 codes/scales): at most 0.1% of the codes and at
    most 0.1% of the 32-element blocks' scale bytes differ; every element within
    one step of the e2m1 grid (signed grid index, both codes put on the finer
    block scale; scale bytes at most one apart), as where fp32 accumulation
    order flips a rounding tie;
  * output: for every token row, max |gpu - oracle| <= 2e-2 * rms(oracle row),
    and exactly zero where the oracle row is zero.
Every workload compares every token; all inputs are seeded synthetic tensors
(workloads module).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

ROW_TOL = 2e-2
CODE_FRAC = 1e-3


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_mxfp4_gb300 import build

    build.build()
    import mixture_experts_mxfp4_gb300 as m

    m.load_library()
    return m


@pytest.fixture(params=[0, 1], ids=["separate_kernels", "single_launch"])
def launch_mode(request, moe):
    """Both launch modes: routing and quantisation as their own kernels, or inside
    the GEMM kernel (single launch; results must be identical)."""
    moe.set_single_launch(request.param)
    yield request.param
    moe.set_single_launch(2)


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def _unpack(p):
    p = np.asarray(p, np.uint8)
    return np.stack([p & 15, p >> 4], axis=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)


_E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def _deq(codes, scales, n):
    v = _E2M1[_unpack(codes)]
    return v * np.repeat(np.ldexp(1.0, scales[..., : n // 32].astype(np.int64) - 127), 32, axis=-1)


def run_gpu(moe, inp, w):
    dev = torch.device("cuda")
    m = moe.MoeMXFP4(w.T, w.D, w.I, w.E, w.K)
    t = {k: v.to(dev) for k, v in inp.items()}
    out = m.forward(t["hidden"], t["w13"], t["w13_scale"], t["w2"], t["w2_scale"],
                    t["topk_ids"], t["topk_weights"])
    torch.cuda.synchronize()
    assert m.device_status() == 0
    return m, t, out


def ws_arrays(m, w):
    pl = m.plan
    R = w.R
    cap = pl.cap
    get = lambda name, dt, shape: m.region(name, dt, shape).cpu().numpy()
    return {
        "sorted_ids": get("sorted_ids", torch.int32, (cap,)),
        "sorted_w": get("sorted_w", torch.float32, (cap,)),
        "block_expert": get("block_expert", torch.int32, (cap // 16,)),
        "seg_start": get("seg_start", torch.int32, (w.E + 1,)),
        "route_pos": get("route_pos", torch.int32, (R,)),
        "num_valid": get("num_valid", torch.int32, (4,)),
        "tiles": get("tiles", torch.int32, (pl.max_tiles, 4)),
        "a1q": get("a1q", torch.uint8, (cap, w.D // 2)),
        "a1s": get("a1s", torch.uint8, (cap, pl.a1s_stride)),
        "a2q": get("a2q", torch.uint8, (cap, w.I // 2)),
        "a2s": get("a2s", torch.uint8, (cap, pl.a2s_stride)),
    }


def check_routing(ws, ref, w, tile_rows):
    n = int(ref["num_valid"][0])
    np.testing.assert_array_equal(ws["num_valid"][:2], ref["num_valid"])
    np.testing.assert_array_equal(ws["sorted_ids"], ref["sorted_ids"])
    np.testing.assert_array_equal(ws["sorted_w"].view(np.uint32), ref["sorted_w"].view(np.uint32))
    np.testing.assert_array_equal(ws["block_expert"], ref["block_expert"])
    np.testing.assert_array_equal(ws["seg_start"], ref["seg_start"])
    np.testing.assert_array_equal(ws["route_pos"], ref["route_pos"])
    # tile list: each expert's padded segment cut into tile_rows pieces, in order
    tiles = []
    ss = ref["seg_start"]
    for e in range(w.E):
        for off in range(0, ss[e + 1] - ss[e], tile_rows):
            tiles.append((e, ss[e] + off, min(tile_rows, ss[e + 1] - ss[e] - off), 0))
    assert ws["num_valid"][2] == len(tiles)
    np.testing.assert_array_equal(ws["tiles"][: len(tiles)], np.array(tiles, np.int32).reshape(-1, 4))
    return n


def _valid_slots(routing, w, tokens=None):
    """Sorted slots holding a valid route (and their route ids), optionally only
    those of the given tokens."""
    n = int(routing["num_valid"][0])
    sids = routing["sorted_ids"][:n]
    slots = np.nonzero(sids < w.R)[0]
    routes = sids[slots].astype(np.int64)
    if tokens is not None:
        keep = np.isin(routes // w.K, np.asarray(tokens, np.int64))
        slots, routes = slots[keep], routes[keep]
    return slots, routes


def check_a1(ws, ref_fw, routing, w, tokens=None):
    slots, routes = _valid_slots(routing, w, tokens)
    assert len(slots) > 0
    toks = routes // w.K
    np.testing.assert_array_equal(ws["a1q"][slots][:, : w.D // 2], ref_fw["a1q"][toks], err_msg="a1q")
    np.testing.assert_array_equal(ws["a1s"][slots][:, : w.D // 32], ref_fw["a1s"][toks], err_msg="a1s")


# e2m1 magnitudes continued past 6 by the same two points per binade: a code on a
# block scale one above the other side's lands here when put on the finer scale
_GRID_EXT = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, 8, 12, 16, 24])


def _signed_grid_index(codes, sbytes, s_fine):
    """Signed index of each element on the e2m1 grid of scale s_fine (<= sbytes)."""
    mag = np.abs(_E2M1[codes]) * np.ldexp(1.0, (sbytes - s_fine).astype(np.int64))
    idx = np.searchsorted(_GRID_EXT, mag)
    assert (idx < len(_GRID_EXT)).all() and (_GRID_EXT[np.minimum(idx, len(_GRID_EXT) - 1)] == mag).all()
    return np.where(codes >= 8, -idx, idx)


def check_a2(ws, ref_fw, routing, w, tokens=None):
    """Requantised intermediate against the oracle's: at most one e2m1 grid step
    per element, at most CODE_FRAC of the codes and of the block scales differ."""
    slots, routes = _valid_slots(routing, w, tokens)
    nb = w.I // 32
    gq, gs = ws["a2q"][slots][:, : w.I // 2], ws["a2s"][slots][:, :nb].astype(np.int64)
    oq, os_ = ref_fw["a2q"][routes], ref_fw["a2s"][routes].astype(np.int64)
    cg, co = _unpack(gq).astype(np.int64), _unpack(oq).astype(np.int64)
    assert (np.abs(gs - os_) <= 1).all(), "a2 scale bytes more than one apart"
    sg, so = np.repeat(gs, 32, axis=1), np.repeat(os_, 32, axis=1)
    fine = np.minimum(sg, so)
    step = np.abs(_signed_grid_index(cg, sg, fine) - _signed_grid_index(co, so, fine))
    bad = np.argwhere(step > 1)
    assert len(bad) == 0, f"a2 route {routes[bad[0][0]]} element {bad[0][1]}: more than one step"
    diff = int(((cg != co) | (sg != so)).sum())
    sdiff = int((gs != os_).sum())
    assert diff <= CODE_FRAC * cg.size, f"{diff} of {cg.size} a2 codes differ"
    assert sdiff <= CODE_FRAC * gs.size, f"{sdiff} of {gs.size} a2 block scales differ"
    return diff, cg.size


def check_out(out_gpu, ref_fw, tokens=None):
    g = out_gpu.float().cpu().numpy()
    o = oracle.bf16_bits_to_f32(ref_fw["out_bf16"])
    rows = range(g.shape[0]) if tokens is None else tokens
    worst = 0.0
    for t in rows:
        rms = float(np.sqrt(np.mean(o[t].astype(np.float64) ** 2)))
        err = float(np.max(np.abs(g[t].astype(np.float64) - o[t])))
        if rms == 0.0:
            assert err == 0.0, f"row {t}: oracle row is zero, gpu max |x| = {err}"
            continue
        worst = max(worst, err / rms)
        assert err <= ROW_TOL * rms, f"row {t}: max err {err} > {ROW_TOL} * rms {rms}"
    return worst


def full_check(moe, w, inp, tokens=None):
    m, t, out = run_gpu(moe, inp, w)
    npi = workloads.to_numpy(inp)
    routing = oracle.route(npi["topk_ids"], npi["topk_weights"], w.E, 16, cap=m.plan.cap)
    ref = oracle.forward(**npi, tokens=tokens, threads=_threads(), want_h=False)
    ws = ws_arrays(m, w)
    check_routing(ws, routing, w, m.plan.tile_rows)
    check_a1(ws, ref, routing, w, tokens)
    check_a2(ws, ref, routing, w, tokens)
    worst = check_out(out, ref, tokens)
    return m, t, out, worst


# ------------------------------------------------------------------ workloads

def test_tiny_workload(moe, launch_mode):
    w = workloads.WORKLOADS[workloads.TINY]
    full_check(moe, w, workloads.make_inputs(w))


def test_decode_t16_full(moe, launch_mode):
    w = workloads.WORKLOADS[workloads.DECODE_T16]
    full_check(moe, w, workloads.make_inputs(w))


def test_decode_t128_full(moe, launch_mode):
    w = workloads.WORKLOADS["decode_T128_D7168_I256_E257_K9"]
    full_check(moe, w, workloads.make_inputs(w))


def test_dense_shard_t512_full(moe):
    w = workloads.WORKLOADS["dense_T512_D7168_I2048_E33_K9"]
    full_check(moe, w, workloads.make_inputs(w))


def test_prefill_zipf_t4096_full(moe):
    w = workloads.WORKLOADS["prefill_zipf_T4096_D7168_I256_E257_K9"]
    full_check(moe, w, workloads.make_inputs(w))


# ------------------------------------------------------------------ edge cases

def _small(T=16, D=256, I=128, E=9, K=3, seed=0):
    w = workloads.custom(T, D, I, E, K)
    return w, workloads.make_inputs(w, seed=seed)


def test_single_token(moe, launch_mode):
    w, inp = _small(T=1)
    full_check(moe, w, inp)


def test_all_routes_on_one_expert(moe, launch_mode):
    w, inp = _small(T=40, E=9, K=1)
    inp["topk_ids"][:] = 4
    full_check(moe, w, inp)


def test_exactly_full_blocks_and_duplicates(moe, launch_mode):
    # expert 2 receives exactly 32 routes (two full blocks); token 0 repeats an expert
    w, inp = _small(T=32, E=5, K=2)
    ids = inp["topk_ids"]
    ids[:, 0] = 2
    ids[:, 1] = torch.arange(32, dtype=torch.int32) % 4 + 1
    ids[0, 1] = 2
    ids[1, 1] = 2
    ids[1, 0] = 3
    full_check(moe, w, inp)


def test_invalid_ids_and_empty_rows(moe, launch_mode):
    w, inp = _small(T=20, E=9, K=3)
    ids = inp["topk_ids"]
    ids[0, :] = -1            # a token with no valid route -> exact zero row
    ids[3, 1] = 9             # == E: out of range
    ids[5, 0] = 1000
    ids[7, 2] = -7
    full_check(moe, w, inp)


def test_dense_shape_small(moe, launch_mode):
    # K = 512-multiple contraction with several pipeline stages, 128-row tiles
    w, inp = _small(T=64, D=1024, I=512, E=3, K=2)
    full_check(moe, w, inp)


def test_large_tiles_mid_shape(moe, launch_mode):
    w, inp = _small(T=256, D=512, I=256, E=5, K=3)
    full_check(moe, w, inp)


@pytest.mark.parametrize("T,D,I,E,K", [
    (8, 128, 128, 1, 1),        # minimum dims, one expert, topk 1
    (12, 256, 128, 40, 16),     # maximum topk
    (24, 256, 128, 1024, 8),    # maximum E (routing histogram of 1024 experts)
    (16, 256, 128, 384, 8),     # 384 experts: the single-launch router at its limit
    (455, 256, 128, 33, 9),     # 4095 routes: one-CTA routing
    (456, 256, 128, 33, 9),     # 4104 routes: routing on many CTAs
])
def test_limits_and_routing_threshold(moe, T, D, I, E, K):
    w, inp = _small(T=T, D=D, I=I, E=E, K=K, seed=5)
    full_check(moe, w, inp)


@pytest.mark.parametrize("shape", [(16, 7168, 256, 257, 9), (256, 512, 256, 5, 3),
                                   (96, 1024, 512, 3, 2), (16, 256, 128, 9, 3),
                                   (200, 2048, 1024, 4, 3)])
def test_forced_tile_widths_and_copy_schemes(moe, shape):
    """Every forced route-tile width and scale-factor copy scheme passes the
    parity checks.  With one MMA-issuing warp (copy schemes 2 and 3) the output
    does not depend on the width or the scheme, bit for bit; with two (scheme 1)
    it does not depend on the width; scheme 4 (layout-warp copies, two MMA warps
    where their accumulators fit, else one) gives scheme 1's or scheme 2's output."""
    w = workloads.custom(*shape)
    inp = workloads.make_inputs(w, seed=9)
    outs = {}
    try:
        for rows in (16, 32, 64, 128):
            for copies in (1, 2, 3, 4):
                moe.set_tuning(rows, copies)
                m, _, out, _ = full_check(moe, w, inp)
                assert m.plan.tile_rows == rows
                outs[(rows, copies)] = out.view(torch.int16).cpu()
    finally:
        moe.set_tuning(0, 0)
    one_warp = [k for k in outs if k[1] in (2, 3)]
    for k in one_warp:
        assert torch.equal(outs[k], outs[one_warp[0]]), k
    for rows in (32, 64):
        assert torch.equal(outs[(rows, 1)], outs[(16, 1)]), rows
    for rows in (16, 32, 64, 128):
        assert (torch.equal(outs[(rows, 4)], outs[(rows, 1)]) or
                torch.equal(outs[(rows, 4)], outs[(rows, 2)])), rows


def test_empty_batch(moe):
    m = moe.MoeMXFP4(0, 256, 128, 9, 3)
    e = torch.empty(0, device="cuda")
    code = moe.forward_ptr(e.data_ptr(), 16, 16, 16, 16, 16, 16, 16, 0, 256, 128, 9, 3, 0)
    assert code == 0
    del m


def test_closed_form_bit_exact(moe, launch_mode):
    """All-ones case from tests/golden/closed_form.txt: exact in every step."""
    D, I, E, K, T = 256, 128, 1, 1, 1
    hidden = torch.ones(T, D, dtype=torch.bfloat16)
    inp = {
        "hidden": hidden,
        "w13": torch.full((E, 2 * I, D // 2), 0x22, dtype=torch.uint8),
        "w13_scale": torch.full((E, 2 * I, D // 32), 127, dtype=torch.uint8),
        "w2": torch.full((E, D, I // 2), 0x22, dtype=torch.uint8),
        "w2_scale": torch.full((E, D, I // 32), 127, dtype=torch.uint8),
        "topk_ids": torch.zeros(T, K, dtype=torch.int32),
        "topk_weights": torch.full((T, K), 0.375, dtype=torch.float32),
    }
    w = workloads.custom(T, D, I, E, K)
    _, _, out = run_gpu(moe, inp, w)
    assert (out.float().cpu() == 3145728.0).all()


def test_deterministic_repeat(moe, launch_mode):
    w = workloads.WORKLOADS[workloads.TINY]
    inp = workloads.make_inputs(w)
    m, t, out = run_gpu(moe, inp, w)
    ref = out.clone()
    for _ in range(5):
        o2 = m.forward(t["hidden"], t["w13"], t["w13_scale"], t["w2"], t["w2_scale"],
                       t["topk_ids"], t["topk_weights"])
        torch.cuda.synchronize()
        assert torch.equal(o2.view(torch.int16), ref.view(torch.int16))


def _padded_weights(inp, Dp, Ip, seed=7):
    """The logical weights inside padded storage (w13 gate rows at 0, up rows at Ip),
    with random e2m1 codes and finite scale bytes in the padding."""
    g = torch.Generator().manual_seed(seed)
    E, I2, Dh = inp["w13"].shape
    I, D = I2 // 2, Dh * 2
    w13 = torch.randint(0, 256, (E, 2 * Ip, Dp // 2), generator=g, dtype=torch.uint8)
    s13 = torch.randint(100, 141, (E, 2 * Ip, Dp // 32), generator=g, dtype=torch.uint8)
    w13[:, :I, : D // 2] = inp["w13"][:, :I]
    w13[:, Ip:Ip + I, : D // 2] = inp["w13"][:, I:]
    s13[:, :I, : D // 32] = inp["w13_scale"][:, :I]
    s13[:, Ip:Ip + I, : D // 32] = inp["w13_scale"][:, I:]
    w2 = torch.randint(0, 256, (E, Dp, Ip // 2), generator=g, dtype=torch.uint8)
    s2 = torch.randint(100, 141, (E, Dp, Ip // 32), generator=g, dtype=torch.uint8)
    w2[:, :D, : I // 2] = inp["w2"]
    s2[:, :D, : I // 32] = inp["w2_scale"]
    return {**inp, "w13": w13, "w13_scale": s13, "w2": w2, "w2_scale": s2}


@pytest.mark.parametrize("T,D,I,Dp,Ip,E,K", [
    (24, 224, 96, 256, 128, 5, 3),      # both dims padded inside one stage
    (40, 992, 416, 1024, 512, 9, 3),    # multi-stage contraction with a padded tail
    (16, 7168, 224, 7168, 256, 33, 9),  # d_model unpadded, d_inter padded
])
def test_padded_dims(moe, launch_mode, T, D, I, Dp, Ip, E, K):
    """Padded weight storage computes the logical problem: the oracle on the
    unpadded weights; routing and quantised hidden rows bit-exact, padding columns
    of the quantised rows zero."""
    w = workloads.custom(T, D, I, E, K)
    inp = workloads.make_inputs(w, seed=11)
    pin = _padded_weights(inp, Dp, Ip)
    dev = torch.device("cuda")
    m = moe.MoeMXFP4(T, D, I, E, K, d_model_pad=Dp, d_inter_pad=Ip)
    t = {k: v.to(dev) for k, v in pin.items()}
    out = m.forward(t["hidden"], t["w13"], t["w13_scale"], t["w2"], t["w2_scale"],
                    t["topk_ids"], t["topk_weights"])
    torch.cuda.synchronize()
    assert m.device_status() == 0
    assert out.shape == (T, D)
    npi = workloads.to_numpy(inp)
    routing = oracle.route(npi["topk_ids"], npi["topk_weights"], E, 16, cap=m.plan.cap)
    ref = oracle.forward(**npi, threads=_threads(), want_h=False)
    cap = m.plan.cap
    a1q = m.region("a1q", torch.uint8, (cap, Dp // 2)).cpu().numpy()
    a1s = m.region("a1s", torch.uint8, (cap, m.plan.a1s_stride)).cpu().numpy()
    a2q = m.region("a2q", torch.uint8, (cap, Ip // 2)).cpu().numpy()
    a2s = m.region("a2s", torch.uint8, (cap, m.plan.a2s_stride)).cpu().numpy()
    ws = {"a1q": a1q[:, : D // 2], "a1s": a1s, "a2q": a2q[:, : I // 2], "a2s": a2s}
    check_a1(ws, ref, routing, w)
    check_a2(ws, ref, routing, w)
    n = int(routing["num_valid"][0])
    valid = routing["sorted_ids"][:n] < w.R
    assert (a1q[:n][valid, D // 2:] == 0).all()
    assert (a2q[:n][valid, I // 2:] == 0).all()
    check_out(out, ref)


@pytest.mark.parametrize("T,D,I,E,K", [
    (64, 2944, 384, 16, 4),    # both widths run wider (3072, 512)
    (200, 1152, 768, 8, 3),    # d_model 9 x 128, d_inter 768 (1536, 1024), 128-route tiles
    (16, 384, 192, 9, 3),      # widths below 512 (512, 256)
    (8, 128, 64, 4, 2),        # d_inter of one 64-feature tile (128)
    (24, 7168, 320, 33, 4),    # d_model as it is, d_inter run wider (512)
])
def test_widths_run_wider(moe, launch_mode, T, D, I, E, K):
    """d_model a multiple of 128 and d_inter of 64 that are not 128, 256 or a
    multiple of 512, with the weights in their own (unpadded) layout: against the
    oracle on the same weights, routing and quantised hidden rows bit-exact, the
    intermediate within one e2m1 step, the activations' extra columns zero, every
    output row within the row bound; the call adds one launch."""
    w = workloads.custom(T, D, I, E, K)
    inp = workloads.make_inputs(w, seed=13)
    m, t, out = run_gpu(moe, inp, w)
    assert out.shape == (T, D)
    pl = m.plan
    Dr, Ir = pl.d_model_run, pl.d_inter_run
    assert (Dr, Ir) != (D, I)
    assert moe.call_launches(T, D, I, E, K) in (3, 5, 7)  # the weight-scale copy + 2, 4 or 6
    npi = workloads.to_numpy(inp)
    routing = oracle.route(npi["topk_ids"], npi["topk_weights"], E, 16, cap=pl.cap)
    ref = oracle.forward(**npi, threads=_threads(), want_h=False)
    cap = pl.cap
    get = lambda name, dt, shape: m.region(name, dt, shape).cpu().numpy()
    ws = {"sorted_ids": get("sorted_ids", torch.int32, (cap,)),
          "sorted_w": get("sorted_w", torch.float32, (cap,)),
          "block_expert": get("block_expert", torch.int32, (cap // 16,)),
          "seg_start": get("seg_start", torch.int32, (E + 1,)),
          "route_pos": get("route_pos", torch.int32, (T * K,)),
          "num_valid": get("num_valid", torch.int32, (4,)),
          "tiles": get("tiles", torch.int32, (pl.max_tiles, 4))}
    check_routing(ws, routing, w, pl.tile_rows)
    a1q = get("a1q", torch.uint8, (cap, Dr // 2))
    a1s = get("a1s", torch.uint8, (cap, pl.a1s_stride))
    a2q = get("a2q", torch.uint8, (cap, Ir // 2))
    a2s = get("a2s", torch.uint8, (cap, pl.a2s_stride))
    ws.update({"a1q": a1q[:, : D // 2], "a1s": a1s, "a2q": a2q[:, : I // 2], "a2s": a2s})
    check_a1(ws, ref, routing, w)
    check_a2(ws, ref, routing, w)
    n = int(routing["num_valid"][0])
    valid = routing["sorted_ids"][:n] < w.R
    assert (a1q[:n][valid, D // 2:] == 0).all()
    assert (a2q[:n][valid, I // 2:] == 0).all()
    check_out(out, ref)


@pytest.mark.parametrize("name", [workloads.DECODE_T16, "decode_T128_D7168_I256_E257_K9"])
def test_topk_sum_entry_matches_forward(moe, name):
    """moe_mxfp4_topk_sum on the forward's own P rows and route map gives the
    forward's output bit for bit (the same kernel and order), with one route made
    invalid; a route map with every route of token 0 off gives it a zero row."""
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, seed=17)
    inp["topk_ids"][0, 1] = -1
    m, t, out = run_gpu(moe, inp, w)
    P = m.region("P", torch.float32, (w.R, w.D)).clone()
    rpos = m.region("route_pos", torch.int32, (w.R,)).clone()
    o2 = torch.full_like(out, float("nan"))
    moe.topk_sum(P, rpos, o2)
    torch.cuda.synchronize()
    assert torch.equal(o2.view(torch.int16), out.view(torch.int16))
    rpos[: w.K] = -1
    moe.topk_sum(P, rpos, o2)
    torch.cuda.synchronize()
    assert (o2[0].float() == 0).all()
    assert torch.equal(o2[1:].view(torch.int16), out[1:].view(torch.int16))


def test_launch_modes_bitwise_identical(moe):
    """Single-launch mode reproduces the separate-kernel output and workspace
    routing arrays bit for bit (same routing order, same quantisation)."""
    w = workloads.WORKLOADS[workloads.DECODE_T16]
    inp = workloads.make_inputs(w, seed=3)
    outs, sids = [], []
    for mode in (0, 1):
        moe.set_single_launch(mode)
        try:
            m, t, out = run_gpu(moe, inp, w)
            torch.cuda.synchronize()
            assert m.device_status() == 0
            outs.append(out.view(torch.int16).cpu())
            sids.append(m.region("sorted_ids", torch.int32, (m.plan.cap,)).cpu().clone())
        finally:
            moe.set_single_launch(2)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(sids[0], sids[1])


@pytest.mark.gpu
def test_nvtx_ranges_change_nothing(moe, launch_mode):
    """With NVTX ranges on (no profiler attached) the forward gives the same
    output bit for bit as with them off, in both launch modes."""
    w = workloads.WORKLOADS[workloads.DECODE_T16]
    inp = workloads.make_inputs(w, seed=5)
    outs = []
    for on in (False, True):
        moe.set_nvtx(on)
        try:
            m, t, out = run_gpu(moe, inp, w)
            torch.cuda.synchronize()
            assert m.device_status() == 0
            outs.append(out.view(torch.int16).cpu())
        finally:
            moe.set_nvtx(False)
    assert torch.equal(outs[0], outs[1])


def test_quantiser_every_bf16_value(moe, launch_mode):
    """Every finite bf16 value goes through the activation quantiser (the quant
    kernel, or the one inside the GEMM kernel in single-launch mode): once in
    bit-pattern order, so a block holds 32 neighbouring values (ties and
    saturation), once shuffled (mixed magnitudes).  Codes and scales must equal
    the oracle's bit for bit.  The GEMM outputs of such inputs overflow and are
    not checked."""
    bits = np.arange(65536, dtype=np.uint32)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    vals = bits[finite].astype(np.uint16)
    rng = np.random.default_rng(11)
    allv = np.concatenate([vals, rng.permutation(vals)])
    D = 256
    allv = np.concatenate([allv, np.zeros((-len(allv)) % D, np.uint16)])
    T = len(allv) // D
    w = workloads.custom(T, D, 128, 9, 1)
    inp = workloads.make_inputs(w, seed=2)
    inp["hidden"] = torch.from_numpy(allv.view(np.int16).reshape(T, D).copy()).view(torch.bfloat16)
    m, t, out = run_gpu(moe, inp, w)
    ws = ws_arrays(m, w)
    f32 = (allv.astype(np.uint32) << 16).view(np.float32).reshape(T, D)
    for tok in range(T):
        pos = int(ws["route_pos"][tok])
        codes, scales = oracle.quant_row(f32[tok])
        np.testing.assert_array_equal(ws["a1q"][pos], codes, err_msg=f"codes of token {tok}")
        np.testing.assert_array_equal(ws["a1s"][pos, : D // 32], scales, err_msg=f"scales of token {tok}")


@pytest.mark.parametrize("shape,act", [
    ((16, 7168, 256, 257, 9), "mxfp4"),   # decode: single launch
    ((64, 512, 256, 17, 5), "mxfp4"),     # 320 routes: separate kernels
    ((820, 256, 128, 9, 5), "mxfp4"),     # 4100 routes: routing on many CTAs
    ((16, 256, 128, 9, 3), "bf16"),       # W4A16 path
], ids=["decode_single", "separate", "multi_cta_routing", "w4a16"])
def test_host_buffers_bitwise_identical(moe, shape, act):
    """hidden, topk_ids, topk_weights and out in pinned host memory: the kernels
    read and write them in place, with the same result bit for bit as with the
    same data in device memory."""
    T, D, I, E, K = shape
    w = workloads.custom(T, D, I, E, K)
    inp = workloads.make_inputs(w, seed=7)
    dev = torch.device("cuda")
    m = moe.MoeMXFP4(T, D, I, E, K, activations=act)
    wts = [inp[k].to(dev) for k in ("w13", "w13_scale", "w2", "w2_scale")]
    d_out = m.forward(inp["hidden"].to(dev), *wts, inp["topk_ids"].to(dev),
                      inp["topk_weights"].to(dev))
    torch.cuda.synchronize()
    assert m.device_status() == 0
    h = {k: inp[k].contiguous().pin_memory() for k in ("hidden", "topk_ids", "topk_weights")}
    h_out = torch.full((T, D), float("nan"), dtype=torch.bfloat16).pin_memory()
    m.forward(h["hidden"], *wts, h["topk_ids"], h["topk_weights"], out=h_out)
    torch.cuda.synchronize()
    assert m.device_status() == 0
    assert torch.equal(h_out.view(torch.int16), d_out.cpu().view(torch.int16))


def test_host_buffers_rejects_pageable(moe):
    w = workloads.custom(16, 256, 128, 9, 3)
    inp = workloads.make_inputs(w)
    m = moe.MoeMXFP4(16, 256, 128, 9, 3)
    dev = torch.device("cuda")
    wts = [inp[k].to(dev) for k in ("w13", "w13_scale", "w2", "w2_scale")]
    with pytest.raises(ValueError):
        m.forward(inp["hidden"], *wts, inp["topk_ids"].to(dev), inp["topk_weights"].to(dev))


# ------------------------------------------------------------------ failure reporting

def test_bounded_wait_timeout_is_reported_and_recoverable(moe):
    """A device wait that runs out (a barrier nothing arrives on, 20 ms limit)
    is reported as MOE_ERR_DEVICE_TIMEOUT; the next forward clears it."""
    w = workloads.WORKLOADS[workloads.TINY]
    inp = workloads.make_inputs(w)
    m, t, out = run_gpu(moe, inp, w)
    moe.set_workspace(m.ws_ptr, m.ws_bytes)
    stream = torch.cuda.current_stream().cuda_stream
    assert moe.check_wait_timeout(20000, stream) == 0
    assert moe.last_device_status(stream) == 6  # MOE_ERR_DEVICE_TIMEOUT
    status = m.region("status", torch.int32, (16,)).cpu().numpy()
    assert status[0] & (1 << 5)
    out2 = m.forward(t["hidden"], t["w13"], t["w13_scale"], t["w2"], t["w2_scale"],
                     t["topk_ids"], t["topk_weights"])
    torch.cuda.synchronize()
    assert m.device_status() == 0
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    assert moe.check_wait_timeout(0, stream) == 1  # limit out of range


@pytest.mark.parametrize("name", [workloads.TINY, workloads.DECODE_T16,
                                  "decode_T128_D7168_I256_E257_K9"])
def test_cuda_graph_replay_matches_direct_calls(moe, name):
    """The forward captured in a CUDA graph and replayed (single launch at decode
    sizes, separate kernels at T = 128) gives the direct call's output bit for bit,
    on every replay, with new inputs copied into the captured buffers in between."""
    w = workloads.WORKLOADS[name]
    dev = torch.device("cuda")
    m = moe.MoeMXFP4(w.T, w.D, w.I, w.E, w.K)
    inp0 = {k: v.to(dev) for k, v in workloads.make_inputs(w, seed=1).items()}
    # a second batch (other hidden states and routes) for the same weights
    inp1 = dict(inp0)
    for k, v in workloads.make_inputs(w, seed=2).items():
        if k in ("hidden", "topk_ids", "topk_weights"):
            inp1[k] = v.to(dev)
    names = ("hidden", "w13", "w13_scale", "w2", "w2_scale", "topk_ids", "topk_weights")
    ref = []
    for inp in (inp0, inp1):
        o = m.forward(*(inp[k] for k in names))
        torch.cuda.synchronize()
        ref.append(o.clone())
    buf = {k: v.clone() for k, v in inp0.items()}
    out = torch.empty(w.T, w.D, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.forward(*(buf[k] for k in names), out=out)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.forward(*(buf[k] for k in names), out=out)
    for it in range(4):
        src = inp0 if it % 2 == 0 else inp1
        for k in ("hidden", "topk_ids", "topk_weights"):
            buf[k].copy_(src[k])
        g.replay()
        torch.cuda.synchronize()
        assert m.device_status() == 0
        assert torch.equal(out.view(torch.int16), ref[it % 2].view(torch.int16)), f"replay {it}"
