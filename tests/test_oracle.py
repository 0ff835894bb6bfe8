"""Pins for the CPU oracle: checks against values the pages and the number
formats fix, closed forms, invariants and an independent fp64 brute force.

These run without a GPU.  A pin here never re-calls the oracle routine it
checks: expected values come from tests/golden (hand-derived, cited), from an
independent library routine (math.ldexp, torch's bf16 cast, numpy fp64 dense
algebra, Python's sort), or from an invariant of the method.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import GOLDEN


# ----------------------------------------------------------------- fixtures

def _golden_e2m1():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            vals[int(c)] = float(v)
    return vals


def _parse_val(tok):
    if tok == "nan":
        return float("nan")
    if tok[0] in "pn" and tok[1:].lstrip("-").isdigit():
        v = math.ldexp(1.0, int(tok[1:]))
        return v if tok[0] == "p" else -v
    return float(tok)


def _golden_quant_cases():
    cases = []
    cur = None
    with open(os.path.join(GOLDEN, "mx_quant_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key == "case":
                cur = {"name": rest[0]}
                cases.append(cur)
            elif key == "v":
                cur["v"] = [_parse_val(t) for t in rest]
            elif key == "s":
                cur["s"] = int(rest[0])
            elif key == "c":
                cur["c"] = [int(t) for t in rest]
    return cases


E2M1 = _golden_e2m1()
E2M1_TABLE = np.array([E2M1[c] for c in range(16)], dtype=np.float64)


def np_dequant(codes, scales, n):
    """Independent fp64 decode of packed e2m1 rows with e8m0 scales (golden table)."""
    codes = np.asarray(codes, np.uint8)
    lead = codes.shape[:-1]
    lo = codes & 0x0F
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(*lead, n)
    vals = E2M1_TABLE[nib]
    sc = np.ldexp(1.0, np.asarray(scales, np.int64) - 127).astype(np.float64)
    return vals * np.repeat(sc, 32, axis=-1)


def unpack_codes(packed):
    p = np.asarray(packed, np.uint8)
    return np.stack([p & 15, p >> 4], axis=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)


# ----------------------------------------------------------------- formats

def test_e2m1_table_matches_format_definition():
    for c in range(16):
        got = oracle.e2m1(c)
        assert got == E2M1[c], (c, got)
        assert math.copysign(1.0, got) == math.copysign(1.0, E2M1[c]), c  # -0 for code 8


def test_e8m0_is_power_of_two():
    for s in range(255):
        assert oracle.e8m0(s) == np.float32(math.ldexp(1.0, s - 127)), s
    assert math.isnan(oracle.e8m0(255))


def test_bf16_rounding_against_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(1e3),
        np.array([1.0, 1.00390625, 1.01171875, 1.0 + 2 ** -8 + 2 ** -20, -1.00390625,
                  3.4e38, -3.4e38, 1e-40, 0.0, -0.0], np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_bits(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, ref)
    # hand cases: ties go to the even bf16 mantissa
    assert oracle.bf16_bits(1.00390625) == 0x3F80  # 1 + 2^-8: tie -> 1.0
    assert oracle.bf16_bits(1.01171875) == 0x3F82  # 1 + 3*2^-8: tie -> even 0x3F82


# ----------------------------------------------------------------- quantiser

@pytest.mark.parametrize("case", _golden_quant_cases(), ids=lambda c: c["name"])
def test_quant_golden_cases(case):
    v = np.array(case["v"], np.float32)
    assert v.shape == (32,)
    codes, s = oracle.quant_block(v)
    assert s == case["s"]
    np.testing.assert_array_equal(unpack_codes(codes[None])[0], np.array(case["c"], np.uint8))


def test_quant_roundtrip_of_representable_values():
    """Every representable value c * 2^X in a block whose amax is 6 * 2^X is
    reproduced exactly, for scales across the whole e8m0 range."""
    for X in [-125, -60, -3, -2, 0, 1, 7, 60, 125]:
        for c in range(16):
            v = np.zeros(32, np.float32)
            v[0] = np.float32(math.ldexp(6.0, X))
            v[1:] = np.float32(math.ldexp(E2M1[c], X))
            codes, s = oracle.quant_block(v)
            assert s == X + 127
            u = unpack_codes(codes[None])[0]
            assert u[0] == 7
            assert (u[1:] == c).all(), (X, c, u)


def test_quant_is_nearest_on_random_blocks():
    """Against an fp64 nearest-grid search: the chosen magnitude is never
    farther than any other grid value (ties are covered by the golden cases)."""
    rng = np.random.default_rng(7)
    grid = E2M1_TABLE[:8]
    for _ in range(300):
        v = (rng.standard_normal(32) * rng.choice([1e-3, 1.0, 37.0])).astype(np.float32)
        codes, s = oracle.quant_block(v)
        amax = float(np.max(np.abs(v)))
        assert s == math.floor(math.log2(amax)) - 2 + 127
        q = np.abs(v.astype(np.float64)) / math.ldexp(1.0, s - 127)
        u = unpack_codes(codes[None])[0]
        mag = grid[u & 7]
        best = np.min(np.abs(q[:, None] - grid[None, :]), axis=1)
        assert np.all(np.abs(q - mag) <= best + 1e-12)
        assert np.all(((u >> 3) == 1) == np.signbit(v))


# ----------------------------------------------------------------- routing

def _route_by_sort(ids, E, bm):
    """Independent construction: Python's stable sort by expert, then padding."""
    R = ids.size
    flat = [int(x) for x in ids.reshape(-1)]
    valid = [r for r in range(R) if 0 <= flat[r] < E]
    order = sorted(valid, key=lambda r: flat[r])  # stable: ascending r within an expert
    seq = []
    blocks = []
    for e in range(E):
        seg = [r for r in order if flat[r] == e]
        if not seg:
            continue
        pad = (-len(seg)) % bm
        seq += seg + [R] * pad
        blocks += [e] * ((len(seg) + pad) // bm)
    return seq, blocks


@pytest.mark.parametrize("T,K,E,bm", [(16, 3, 9, 16), (7, 4, 5, 4), (33, 9, 257, 16), (1, 1, 1, 8)])
def test_route_against_sort(T, K, E, bm):
    rng = np.random.default_rng(T * 100 + K)
    ids = rng.integers(-2, E + 2, size=(T, K)).astype(np.int32)  # duplicates + out-of-range ids
    w = rng.standard_normal((T, K)).astype(np.float32)
    res = oracle.route(ids, w, E, bm)
    seq, blocks = _route_by_sort(ids, E, bm)
    n = len(seq)
    R = T * K
    assert res["num_valid"][0] == n
    assert res["num_valid"][1] == int(((ids >= 0) & (ids < E)).sum())
    np.testing.assert_array_equal(res["sorted_ids"][:n], np.array(seq, np.int32))
    assert (res["sorted_ids"][n:] == R).all()
    np.testing.assert_array_equal(res["block_expert"][: len(blocks)], np.array(blocks, np.int32))
    assert (res["block_expert"][len(blocks):] == -1).all()
    flat_w = w.reshape(-1)
    for p in range(res["cap"]):
        r = res["sorted_ids"][p]
        assert res["sorted_w"][p] == (flat_w[r] if r < R else 0.0)
    for r in range(R):
        p = res["route_pos"][r]
        if 0 <= ids.reshape(-1)[r] < E:
            assert res["sorted_ids"][p] == r
        else:
            assert p == -1
    # invariants: each segment a multiple of bm, fewer than bm padding slots per expert
    ss = res["seg_start"]
    assert ((ss[1:] - ss[:-1]) % bm == 0).all()
    counts = np.bincount(ids.reshape(-1)[(ids.reshape(-1) >= 0) & (ids.reshape(-1) < E)], minlength=E)
    assert ((ss[1:] - ss[:-1]) - counts < bm).all()
    assert res["cap"] >= n


# ----------------------------------------------------------------- closed forms

def _closed_form_cases():
    rows = []
    with open(os.path.join(GOLDEN, "closed_form.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            t = line.split()
            rows.append(dict(name=t[0], hidden=float(t[1]), gate=int(t[2]), up=int(t[3]),
                             down=int(t[4]), s13=int(t[5]), s2=int(t[6]), w=float(t[7]),
                             out=float(t[8]), a1s=int(t[9]), a2s=int(t[10])))
    return rows


@pytest.mark.parametrize("case", _closed_form_cases(), ids=lambda c: c["name"])
def test_closed_form_one_token_one_expert(case):
    D, I, E, K = 256, 128, 1, 1
    hidden = torch.full((1, D), case["hidden"], dtype=torch.bfloat16)
    hb = hidden.view(torch.int16).numpy().view(np.uint16)
    w13 = np.zeros((E, 2 * I, D // 2), np.uint8)
    w13[:, :I] = case["gate"] * 17  # both nibbles
    w13[:, I:] = case["up"] * 17
    w13s = np.full((E, 2 * I, D // 32), case["s13"], np.uint8)
    w2 = np.full((E, D, I // 2), case["down"] * 17, np.uint8)
    w2s = np.full((E, D, I // 32), case["s2"], np.uint8)
    ids = np.zeros((1, K), np.int32)
    tw = np.full((1, K), case["w"], np.float32)
    res = oracle.forward(hb, w13, w13s, w2, w2s, ids, tw)
    out = oracle.bf16_bits_to_f32(res["out_bf16"])
    assert (out == np.float32(case["out"])).all(), (case["name"], out[0, :4])
    assert (res["a1s"] == case["a1s"]).all()
    assert (res["a2s"] == case["a2s"]).all()


# ----------------------------------------------------------------- invariants

@pytest.fixture(scope="module")
def tiny():
    w = workloads.WORKLOADS[workloads.TINY]
    return w, workloads.to_numpy(workloads.make_inputs(w))


def test_zero_weight_equals_dropping_the_route(tiny):
    w, inp = tiny
    base = dict(inp)
    tw = inp["topk_weights"].copy()
    ids = inp["topk_ids"].copy()
    rng = np.random.default_rng(3)
    picks = [(int(rng.integers(w.T)), int(rng.integers(w.K))) for _ in range(6)]
    for t, k in picks:
        tw[t, k] = 0.0
        ids[t, k] = -1
    zero_w = oracle.forward(**{**base, "topk_weights": tw})
    dropped = oracle.forward(**{**base, "topk_ids": ids, "topk_weights": tw})
    np.testing.assert_array_equal(zero_w["out_bf16"], dropped["out_bf16"])
    np.testing.assert_array_equal(zero_w["out_f32"], dropped["out_f32"])


def test_expert_permutation_invariance(tiny):
    w, inp = tiny
    rng = np.random.default_rng(11)
    perm = rng.permutation(w.E)  # new id of old expert e is perm[e]
    inv = np.argsort(perm)
    ref = oracle.forward(**inp)
    p = dict(inp)
    p["w13"] = inp["w13"][inv]
    p["w13_scale"] = inp["w13_scale"][inv]
    p["w2"] = inp["w2"][inv]
    p["w2_scale"] = inp["w2_scale"][inv]
    p["topk_ids"] = perm[inp["topk_ids"]].astype(np.int32)
    got = oracle.forward(**p)
    np.testing.assert_array_equal(got["out_bf16"], ref["out_bf16"])
    np.testing.assert_array_equal(got["a2q"], ref["a2q"])
    # routing permutes accordingly: expert perm[e]'s segment holds expert e's routes
    bm = 4
    r0 = oracle.route(inp["topk_ids"], inp["topk_weights"], w.E, bm)
    r1 = oracle.route(p["topk_ids"], p["topk_weights"], w.E, bm)
    for e in range(w.E):
        a = r0["sorted_ids"][r0["seg_start"][e]:r0["seg_start"][e + 1]]
        b = r1["sorted_ids"][r1["seg_start"][perm[e]]:r1["seg_start"][perm[e] + 1]]
        np.testing.assert_array_equal(a, b)


def test_thread_count_and_token_subset_do_not_change_results(tiny):
    w, inp = tiny
    one = oracle.forward(**inp, threads=1)
    many = oracle.forward(**inp, threads=4)
    for key in ("out_bf16", "out_f32", "a1q", "a1s", "a2q", "a2s", "h"):
        np.testing.assert_array_equal(one[key], many[key])
    sub = [3, 0, 11]
    part = oracle.forward(**inp, tokens=sub)
    np.testing.assert_array_equal(part["out_bf16"][sub], one["out_bf16"][sub])


@pytest.mark.parametrize("T", [1, 4])
def test_dense_fp64_brute_force(tiny, T):
    """Dequantise everything to fp64 dense matrices and route through one-hot
    expert masks; compare each stage of the oracle.  Catches indexing, nibble
    order, scale indexing, gate/up order and top-k weighting mistakes."""
    w, inp = tiny
    inp = {k: (v[:T] if k in ("hidden_bits", "topk_ids", "topk_weights") else v)
           for k, v in inp.items()}
    ids = inp["topk_ids"].copy()
    ids[0, 0] = ids[0, 1] if w.K > 1 else ids[0, 0]  # a duplicate expert inside one token
    inp["topk_ids"] = ids
    D, I, E, K = w.D, w.I, w.E, w.K
    res = oracle.forward(**inp)

    hid = oracle.bf16_bits_to_f32(inp["hidden_bits"]).astype(np.float32)
    # a1 rows: the pinned quantiser applied to each token row
    for t in range(T):
        c, s = oracle.quant_row(hid[t])
        np.testing.assert_array_equal(res["a1q"][t], c)
        np.testing.assert_array_equal(res["a1s"][t], s)
    A1 = np_dequant(res["a1q"], res["a1s"], D)  # [T, D]
    W13 = np_dequant(inp["w13"], inp["w13_scale"], D)  # [E, 2I, D]
    W2 = np_dequant(inp["w2"], inp["w2_scale"], I)  # [E, D, I]
    M = np.zeros((T, K, E))
    for t in range(T):
        for k in range(K):
            M[t, k, ids[t, k]] = 1.0
    G = np.einsum("tke,enj,tj->tkn", M, W13[:, :I], A1)
    U = np.einsum("tke,enj,tj->tkn", M, W13[:, I:], A1)
    H = G / (1.0 + np.exp(-G)) * U
    h_or = res["h"].reshape(T, K, I).astype(np.float64)
    # oracle h = bf16(fp32 sums): within one bf16 rounding + fp32 accumulation of D terms
    absG = np.einsum("tke,enj,tj->tkn", M, np.abs(W13[:, :I]), np.abs(A1))
    absU = np.einsum("tke,enj,tj->tkn", M, np.abs(W13[:, I:]), np.abs(A1))
    bound = 2.0 ** -8 * np.abs(H) + 4 * D * 2.0 ** -24 * (absG * np.abs(U) + absU * np.abs(G)) + 1e-30
    assert np.all(np.abs(h_or - H) <= bound)
    # a2 rows are the pinned quantiser applied to the oracle's h rows (index consistency)
    for r in range(T * K):
        c, s = oracle.quant_row(res["h"][r])
        np.testing.assert_array_equal(res["a2q"][r], c)
        np.testing.assert_array_equal(res["a2s"][r], s)
    A2 = np_dequant(res["a2q"], res["a2s"], I).reshape(T, K, I)
    Y = np.einsum("tke,enj,tkj->tkn", M, W2, A2)
    OUT = np.einsum("tk,tkn->tn", inp["topk_weights"].astype(np.float64), Y)
    absY = np.einsum("tke,enj,tkj->tkn", M, np.abs(W2), np.abs(A2))
    absO = np.einsum("tk,tkn->tn", np.abs(inp["topk_weights"].astype(np.float64)), absY)
    tol = 4 * (I + K) * 2.0 ** -24 * absO + 1e-30
    assert np.all(np.abs(res["out_f32"].astype(np.float64) - OUT) <= tol)
    # the output is the bf16 rounding of out_f32
    ref_bits = torch.from_numpy(res["out_f32"]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(res["out_bf16"], ref_bits)


@pytest.mark.parametrize("T", [1, 4])
def test_w4a16_dense_fp64_brute_force(tiny, T):
    """The oracle's bf16-activation mode (quant_act=False: no activation quantiser,
    the bf16 SwiGLU output feeds stage 2 directly, as in solution.py's
    _reference_forward) against fp64 dense matrices through one-hot expert masks."""
    w, inp = tiny
    inp = {k: (v[:T] if k in ("hidden_bits", "topk_ids", "topk_weights") else v)
           for k, v in inp.items()}
    ids = inp["topk_ids"]
    D, I, E, K = w.D, w.I, w.E, w.K
    res = oracle.forward(**inp, quant_act=False)
    X = oracle.bf16_bits_to_f32(inp["hidden_bits"]).astype(np.float64)  # [T, D], exact
    W13 = np_dequant(inp["w13"], inp["w13_scale"], D)
    W2 = np_dequant(inp["w2"], inp["w2_scale"], I)
    M = np.zeros((T, K, E))
    for t in range(T):
        for k in range(K):
            M[t, k, ids[t, k]] = 1.0
    G = np.einsum("tke,enj,tj->tkn", M, W13[:, :I], X)
    U = np.einsum("tke,enj,tj->tkn", M, W13[:, I:], X)
    H = G / (1.0 + np.exp(-G)) * U
    h_or = res["h"].reshape(T, K, I).astype(np.float64)
    absG = np.einsum("tke,enj,tj->tkn", M, np.abs(W13[:, :I]), np.abs(X))
    absU = np.einsum("tke,enj,tj->tkn", M, np.abs(W13[:, I:]), np.abs(X))
    bound = 2.0 ** -8 * np.abs(H) + 4 * D * 2.0 ** -24 * (absG * np.abs(U) + absU * np.abs(G)) + 1e-30
    assert np.all(np.abs(h_or - H) <= bound)
    # h is already a bf16 value: widening its bf16 bits gives it back
    hb = torch.from_numpy(res["h"]).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(hb, res["h"])
    # stage 2 consumes h itself (no requantisation)
    Y = np.einsum("tke,enj,tkj->tkn", M, W2, h_or)
    OUT = np.einsum("tk,tkn->tn", inp["topk_weights"].astype(np.float64), Y)
    absY = np.einsum("tke,enj,tkj->tkn", M, np.abs(W2), np.abs(h_or))
    absO = np.einsum("tk,tkn->tn", np.abs(inp["topk_weights"].astype(np.float64)), absY)
    tol = 4 * (I + K) * 2.0 ** -24 * absO + 1e-30
    assert np.all(np.abs(res["out_f32"].astype(np.float64) - OUT) <= tol)
    ref_bits = torch.from_numpy(res["out_f32"]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(res["out_bf16"], ref_bits)
    # and it differs from the quantised path (the mode switch is live)
    q = oracle.forward(**inp)
    assert not np.array_equal(q["out_bf16"], res["out_bf16"])


def test_invalid_ids_contribute_nothing(tiny):
    w, inp = tiny
    ids = inp["topk_ids"].copy()
    ids[:, 0] = w.E + 5
    ids[:, 1] = -3
    res = oracle.forward(**{**inp, "topk_ids": ids})
    keep = inp["topk_ids"].copy()
    keep[:, 0] = -1
    keep[:, 1] = -1
    ref = oracle.forward(**{**inp, "topk_ids": keep})
    np.testing.assert_array_equal(res["out_bf16"], ref["out_bf16"])
    all_bad = np.full_like(ids, -1)
    z = oracle.forward(**{**inp, "topk_ids": all_bad})
    assert (z["out_bf16"] == 0).all()
