"""CPU oracle for the fused MXFP4 Mixture-of-Experts forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``mixture_experts_mxfp4_gb300``) never does, and the
two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp32, single ascending loops);
this module only builds it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_LIB = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FMA contraction). Returns the .so path."""
    need = force or not os.path.exists(_LIB)
    if not need:
        lib_m = os.path.getmtime(_LIB)
        need = any(os.path.getmtime(p) > lib_m for p in (_SRC, _HDR))
    if need:
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # MOE_ORACLE_LIB: a given build of moe_oracle.c (the mutation tests load
            # copies with a planted mistake this way); otherwise build and load ours
            path = os.environ.get("MOE_ORACLE_LIB")
            if not path:
                build()
                path = _LIB
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.moe_oracle_e2m1.restype = ctypes.c_float
            lib.moe_oracle_e2m1.argtypes = [i]
            lib.moe_oracle_e8m0.restype = ctypes.c_float
            lib.moe_oracle_e8m0.argtypes = [i]
            lib.moe_oracle_bf16_bits.restype = ctypes.c_uint16
            lib.moe_oracle_bf16_bits.argtypes = [ctypes.c_float]
            lib.moe_oracle_quant_block.restype = None
            lib.moe_oracle_quant_block.argtypes = [P, P, P]
            lib.moe_oracle_quant_row.restype = None
            lib.moe_oracle_quant_row.argtypes = [P, i, P, P]
            lib.moe_oracle_route_capacity.restype = i
            lib.moe_oracle_route_capacity.argtypes = [i, i, i, i]
            lib.moe_oracle_route.restype = i
            lib.moe_oracle_route.argtypes = [P, P, i, i, i, i, i, P, P, P, P, P, P]
            lib.moe_oracle_forward.restype = i
            lib.moe_oracle_forward.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, P, i, i,
                                               P, P, P, P, P, P, P, i]
            lib.moe_oracle_max_threads.restype = i
            lib.moe_oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1(code: int) -> float:
    return float(_load().moe_oracle_e2m1(int(code)))


def e8m0(s: int) -> float:
    return float(_load().moe_oracle_e8m0(int(s)))


def bf16_bits(x: float) -> int:
    return int(_load().moe_oracle_bf16_bits(float(x)))


def quant_block(v):
    """MX-quantise 32 values -> (16 code bytes, scale byte)."""
    v = _c(v, np.float32)
    assert v.shape == (32,)
    codes = np.zeros(16, np.uint8)
    scale = np.zeros(1, np.uint8)
    _load().moe_oracle_quant_block(_ptr(v), _ptr(codes), _ptr(scale))
    return codes, int(scale[0])


def quant_row(v):
    """MX-quantise a row (length % 32 == 0) -> (codes [n/2], scales [n/32])."""
    v = _c(v, np.float32).reshape(-1)
    n = v.shape[0]
    assert n % 32 == 0
    codes = np.zeros(n // 2, np.uint8)
    scales = np.zeros(n // 32, np.uint8)
    _load().moe_oracle_quant_row(_ptr(v), n, _ptr(codes), _ptr(scales))
    return codes, scales


def route_capacity(T: int, topk: int, E: int, bm: int) -> int:
    return int(_load().moe_oracle_route_capacity(T, topk, E, bm))


def route(topk_ids, topk_weights, E: int, bm: int, cap: int | None = None) -> dict:
    """Counting sort of routes by expert, padded to bm (see moe_oracle_route)."""
    ids = _c(topk_ids, np.int32)
    T, K = ids.shape
    w = _c(topk_weights, np.float32).reshape(T, K)
    if cap is None:
        cap = route_capacity(T, K, E, bm)
    out = {
        "sorted_ids": np.zeros(cap, np.int32),
        "sorted_w": np.zeros(cap, np.float32),
        "block_expert": np.zeros(max(cap // bm, 0), np.int32),
        "seg_start": np.zeros(E + 1, np.int32),
        "route_pos": np.zeros(T * K, np.int32),
        "num_valid": np.zeros(2, np.int32),
    }
    rc = _load().moe_oracle_route(_ptr(ids), _ptr(w), T, K, E, bm, cap, _ptr(out["sorted_ids"]),
                                  _ptr(out["sorted_w"]), _ptr(out["block_expert"]),
                                  _ptr(out["seg_start"]), _ptr(out["route_pos"]),
                                  _ptr(out["num_valid"]))
    if rc != 0:
        raise ValueError("oracle route: bad arguments or capacity too small")
    out["cap"] = cap
    out["bm"] = bm
    return out


def max_threads() -> int:
    return int(_load().moe_oracle_max_threads())


def forward(hidden_bits, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights,
            tokens=None, quant_act: bool = True, threads: int = 1,
            want_h: bool = True) -> dict:
    """Run the oracle forward.

    hidden_bits: uint16 [T, D] (bf16 bit patterns); w13 uint8 [E, 2I, D/2];
    w13_scale uint8 [E, 2I, D/32]; w2 uint8 [E, D, I/2]; w2_scale uint8 [E, D, I/32];
    topk_ids int32 [T, K]; topk_weights float32 [T, K]; tokens: optional list of token
    indices to compute (others are left zero).
    """
    hid = _c(hidden_bits, np.uint16)
    T, D = hid.shape
    w13 = _c(w13, np.uint8)
    E, I2, Dh = w13.shape
    I = I2 // 2
    assert Dh * 2 == D
    w13s = _c(w13_scale, np.uint8)
    w2 = _c(w2, np.uint8)
    w2s = _c(w2_scale, np.uint8)
    assert w13s.shape == (E, 2 * I, D // 32)
    assert w2.shape == (E, D, I // 2) and w2s.shape == (E, D, I // 32)
    ids = _c(topk_ids, np.int32)
    K = ids.shape[1]
    tw = _c(topk_weights, np.float32).reshape(T, K)
    tok = None if tokens is None else _c(tokens, np.int32).reshape(-1)
    R = T * K
    res = {
        "a1q": np.zeros((T, D // 2), np.uint8),
        "a1s": np.zeros((T, D // 32), np.uint8),
        "h": np.zeros((R, I), np.float32) if want_h else None,
        "a2q": np.zeros((R, I // 2), np.uint8),
        "a2s": np.zeros((R, I // 32), np.uint8),
        "out_f32": np.zeros((T, D), np.float32),
        "out_bf16": np.zeros((T, D), np.uint16),
    }
    rc = _load().moe_oracle_forward(
        _ptr(hid), _ptr(w13), _ptr(w13s), _ptr(w2), _ptr(w2s), _ptr(ids), _ptr(tw),
        T, D, I, E, K, _ptr(tok), 0 if tok is None else int(tok.shape[0]), 1 if quant_act else 0,
        _ptr(res["a1q"]), _ptr(res["a1s"]), _ptr(res["h"]), _ptr(res["a2q"]), _ptr(res["a2s"]),
        _ptr(res["out_f32"]), _ptr(res["out_bf16"]), int(threads))
    if rc != 0:
        raise ValueError("oracle forward: bad arguments")
    return res


def bf16_bits_to_f32(bits):
    """Widen bf16 bit patterns to fp32 (a bit shift; no rounding)."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)
