"""Seeded synthetic inputs for the fused MXFP4 MoE forward.

Used by both the tests/benchmark (device copies) and the CPU oracle.  This module
only draws random tensors; it holds none of the method's arithmetic.

Shapes and generator idioms follow the DeepSeek-R1-shaped self-test of
kernelbot-amd-moe-mxfp4-723815 (solution.py, ``_make``): uniform random code
bytes, distinct routed expert ids per token from a random permutation, the
shared expert id appended last with weight 1.0, softmax router weights.  Scale
bytes are drawn uniformly from [118, 124] so that values span several binades.

Draw order (one ``torch.Generator('cpu')`` seeded with ``seed``):
  1. hidden  = randn(T, D) -> bf16
  2. w13     = randint(0, 256, [E, 2I, D/2]) uint8
  3. w13_scale = randint(118, 125, [E, 2I, D/32]) uint8
  4. w2      = randint(0, 256, [E, D, I/2]) uint8;  w2_scale = randint(118, 125, [E, D, I/32])
  5. routed ids: per token randperm(E-1)[:K-1] (uniform), or, for the skewed
     prefill workload, K-1 draws without replacement from p(e) ~ (e+1)^-s
     (Zipf, expert 0 hottest) via sequential weighted sampling; then id E-1.
  6. weights: softmax(randn(T, K-1)) for the routed slots, 1.0 for the shared slot.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    I: int
    E: int
    K: int
    zipf: float | None = None

    @property
    def R(self) -> int:
        return self.T * self.K


# The five workloads: a tiny case the oracle finishes in well under a second,
# two DeepSeek-R1-style decode batches, a dense-expert shard, and a skewed
# prefill batch.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_T16_D256_I128_E9_K3", 16, 256, 128, 9, 3),
        Workload("decode_T16_D7168_I256_E257_K9", 16, 7168, 256, 257, 9),
        Workload("decode_T128_D7168_I256_E257_K9", 128, 7168, 256, 257, 9),
        Workload("dense_T512_D7168_I2048_E33_K9", 512, 7168, 2048, 33, 9),
        Workload("prefill_zipf_T4096_D7168_I256_E257_K9", 4096, 7168, 256, 257, 9, zipf=1.2),
    ]
}
ORDER = list(WORKLOADS)
TINY = ORDER[0]
DECODE_T16 = ORDER[1]


def custom(T, D, I, E, K, zipf=None, name=None) -> Workload:
    return Workload(name or f"custom_T{T}_D{D}_I{I}_E{E}_K{K}", T, D, I, E, K, zipf)


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw the inputs of workload ``w`` on the CPU (torch tensors)."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    T, D, I, E, K = w.T, w.D, w.I, w.E, w.K
    hidden = torch.randn(T, D, generator=g).to(torch.bfloat16)
    w13 = torch.randint(0, 256, (E, 2 * I, D // 2), generator=g, dtype=torch.uint8)
    w13_scale = torch.randint(118, 125, (E, 2 * I, D // 32), generator=g, dtype=torch.uint8)
    w2 = torch.randint(0, 256, (E, D, I // 2), generator=g, dtype=torch.uint8)
    w2_scale = torch.randint(118, 125, (E, D, I // 32), generator=g, dtype=torch.uint8)
    n_routed = E - 1
    n_ept = K - 1
    if n_ept > 0:
        if w.zipf is None:
            routed = torch.stack([torch.randperm(n_routed, generator=g)[:n_ept] for _ in range(T)])
        else:
            p = (torch.arange(n_routed, dtype=torch.float64) + 1.0) ** (-w.zipf)
            p = (p / p.sum()).expand(T, n_routed).contiguous()
            routed = torch.multinomial(p, n_ept, replacement=False, generator=g)
        routed = routed.to(torch.int32)
        rw = torch.softmax(torch.randn(T, n_ept, generator=g), dim=-1).to(torch.float32)
    else:
        routed = torch.zeros(T, 0, dtype=torch.int32)
        rw = torch.zeros(T, 0, dtype=torch.float32)
    shared = torch.full((T, 1), E - 1, dtype=torch.int32)
    topk_ids = torch.cat([routed, shared], dim=1).contiguous()
    topk_weights = torch.cat([rw, torch.ones(T, 1, dtype=torch.float32)], dim=1).contiguous()
    return {
        "hidden": hidden.contiguous(),
        "w13": w13,
        "w13_scale": w13_scale,
        "w2": w2,
        "w2_scale": w2_scale,
        "topk_ids": topk_ids,
        "topk_weights": topk_weights,
    }


def to_numpy(inp: dict) -> dict:
    """numpy views for the oracle: bf16 hidden as uint16 bit patterns."""
    return {
        "hidden_bits": inp["hidden"].view(torch.int16).numpy().view(np.uint16),
        "w13": inp["w13"].numpy(),
        "w13_scale": inp["w13_scale"].numpy(),
        "w2": inp["w2"].numpy(),
        "w2_scale": inp["w2_scale"].numpy(),
        "topk_ids": inp["topk_ids"].numpy(),
        "topk_weights": inp["topk_weights"].numpy(),
    }


def touched_experts(topk_ids, E: int) -> int:
    """Number of distinct expert ids in [0, E) that receive at least one route."""
    ids = np.asarray(topk_ids).reshape(-1)
    ids = ids[(ids >= 0) & (ids < E)]
    return int(np.unique(ids).shape[0])
