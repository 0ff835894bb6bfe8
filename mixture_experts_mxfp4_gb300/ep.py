"""Expert-parallel dispatch and combine around the single-GPU fused MoE forward.

The experts of a layer are split into contiguous ranges, one per rank (the
sparse 257-expert layer of the DeepSeek-style workloads over 8 GPUs gives ~32
experts per rank, the shape of the 33-expert dense-shard workload; the page
kernelbot-amd-moe-mxfp4-754773 contrasts such sparse and dense expert layers).
Each rank holds its own batch of tokens.  A forward on every rank:

1. dispatch: every route (t, k) whose expert id is in [0, E) goes to the rank
   that owns the expert, with the token's hidden row, the expert's local id and
   the top-k weight (routes travel in ascending route id t * topk + k);
2. local forward: the owning rank runs the fused forward over the routes it
   received, one route per row (topk = 1), and keeps each route's fp32 row
   w * (W2[e] . Q(bf16(silu(g) * u))) -- with the library these are the P rows
   of its workspace (`library_local_forward`);
3. combine: the rows go back to their tokens' ranks, which add each token's rows
   in ascending k in fp32 from zero and round once to bf16: the arithmetic and
   the order of the single-GPU forward, so the result equals it bit for bit.  On
   the GPU the library's top-k sum kernel does it (moe_mxfp4_topk_sum); with CPU
   tensors (gloo process groups) the same sum runs on the host.

Communication uses the torch.distributed collectives of the caller's process
group (all_to_all_single; NCCL for GPU tensors, gloo for CPU tensors).  Sending
each route's fp32 row makes the combine exact at topk * d_model * 4 bytes per
token; per-rank partial sums rounded to bf16 would move far fewer bytes but
round every partial, which the single-GPU result does not.
"""
from __future__ import annotations

from typing import Callable

import torch
import torch.distributed as dist


def expert_ranges(E: int, world: int):
    """Contiguous expert ranges [(first, count)] per rank; counts differ by at most
    one, the earlier ranks taking the extra experts."""
    if world < 1 or E < world:
        raise ValueError("need at least one expert per rank")
    base, extra = divmod(E, world)
    out, first = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((first, n))
        first += n
    return out


def expert_owner(E: int, world: int) -> torch.Tensor:
    """Owning rank of each expert id (int64 [E])."""
    own = torch.empty(E, dtype=torch.int64)
    for r, (f, n) in enumerate(expert_ranges(E, world)):
        own[f:f + n] = r
    return own


def _a2a(out: torch.Tensor, inp: torch.Tensor, out_splits, in_splits, group):
    dist.all_to_all_single(out, inp, list(out_splits), list(in_splits), group=group)


def ep_forward(hidden: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, E: int,
               local_forward: Callable, group=None) -> torch.Tensor:
    """Expert-parallel forward of this rank's tokens (see the module docstring).

    hidden bf16 [T, D]; topk_ids int32 [T, K] (global expert ids; ids outside
    [0, E) contribute nothing); topk_weights fp32 [T, K].  local_forward(h, ids, w)
    receives this rank's routes as rows (h bf16 [n, D], ids int32 [n, 1] local
    expert ids, w fp32 [n, 1]) and returns their fp32 rows w * y [n, D].  Returns
    bf16 [T, D].  All tensors on one device (CPU for gloo, CUDA for NCCL).
    """
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    dev = hidden.device
    T, D = hidden.shape
    K = topk_ids.shape[1]
    ranges = expert_ranges(E, world)
    first = torch.tensor([f for f, _ in ranges], dtype=torch.int64, device=dev)
    owner = expert_owner(E, world).to(dev)

    ids = topk_ids.reshape(-1).to(torch.int64)
    valid = (ids >= 0) & (ids < E)
    rid = torch.nonzero(valid).squeeze(1)                      # valid route ids, ascending
    dest = owner[ids[rid]]
    dest_sorted, order = torch.sort(dest, stable=True)          # by rank, ascending route id within
    rid_s = rid[order]
    send_counts = torch.bincount(dest_sorted, minlength=world).to(torch.int64)
    recv_counts = torch.empty_like(send_counts)
    _a2a(recv_counts, send_counts, [1] * world, [1] * world, group)
    sc = send_counts.cpu().tolist()
    rc = recv_counts.cpu().tolist()
    n_recv = sum(rc)

    # dispatch: hidden rows (bf16 pairs moved as 32-bit words), local expert ids, weights
    h_send = hidden[rid_s // K].contiguous()
    lid_send = (ids[rid_s] - first[dest_sorted]).to(torch.int32).contiguous()
    w_send = topk_weights.reshape(-1)[rid_s].contiguous()
    h_recv = torch.empty(n_recv, D, dtype=torch.bfloat16, device=dev)
    _a2a(h_recv.view(torch.int32), h_send.view(torch.int32), rc, sc, group)
    lid_recv = torch.empty(n_recv, dtype=torch.int32, device=dev)
    _a2a(lid_recv, lid_send, rc, sc, group)
    w_recv = torch.empty(n_recv, dtype=torch.float32, device=dev)
    _a2a(w_recv, w_send, rc, sc, group)

    # local forward over the received routes (this rank's experts: ranges[rank])
    if n_recv:
        rows = local_forward(h_recv, lid_recv.view(-1, 1), w_recv.view(-1, 1))
        rows = rows.to(torch.float32).contiguous()
        assert rows.shape == (n_recv, D)
    else:
        rows = torch.empty(0, D, dtype=torch.float32, device=dev)

    # combine: rows back to their routes' ranks, by route id
    back = torch.empty(len(rid_s), D, dtype=torch.float32, device=dev)
    _a2a(back, rows, sc, rc, group)
    P = torch.zeros(T * K, D, dtype=torch.float32, device=dev)
    P[rid_s] = back
    if dev.type == "cuda":
        import mixture_experts_mxfp4_gb300 as moe

        route_pos = torch.where(valid, 0, -1).to(torch.int32)  # >= 0: the route counts
        out = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
        return moe.topk_sum(P, route_pos, out)
    P = P.view(T, K, D)
    vk = valid.view(T, K)
    acc = torch.zeros(T, D, dtype=torch.float32, device=dev)
    for k in range(K):  # ascending k, fp32, invalid routes skipped
        acc = torch.where(vk[:, k:k + 1], acc + P[:, k], acc)
    return acc.to(torch.bfloat16)


def library_local_forward(w13: torch.Tensor, w13_scale: torch.Tensor, w2: torch.Tensor,
                          w2_scale: torch.Tensor, first: int, count: int):
    """local_forward for ep_forward on a GPU: this rank's experts [first,
    first + count) of the full weights (device tensors), run by the library with
    one route per row; returns the fp32 rows w * y (the workspace P rows)."""
    import mixture_experts_mxfp4_gb300 as moe

    lw13, ls13 = w13[first:first + count], w13_scale[first:first + count]
    lw2, ls2 = w2[first:first + count], w2_scale[first:first + count]
    I = lw13.shape[1] // 2
    D = lw13.shape[2] * 2

    def run(h, ids, w):
        n = h.shape[0]
        m = moe.MoeMXFP4(n, D, I, count, 1, device=h.device)
        m.forward(h.contiguous(), lw13, ls13, lw2, ls2, ids.contiguous(), w.contiguous())
        torch.cuda.synchronize(h.device)
        if m.device_status() != 0:
            raise RuntimeError("device status after the local forward")
        return m.region("P", torch.float32, (n, D)).clone()

    return run
