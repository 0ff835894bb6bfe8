"""Expert-parallel dispatch and combine (mixture_experts_mxfp4_gb300.ep) with two
gloo ranks on the CPU.  Each rank holds its own tokens and the experts of its
contiguous range; the oracle stands in for each rank's local forward (one route
per row, topk = 1, which gives each route's fp32 row w * y exactly).  Every
rank's result must equal the single-device oracle forward of its tokens bit for
bit: the combine adds the same fp32 rows in the same ascending-k order."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads
from mixture_experts_mxfp4_gb300 import ep

CASES = [
    # T per rank, D, I, E, K
    (24, 256, 128, 9, 3),
    (16, 256, 128, 33, 9),
    (5, 128, 128, 3, 2),
]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _oracle_local(npi, first, count):
    def run(h, ids, w):
        hb = h.view(torch.int16).numpy().view(np.uint16)
        res = oracle.forward(hb, npi["w13"][first:first + count], npi["w13_scale"][first:first + count],
                             npi["w2"][first:first + count], npi["w2_scale"][first:first + count],
                             ids.numpy(), w.numpy(), want_h=False)
        return torch.from_numpy(res["out_f32"])
    return run


def _inputs(case, world, seed=0):
    T, D, I, E, K = case
    w = workloads.custom(T * world, D, I, E, K)
    inp = workloads.make_inputs(w, seed=seed)
    ids = inp["topk_ids"]
    ids[0, 0] = -1                 # an invalid id
    ids[1, :] = E + 3              # a token with no valid route
    if E >= 6:
        ids[2, :] = torch.arange(K, dtype=torch.int32) % 2 + E - 2  # all routes on the last rank's experts
    return inp


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for ci, case in enumerate(CASES):
            T, D, I, E, K = case
            inp = _inputs(case, world)
            npi = workloads.to_numpy(inp)
            first, count = ep.expert_ranges(E, world)[rank]
            sl = slice(rank * T, (rank + 1) * T)
            out = ep.ep_forward(inp["hidden"][sl].contiguous(), inp["topk_ids"][sl].contiguous(),
                                inp["topk_weights"][sl].contiguous(), E,
                                _oracle_local(npi, first, count))
            ref = oracle.forward(**npi, want_h=False)["out_bf16"][sl]
            got = out.view(torch.int16).numpy().view(np.uint16)
            np.testing.assert_array_equal(got, ref, err_msg=f"rank {rank} case {case}")
        open(os.path.join(out_dir, f"ok{rank}"), "w").write("ok")
    finally:
        dist.destroy_process_group()


def test_expert_ranges():
    assert ep.expert_ranges(257, 8) == [(0, 33)] + [(33 + 32 * i, 32) for i in range(7)]
    assert ep.expert_ranges(9, 2) == [(0, 5), (5, 4)]
    own = ep.expert_owner(9, 2)
    assert own.tolist() == [0, 0, 0, 0, 0, 1, 1, 1, 1]
    with pytest.raises(ValueError):
        ep.expert_ranges(2, 3)


def test_ep_two_gloo_ranks_match_single_device(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        assert (tmp_path / f"ok{r}").exists()
