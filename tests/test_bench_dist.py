"""The benchmark's multi-process path on CPU: two gloo ranks exercise the
max-over-ranks timing and the whole-job aggregation that bench.py uses under
torchrun (replicas only: each rank runs its own forward, no exchange step)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, seconds, q):
    import torch.distributed as dist

    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        slowest = bench.max_over_ranks(seconds[rank], world)
        value = bench.aggregate_value(16 * 100, world, slowest)
        dist.barrier()
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_and_whole_job_value(world):
    port = _free_port()
    seconds = [0.0125, 0.0150][:world]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, seconds, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, value in got:
        assert slowest == max(seconds)
        # units of all ranks divided by the slowest rank's time
        assert value == pytest.approx(16 * 100 * world / max(seconds))


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.aggregate_value(1600, 1, 0.01) == pytest.approx(160000.0)
