"""The bench's multi-rank host logic on CPU: two gloo ranks, no GPU.

Each rank runs its own independent decode problem in the real benchmark (no
data exchange); the only cross-rank steps are the barriers and the max over
ranks of the timed region, which these ranks exercise here."""
import os
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup()
        bench.barrier(w)
        ms = 10.0 + 5.0 * r                        # rank r "took" 10 + 5r ms
        slowest = bench.max_over_ranks(ms, w)
        value = bench.weak_scaling_value(1e9, w, 4, slowest)
        q.put((r, w, local, slowest, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_take_the_slowest_time(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for r, w, local, slowest, value in res:
        assert w == world and local == r
        assert slowest == 10.0 + 5.0 * (world - 1)
        # all ranks' bytes (world x 4 steps x 1 GB) over the slowest rank's time
        assert abs(value - world * 4 * 1e9 / (slowest * 1e-3) / 1e9) < 1e-9
