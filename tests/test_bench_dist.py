"""The bench's multi-rank path on CPU: two gloo ranks agree on the slowest
rank's time and on the whole-job throughput (no GPU needed)."""
import os
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, _ = bench.dist_env()
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)
    mine = 10.0 + 5.0 * rank           # ms of this rank's timed region
    slowest = bench.max_over_ranks(mine, ws, torch.device("cpu"))
    value = bench.aggregate(slowest, steps=4, units_per_step_per_rank=64, world=ws)
    results[rank] = (slowest, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    port = 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        slowest, value = results[r]
        assert slowest == 15.0
        assert abs(value - 64 * 4 * 2 / 0.015) < 1e-6
