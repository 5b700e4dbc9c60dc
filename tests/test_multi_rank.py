"""Host logic of the multi-GPU benchmark path with two gloo ranks on CPU:
each rank solves its own batch (weak scaling), the job time is the slowest
rank's and the job throughput counts every rank's problems."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank               # rank 1 is slower
    t, total = bench.aggregate(ms, 32768, world, dist, "cpu")
    seeds = [None] * world
    dist.all_gather_object(seeds, bench.rank_seed(rank))
    out[rank] = (t, total, seeds)
    dist.destroy_process_group()


def test_two_rank_aggregate_and_distinct_batches():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    for rank in range(world):
        t, total, seeds = res[rank]
        assert t == 15.0                  # max over ranks
        assert total == 2 * 32768         # every rank's problems count
        assert len(set(seeds)) == world   # ranks solve different batches


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.aggregate(3.5, 100, 1) == (3.5, 100)
