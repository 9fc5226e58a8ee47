"""The multi-GPU path of bench.py is replicas only: each rank decodes its own batch
and the ranks exchange nothing but the barrier and the max of the timed region.  This
runs that host-side logic as two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 0.5 + 0.25 * rank          # rank 1 is the slower one
        steps = 40
        e_max = bench.max_over_ranks(elapsed, dist, "cpu")
        dist.barrier()
        out[rank] = (bench.replica_seed(7, rank), e_max, bench.job_throughput(steps, world, e_max))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_count_every_rank_steps():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    seeds = sorted(r[0] for r in res.values())
    assert seeds == [7, 1007]                     # distinct synthetic batches per rank
    for _, e_max, value in res.values():
        assert e_max == pytest.approx(0.75)        # the slowest rank's time
        assert value == pytest.approx(2 * 40 / 0.75)  # whole-job steps/s
