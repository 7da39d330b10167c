"""Host logic of the multi-rank bench path on CPU: two gloo ranks run
independent replicas; the job time is the slowest rank's and the throughput
counts every rank's tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 100.0 + 50.0 * rank          # rank 1 is the slower replica
    worst = bench.max_over_ranks(local_ms, world, "cpu")
    out[rank] = (worst, bench.job_throughput(4096, world, 10, worst))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_rank_replicas_take_the_slowest_rank(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    worst, tput = res[0]
    assert worst == 150.0
    assert tput == pytest.approx(world * 4096 * 10 / 0.150)


def test_single_rank_needs_no_collective():
    import bench
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.job_throughput(4096, 1, 100, 500.0) == pytest.approx(4096 * 100 / 0.5)
