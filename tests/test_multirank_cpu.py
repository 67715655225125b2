"""The N > 1 path of the benchmark on CPU: two gloo ranks, each timing its
own replica; the job rate uses the slowest rank (weak scaling).  No GPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    my_ms = [120.0, 150.0][rank]  # rank 1 is the slow one
    slowest = bench.max_over_ranks(my_ms, device="cpu")
    rate = bench.job_throughput(1000, 10, world, slowest)
    dist.barrier()
    results[rank] = (slowest, rate)
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_whole_job_rate():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(2, port, results), nprocs=2, join=True)
        res = dict(results)
    assert res[0][0] == res[1][0] == 150.0
    # 2 ranks x 1000 units x 10 steps in 150 ms
    assert res[0][1] == pytest.approx(2 * 1000 * 10 / 0.150)


def test_single_process_passes_time_through():
    import bench

    assert bench.max_over_ranks(42.0) == 42.0
    assert bench.job_throughput(5, 4, 1, 1000.0) == pytest.approx(20.0)
