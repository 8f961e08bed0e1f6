"""The multi-rank path of the benchmark on CPU: two gloo ranks, each timing its own replica;
the job's time is the slowest rank's and its value counts both replicas (weak scaling)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]                          # rank 1 is the slower one
    bench.barrier(world)
    slowest = bench.max_over_ranks(ms, world)
    value = bench.job_value(1e9, world, slowest, 1e9)   # 1 GB per rank
    out[rank] = (slowest, value)
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_both_replicas():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    slowest, value = res[0]
    assert slowest == 5.0
    assert value == pytest.approx(2 * 1e9 / 5e-3 / 1e9)   # 400 GB/s for 2 GB in 5 ms


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_value(2e9, 1, 10.0, 1e9) == pytest.approx(200.0)
