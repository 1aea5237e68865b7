"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): each
rank draws its own batch, and the job-level numbers are the slowest rank's
time with the units of every rank summed."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    wl = bench.rank_workload("tiny", rank)
    times, units = bench.combine_ranks([10.0 + 5 * rank, 3.0 - rank], [100.0 * (rank + 1), 2.0],
                                       world, torch.device("cpu"))
    q.put((rank, times, units, wl.q.float().sum().item(), wl.seed))
    dist.destroy_process_group()


def test_two_ranks_combine_max_time_and_sum_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, units, _, _ in res:
        assert times == [15.0, 3.0]          # max over ranks
        assert units == [300.0, 4.0]         # summed over ranks
    assert res[0][4] != res[1][4]            # distinct seeds
    assert res[0][3] != res[1][3]            # distinct batches


def test_single_rank_combine_is_identity():
    import bench

    times, units = bench.combine_ranks([1.5], [7.0], 1, torch.device("cpu"))
    assert times == [1.5] and units == [7.0]
