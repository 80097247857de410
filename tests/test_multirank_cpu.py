"""The multi-rank host logic of bench.py on CPU ranks (gloo, world size 2).

With N GPUs every rank runs its own copy of the workload (the (sequence, head)
chains are independent problems: no data-path collective); the only cross-rank
steps are the barriers around the timed region and the max over ranks of the
measured times, from which the whole-job throughput is computed.
"""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    # rank r "measured" (10 + r) ms and (4 + 2r) ms: everyone must see the maxima
    elapsed, kernel = bench.max_over_ranks([10.0 + rank, 4.0 + 2 * rank], dist)
    value = bench.job_throughput(world, 524288, 50, elapsed * 50 / 1e3)
    dist.barrier()
    q.put((rank, elapsed, kernel, value))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, PORT, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, elapsed, kernel, value in res:
        assert elapsed == 11.0 and kernel == 6.0
        assert value == pytest.approx(2 * 524288 / 11e-3)


PORT = _free_port()


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_throughput(1, 1000, 10, 2.0) == 5000.0
