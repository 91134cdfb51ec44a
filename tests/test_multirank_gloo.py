"""The benchmark's multi-rank host logic on CPU: two gloo ranks (127.0.0.1).

Every rank runs its own copy of the workload (weak scaling, no collective in
the data path); the job time is the maximum over ranks and the whole-job
throughput counts every rank's bytes.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        # rank r was slower by r milliseconds
        ms, kern = bench.max_over_ranks([1.0 + rank, 0.5 + 0.25 * rank], world, "cpu")
        dist.barrier()
        q.put((rank, ms, kern, bench.job_gbs(1e9, ms, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms, kern, gbs in got:
        assert ms == 2.0 and kern == 0.75          # the slowest rank sets the job time
        assert gbs == pytest.approx(2e9 / 2e-3 / 1e9)   # both ranks' bytes over the max time


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1, "cpu") == [1.5, 2.5]
    assert bench.job_gbs(2e9, 1.0, 1) == pytest.approx(2000.0)
