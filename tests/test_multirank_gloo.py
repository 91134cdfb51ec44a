"""Multi-rank host logic on CPU: two gloo ranks (127.0.0.1).

* The benchmark: every rank runs its own copy of the workload (weak scaling,
  no collective in the data path); the job time is the maximum over ranks and
  the whole-job throughput counts every rank's bytes.
* The optional sequence-split sharding: ranks attend disjoint parts of one
  sequence, all-gather their partial (O, LSE) - the one exchange step - and
  LSE-merge them into the whole sequence's result (float64 oracle).
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


def _split_worker(rank, world, port, q):
    """Rank r attends its share of one sequence's entries (the optional
    sequence-split sharding: rank 0 the first half of the global tokens, rank 1
    the rest plus the window), the partial (O, LSE) pairs are all-gathered -
    the path's one exchange - and every rank LSE-merges them."""
    import numpy as np
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import workloads as W
        from oracle import attention as A
        from oracle import cache as C
        from oracle import formats as F
        wl = W.make_dense("split", 41, 1, 8, 128, [300])
        ts, tw = C.tensor_scales(wl)
        Kp, Vp = C.fill_pages(wl, ts, ts)
        K = C.dequant_seq(wl, Kp, ts, 0, 300)
        V = C.dequant_seq(wl, Vp, ts, 0, 300)
        kw, vw = C.window_codes(wl, tw, tw, 0)
        Kw, Vw = F.fp8_dequantize(kw, tw), F.fp8_dequantize(vw, tw)
        qv = F.bf16_to_f64(wl.q_bits_seq(0))
        scale = 1.0 / np.sqrt(128)
        if rank == 0:
            O, L = A.segment(qv, K[:150], V[:150], scale)
        else:
            O, L = A.segment(qv, np.concatenate([K[150:], Kw]), np.concatenate([V[150:], Vw]), scale)
        mine = torch.from_numpy(np.concatenate([O, L[:, None]], 1))
        parts = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)
        p0, p1 = parts[0].numpy(), parts[1].numpy()
        Om, Lm = A.merge(p0[:, :-1], p0[:, -1], p1[:, :-1], p1[:, -1])
        Of, Lf = A.decode(qv, K, V, Kw, Vw, scale)
        q.put((rank, float(np.abs(Om - Of).max()), float(np.abs(Lm - Lf).max())))
    finally:
        dist.destroy_process_group()


def test_sequence_split_exchange_two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_split_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    for rank, eo, el in sorted(q.get(timeout=5) for _ in range(world)):
        assert eo < 1e-12 and el < 1e-12, (rank, eo, el)
