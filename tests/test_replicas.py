"""The N-replica harness of bench.py on CPU: two gloo ranks, each with its own
step time, agree on the slowest rank's time and on the whole-job value."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_init()
    ms = 2.0 + rank  # rank 1 is the slow one
    dist.barrier()
    worst = bench.max_over_ranks(ms, w)
    value = bench.job_tflops(1e12, w, worst)
    q.put((r, lr, w, worst, value))
    dist.destroy_process_group()


def test_two_replicas_aggregate_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, lr, w, worst, value) in enumerate(results):
        assert (r, lr, w) == (rank, rank, 2)
        assert worst == 3.0  # max over ranks
        assert value == pytest.approx(2e12 / 3e-3 / 1e12)  # both ranks' work / slowest time


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)
