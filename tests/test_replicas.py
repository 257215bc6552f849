"""Multi-process path of the benchmark (replicas, no data-path collective):
two CPU ranks over gloo check the aggregation bench.py applies under
torchrun -- the job's time is the slowest rank's, the job's rate counts the
work of every rank."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench._dist()
    # rank-dependent local timings: rank 1 is slower on the first value,
    # rank 0 on the second
    vals = bench._max_over_ranks([1.0 + rank, 5.0 - rank], torch.device("cpu"))
    rate = bench._job_rate(1e9, vals[0], ws)
    q.put((r, ws, local, vals, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_aggregation_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, (r, ws, local, vals, rate) in enumerate(res):
        assert (r, ws, local) == (rank, 2, rank)
        assert vals == [2.0, 5.0]          # max over ranks, element-wise
        # 1e9 bytes per rank, 2 ranks, 2 ms: 1 TB/s for the whole job
        assert rate == pytest.approx(1.0)


def test_single_process_values_pass_through():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench._job_rate(2e9, 1.0, 1) == pytest.approx(2.0)
