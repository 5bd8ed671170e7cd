"""The benchmark's multi-rank arithmetic on two CPU ranks (gloo): every rank
reports the slowest rank's step time, and the job's throughput counts every
rank's tokens (weak scaling: each rank runs its own replica of the workload)."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier()
    ms_rank = [120.0, 200.0][rank]           # rank 1 is the slow one
    ms_step, value = bench.aggregate(ms_rank, 100, 16, world)
    q.put((rank, ms_step, value, bench.reduce_max(float(rank))))
    dist.destroy_process_group()


def test_two_ranks_report_the_slowest_and_sum_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms_step, value, mx in got:
        assert ms_step == pytest.approx(2.0)             # 200 ms / 100 steps, on both ranks
        assert value == pytest.approx(2 * 16 / 2e-3)    # both ranks' tokens over the slowest time
        assert mx == 1.0


def test_single_process_is_the_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.aggregate(50.0, 10, 16, 1) == (5.0, 16 / 5e-3)
