"""Host logic of bench.py's multi-rank path, run as two gloo ranks on the CPU.

Every rank runs its own replica of the workload. The timed region ends in a barrier, and the time
reported is the maximum over ranks. The value is the whole job's units divided by that maximum.
"""

import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    bench.barrier()
    slowest = bench.max_over_ranks(times[rank])
    value = bench.whole_job_rate(1000, w, slowest)
    out[rank] = (r, w, local, slowest, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_the_whole_job_rate():
    port = 29500 + os.getpid() % 2000
    times = [0.5, 2.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, times, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        r, w, local, slowest, value = res[rank]
        assert (r, w, local) == (rank, 2, rank)
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(1000 * 2 / 2.0)


def test_single_process_helpers_are_identities(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.whole_job_rate(500, 1, 0.5) == 1000.0
