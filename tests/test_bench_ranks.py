"""The replica aggregation bench.py uses with N > 1 (one process per GPU, no
data-path collective): the slowest rank's time is reported and the value
counts every rank's tokens. Checked with two gloo ranks on the CPU."""

import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = bench.slowest_rank(0.5 + rank, world, torch.device("cpu"))  # rank 1 is slower
    out[rank] = (ms, bench.whole_job_tokens_per_s(world, ms))
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time_and_all_tokens():
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        got = dict(out)
    for r in (0, 1):
        ms, tok_s = got[r]
        assert ms == pytest.approx(1.5)
        assert tok_s == pytest.approx(2 * 1000.0 / 1.5)


def test_one_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.slowest_rank(0.25, 1, torch.device("cpu")) == 0.25
    assert bench.whole_job_tokens_per_s(1, 0.5) == pytest.approx(2000.0)
