"""Host logic of the N > 1 benchmark path (independent replicas, no
collective in the step): the slowest rank's time is what every rank reports,
and throughput counts all replicas.  Two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is slower
        got = bench.max_over_ranks(ms, world, torch.device("cpu"))
        out[rank] = (got, bench.replica_throughput(1_000_000, world, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_slowest_time_and_total_throughput():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, tput = res[0]
    assert ms == 15.0
    assert tput == pytest.approx(2 * 1_000_000 / 0.015)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.replica_throughput(8_030_261_248, 1, 20.0) == pytest.approx(8_030_261_248 / 0.02)
