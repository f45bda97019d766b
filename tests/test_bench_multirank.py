"""The benchmark's multi-rank path on CPU: two gloo ranks, replicas with no
collective on the data path; the step time is the max over ranks and the
job throughput counts every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, torch.device("cpu"))
        out[rank] = (ms, bench.job_throughput(1e12, world, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms, tf = out[r]
        assert ms == pytest.approx(15.0)           # the slower rank decides
        assert tf == pytest.approx(2 * 1e12 / 15e-3 / 1e12)  # both ranks' work counts


def test_single_rank_passthrough():
    import bench

    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.job_throughput(2e12, 1, 1000.0) == pytest.approx(2.0)
