"""The replicas path of the benchmark (N > 1 ranks, one workload per rank) on
CPU with the gloo backend, world size 2: the whole-job number must be the
slowest rank's time with every rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, gbs = bench.aggregate_ranks(times[rank], 1.0e9, dist, "cpu")
        out[rank] = (ms, gbs)
    finally:
        dist.destroy_process_group()


def test_replicas_take_max_time_and_sum_bytes():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    times = [2.0, 5.0]               # ms per step on rank 0 and rank 1
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, gbs = out[r]
        assert ms == 5.0                              # the slowest rank
        assert gbs == pytest.approx(2 * 1.0e9 / 5e-3 / 1e9)   # both ranks' bytes


def test_single_process_needs_no_group():
    ms, gbs = bench.aggregate_ranks(4.0, 2.0e9, None)
    assert ms == 4.0 and gbs == pytest.approx(500.0)
