"""Multi-process path of bench.py on CPU (gloo, world size 2).

GDPA shards as independent replicas (one per GPU, no collective on the data
path); the only cross-rank operations are the max-over-ranks step time and
the whole-job throughput derived from it. Both are exercised here with two
gloo ranks on the host.
"""

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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_ms = [120.0, 150.0][rank]  # rank 1 is the slowest replica
        slowest = bench.reduce_max(per_rank_ms, dist)
        value = bench.replica_throughput(1e12, 10, world, slowest)
        out[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_throughput():
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    slowest, value = res[0]
    assert slowest == 150.0
    # 2 replicas x 10 steps x 1e12 FLOP in 150 ms -> 133.33 TFLOP/s for the whole job
    assert value == pytest.approx(2 * 10 * 1e12 / 0.150 / 1e12)


def test_single_process_reduce_is_identity():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.replica_throughput(2e12, 5, 1, 1000.0) == pytest.approx(10.0)
