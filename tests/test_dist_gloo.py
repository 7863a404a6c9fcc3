"""Host-side multi-rank logic of the benchmark, on two gloo ranks (CPU only).

Decode shards by sequence: every rank decodes its own batch and no data crosses
ranks; the only exchange is the max of the per-rank times.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = [0.25, 0.4][rank]
    t_max = bench.max_over_ranks(t, dist)
    rate = bench.whole_job_rate(1e9, world, 10, t_max)
    q.put((rank, bench.rank_seed(rank), t_max, rate))
    dist.destroy_process_group()


def test_two_rank_aggregation_is_max_and_weak():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, t0, v0), (r1, s1, t1, v1) = res
    assert s0 != s1  # distinct batches per rank
    assert t0 == t1 == 0.4  # every rank reports the slowest rank's time
    assert v0 == v1 == pytest.approx(2 * 1e9 * 10 / 0.4 / 1e9)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(0.3, None) == 0.3
    assert bench.whole_job_rate(2e9, 1, 5, 1.0) == pytest.approx(10.0)
