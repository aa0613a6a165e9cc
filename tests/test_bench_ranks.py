"""Rank aggregation of bench.py on CPU: world_size-2 gloo process group.

The bench runs one replica per GPU (the path has no exchange step); its
reported value is the bytes of all ranks over the slowest rank's step time.
These tests run that host logic with two gloo ranks on 127.0.0.1. The last
test checks that the committed ncu traffic record still matches the decode
kernel's sources.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(times[rank])
        v = bench.whole_job_value(world, 1e9, t)
        out.put((rank, t, v))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [0.004, 0.005]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == pytest.approx(0.005)            # every rank sees the slowest time
        assert v == pytest.approx(2 * 1e9 / 0.005 / 1e9)


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.whole_job_value(1, 2e9, 0.5) == pytest.approx(4.0)


@pytest.mark.parametrize("launch", ["gate+up", "down"])
def test_traffic_record_matches_kernel_sources(launch):
    """The committed ncu traffic record still hashes to the decode kernel's
    sources (a changed kernel needs a new capture) and reads close to the
    algorithmic bytes."""
    sys.path.insert(0, ROOT)
    import bench
    t = bench.load_traffic("k_moe_tma " + launch, 1e8)
    assert t is not None, "profiles/traffic.json is stale for the decode kernel"
    assert 1.0 <= t / 1e8 < 1.2
