"""The N > 1 path of bench.py on CPU: world_size-2 gloo process group.

The SGEMM problem is run as independent replicas, one per GPU, with no collective on the
data path. What the multi-rank run adds is host logic: a barrier around the timed region and
the max over ranks of the elapsed time, from which the whole-job throughput is computed.
These tests exercise exactly that logic (bench.Dist) with two CPU ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist()
    try:
        assert d.world == world and d.rank == rank
        d.barrier()
        t_max = d.max(times[rank])
        # whole-job throughput: every rank's work over the slowest rank's time
        value = bench.replica_throughput(1e12, 10, d.world, t_max)
        d.barrier()
        out.put((rank, t_max, value))
    finally:
        d.close()


def test_two_rank_barrier_and_max_timing():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [1.25, 2.5]
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(out.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [2.5, 2.5]          # every rank sees the slowest time
    assert res[0][2] == pytest.approx(1e12 * 10 * 2 / 2.5 / 1e12)  # TFLOP/s, whole job
    assert res[0][2] == res[1][2]


def test_single_process_dist_is_noop():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    d = bench.Dist()
    assert d.world == 1 and d.pg is None
    assert d.max(3.5) == 3.5
    d.barrier()
    assert bench.replica_throughput(2e12, 4, 1, 2.0) == pytest.approx(4.0)
