"""The N > 1 host path of bench.py on CPU ranks (gloo, world size 2).

The library runs one GPU per process and the path is run as independent
replicas (no data-path collective), so what crosses ranks is the timing:
the whole job's time is the slowest rank's, and the rate counts every
rank's units.  Ranks are spawned processes with a TCP rendezvous on
127.0.0.1.
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


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) * 10 ms: the job took the slowest rank's 20 ms
        t = bench.max_over_ranks((rank + 1) * 10.0, "cpu")
        rate = bench.whole_job_rate(4096, world, 5, t / 1e3)
        out.put((rank, t, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rate_gloo_world2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, rate in got:
        assert t == 20.0
        assert rate == pytest.approx(4096 * 2 * 5 / 0.020)


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(10, 1, 2, 4.0) == 5.0
