"""Multi-rank host paths on CPU ranks (gloo, world size 2).

bench.py runs the path as independent replicas (no data-path collective),
so what crosses ranks there is the timing: the whole job's time is the
slowest rank's, and the rate counts every rank's units.  The
vocabulary-parallel form exchanges row states and dX parts; its protocol is
run here with the oracle's arithmetic on each rank.  Ranks are spawned
processes with a TCP rendezvous on 127.0.0.1.
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


def _vocab_rank_main(rank, world, port, out):
    """One rank of the vocabulary-parallel protocol: this rank holds W rows
    [v0, v1); it gathers every rank's row states, runs the (replicated) loss
    stage, and all-reduces its dX part.  The arithmetic is the oracle's."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle as O
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(5)
        B, T, H, V, tau = 3, 6, 8, 70, 0.9
        N = B * T
        X = rng.standard_normal((N, H)); W = rng.standard_normal((V, H)) * 0.4
        b = rng.standard_normal(V) * 0.1; y = rng.integers(0, V, N)
        mask = (rng.random(N) > 0.2).astype(np.uint8); adv = np.array([1.0, -0.7, 0.4])
        prob = O.Problem(B, T, O.GMPO, 0.2, 0.3, 0.0, tau)
        _, lp0, _ = O.row_stats(X, W, b, y, tau)
        old = lp0 + rng.normal(0, 0.2, N)
        cut = [0, 29, V]                       # uneven shards
        v0, v1 = cut[rank], cut[rank + 1]
        st = O.shard_state(X, W[v0:v1], b[v0:v1], y, tau, v0)
        mine = torch.tensor(np.stack([st["m"], st["s"], st["w"], st["zy"]], axis=1))
        got = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)
        states = [dict(m=g[:, 0].numpy(), s=g[:, 1].numpy(), w=g[:, 2].numpy(), zy=g[:, 3].numpy()) for g in got]
        lse, logp, ent = O.merge_states(states, y, V)
        res = O.loss_stage(prob, logp, ent, old, None, adv, mask)
        dx, dw, db = O.shard_grads(X, W[v0:v1], b[v0:v1], y, tau, v0, lse, res.c)
        dxt = torch.tensor(dx)
        dist.all_reduce(dxt)
        ref = O.fwd_bwd(prob, X, W, b, y, old, None, adv, mask)
        ok = (abs(res.loss - ref["loss"]) <= 1e-12 * abs(ref["loss"])
              and np.allclose(dxt.numpy(), ref["dX"], rtol=1e-11, atol=1e-15)
              and np.allclose(dw, ref["dW"][v0:v1], rtol=1e-11, atol=1e-15)
              and np.allclose(db, ref["db"][v0:v1], rtol=1e-11, atol=1e-15))
        out.put((rank, bool(ok), float(res.loss)))
    finally:
        dist.destroy_process_group()


def test_vocab_parallel_protocol_gloo_world2():
    """The vocabulary-parallel exchange (all-gather of row states, replicated
    loss, all-reduce of dX parts) on two CPU ranks reproduces the whole
    vocabulary's loss and gradients, and both ranks hold the same loss."""
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_vocab_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert all(ok for _, ok, _ in got)
    assert got[0][2] == got[1][2]


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(10, 1, 2, 4.0) == 5.0
