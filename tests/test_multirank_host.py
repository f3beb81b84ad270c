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


# ---------------------------------------------------------------- batch split over ranks by sequences
def _keys(h32):
    """Order-preserving uint32 keys of fp32 values."""
    import numpy as np
    u = np.asarray(h32, np.float32).view(np.uint32)
    return np.where(u & np.uint32(0x80000000), ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def _key_value(k):
    import numpy as np
    k = np.uint32(k)
    u = (k & np.uint32(0x7fffffff)) if (k & np.uint32(0x80000000)) else ~k
    return float(np.array([u], np.uint32).view(np.float32)[0])


def _distributed_threshold(keys, q, allreduce):
    """The ranks' joint radix selection (four 8-bit passes) of the order
    statistics at (1-q)(n_act-1) of every rank's active keys: each pass
    counts the local keys under the current prefixes, the counts are summed
    over ranks, and every rank takes the same select step."""
    import math
    import numpy as np
    k, prefix, frac = [0, 0], [0, 0], 0.0
    for pass_ in range(4):
        shift = 24 - 8 * pass_
        d = ((keys >> shift) & 255).astype(np.int64)
        counts = np.zeros(512, np.int64)
        if pass_ == 0:
            counts[:256] = np.bincount(d, minlength=256)
        else:
            hp = keys >> (shift + 8)
            counts[:256] = np.bincount(d[hp == prefix[0]], minlength=256)
            counts[256:] = np.bincount(d[hp == prefix[1]], minlength=256)
        counts = allreduce(counts)
        if pass_ == 0:
            n = int(counts[:256].sum())
            if n == 0:
                return float("nan")
            pos = (1.0 - q) * (n - 1)
            lo = min(int(math.floor(pos)), n - 1)
            k, frac = [lo, min(lo + 1, n - 1)], pos - lo
        for j in range(2):
            h = counts[:256] if pass_ == 0 else counts[256 * j:256 * (j + 1)]
            cum, b = 0, 0
            while b < 255 and cum + h[b] <= k[j]:
                cum += int(h[b])
                b += 1
            k[j] -= cum
            prefix[j] = (prefix[j] << 8) | b
    vlo, vhi = _key_value(prefix[0]), _key_value(prefix[1])
    return vlo + frac * (vhi - vlo)


def _dp_rank_main(rank, world, port, out):
    """One rank of the sequence-split protocol with the oracle's arithmetic:
    the joint entropy threshold from summed counts, then this rank's loss
    share and batch sums (summed over ranks), finished by the library's
    host-only rlloss_metrics_from_sums."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle as O
    from lm_head_log_tma_gb300 import rlloss as R
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(9)
        B, T, q, beta = 5, 40, 0.2, 0.04
        N = B * T
        ent = rng.normal(4.0, 0.8, N).astype(np.float32)
        ent[7] = ent[11] = ent[3]                           # ties
        mask = (rng.random(N) > 0.25).astype(np.uint8)
        logp = rng.normal(-3.0, 1.0, N)
        old = logp + rng.normal(0, 0.3, N)
        ref = logp + rng.normal(0, 0.1, N)
        adv = np.array([1.0, -1.0, 0.0, 0.7, -0.4])
        cut = [0, 2, B]                                     # uneven: 2 and 3 sequences
        a, e = cut[rank], cut[rank + 1]
        sl = slice(a * T, e * T)

        def allreduce(x):
            t = torch.tensor(x, dtype=torch.float64 if x.dtype == np.float64 else torch.int64)
            dist.all_reduce(t)
            return t.numpy()

        thr = _distributed_threshold(_keys(ent[sl])[mask[sl] != 0], q, allreduce)
        othr, oe = O.entropy_threshold(ent.astype(np.float64), mask, q)
        my_e = ((mask[sl] != 0) & (ent[sl].astype(np.float64) >= thr)).astype(np.uint8)
        # this rank's share: its sequences' terms (oracle, mean over its own
        # sequences, times their count) and sums that add over ranks
        Br = e - a
        r = O.gmpo_loss(logp[sl], old[sl], ref[sl], adv[a:e], mask[sl], Br, T, 0.2, 0.3, beta=beta,
                        emask_override=my_e)
        n_i = (mask[sl].reshape(Br, T) != 0).sum(axis=1)
        nh = float((n_i > 0).sum())
        n_act = r.metrics[3]
        sums = np.array([r.loss * Br, n_act, r.metrics[1], r.metrics[2] * n_act, r.metrics[5],
                         r.metrics[6] * nh, r.metrics[7] * nh, nh])
        tot = allreduce(sums)
        cfg = R.make_cfg(B, T, eps_low=0.2, eps_high=0.3, beta=beta, top_entropy_quantile=q)
        loss, metrics = R.rlloss_metrics_from_sums(cfg, B, tot.tolist(), thr)
        full = O.gmpo_loss(logp, old, ref, adv, mask, B, T, 0.2, 0.3, beta=beta, entropy=ent, q=q)
        c_share = r.c * Br / B                              # dL/dlogp of the whole batch's loss
        ok = (thr == othr and np.array_equal(my_e, oe[sl])
              and np.float32(loss) == np.float32(full.loss)
              and np.allclose(metrics, np.float32(full.metrics), rtol=1e-6, equal_nan=True)
              and np.allclose(c_share, full.c[sl], rtol=1e-12, atol=1e-18))
        out.put((rank, bool(ok), float(thr), float(loss)))
    finally:
        dist.destroy_process_group()


def test_sequence_split_protocol_gloo_world2():
    """Two CPU ranks holding 2 and 3 of 5 sequences: the threshold from
    summed per-pass counts equals the whole batch's (the oracle's sort), the
    mask bits match, and the loss, metrics and dL/dlogp assembled from the
    ranks' sums equal the whole batch's."""
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_dp_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert all(ok for _, ok, _, _ in got), got
    assert got[0][2] == got[1][2] and got[0][3] == got[1][3]


def test_distributed_threshold_matches_sort_on_one_rank():
    """The selection with one rank (no exchange) on many shapes: ties, a
    single token, all equal, negative values, q at 0 and 1."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import oracle as O
    rng = np.random.default_rng(3)
    ident = lambda x: x
    for n, q in ((1, 0.2), (2, 0.5), (7, 0.0), (7, 1.0), (300, 0.37), (1000, 0.8), (64, 0.5)):
        h = rng.normal(0.5, 2.0, n).astype(np.float32)
        h[: n // 4] = h[0]
        if n == 64:
            h[:] = np.float32(1.25)
        thr = _distributed_threshold(_keys(h), q, ident)
        othr, _ = O.entropy_threshold(h.astype(np.float64), np.ones(n, np.uint8), q)
        assert thr == othr, (n, q, thr, othr)
