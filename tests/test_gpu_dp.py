"""Batch split over ranks by whole sequences, on one GPU, through the C ABI.

The sequences of a batch are cut into uneven groups, one per emulated rank.
Each rank runs the distributed entropy quantile (its counts per pass; the
counts are summed over ranks here with torch on the same device, which is
the all-reduce a multi-rank run makes), its loss stage with the whole
batch's sequence count, and its backward; the summed batch sums give the
loss and metrics.  Everything is compared with the same steps run once on
the whole batch, and the loss with the fp64 oracle.
"""
import math

import numpy as np
import pytest
import torch

from lm_head_log_tma_gb300.workloads import GSPO_TOKEN, Workload

from parity import Case, cfg_of
from test_gpu_parity import MID

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_log_tma_gb300 import rlloss
    return rlloss


SPLITS = [
    (MID[2], [0, 2, 3, 5]),                 # entropy mask q = 0.2, tau = 0.7: three ranks
    (MID[1], [0, 1, 4]),                    # bias, K3 KL, asymmetric eps, {+1, -1, 0} advantages
    (MID[3], [0, 3, 6]),                    # GSPO-token
    (MID[2].with_(top_entropy_quantile=0.5, seed=131), [0, 4, 5]),
]


def _whole_and_split(R, spec, cuts):
    case = Case(spec)
    i = case.inp
    dev = "cuda"
    t = lambda x: None if x is None else x.to(dev)
    cfg = cfg_of(R, spec)
    X, W, b, tg = t(i.X), t(i.W), t(i.b), t(i.targets)
    old, ref, adv, mask = t(case.old), t(case.ref), t(i.adv), t(i.mask)
    fw = R.forward(cfg, X, W, b, tg)
    whole = R.loss_from_logp(cfg, fw["logp"], fw["entropy"], old, ref, adv, mask)

    T, Bg = spec.T, spec.B
    ranks = list(zip(cuts[:-1], cuts[1:]))
    rows = lambda x, a, e: None if x is None else x[a * T:e * T]
    q = spec.top_entropy_quantile
    use_mask = q < 1.0
    states = [R.alloc_select_state() for _ in ranks]
    thr = float("nan")
    if use_mask:
        for pass_ in range(R.SELECT_PASSES):
            counts = [R.entropy_hist(rows(fw["entropy"], a, e), rows(mask, a, e), pass_, st)
                      for (a, e), st in zip(ranks, states)]
            total = torch.stack(counts).sum(0, dtype=torch.int64).to(torch.int32)   # the all-reduce
            for st in states:
                R.entropy_select(pass_, total, q, st)
        torch.cuda.synchronize()
        thrs = [R.rlloss_select_threshold(st) for st in states]
        assert all(x == thrs[0] for x in thrs)
        thr = thrs[0]

    N = spec.N
    dlogp = torch.empty(N, device=dev)
    emask = torch.empty(N, dtype=torch.uint8, device=dev)
    sums = torch.zeros(R.NSUMS, dtype=torch.float64, device=dev)
    for (a, e), st in zip(ranks, states):
        cfg_r = cfg_of(R, spec.with_(B=e - a))
        o = R.loss_from_logp_dp(cfg_r, Bg, st if use_mask else None, rows(fw["logp"], a, e),
                                rows(fw["entropy"], a, e), rows(old, a, e), rows(ref, a, e), adv[a:e],
                                rows(mask, a, e))
        torch.cuda.synchronize()
        assert R.rlloss_get_device_status(o["workspace"]) == 0
        sums += o["sums"]                                                          # the all-reduce
        dlogp[a * T:e * T] = o["dlogp"]
        emask[a * T:e * T] = o["emask"]
    loss, metrics = R.rlloss_metrics_from_sums(cfg, Bg, sums.cpu().tolist(), thr)
    return case, cfg, (X, W, b, tg), fw, whole, dict(loss=loss, metrics=metrics, dlogp=dlogp, emask=emask,
                                                      thr=thr, ranks=ranks)


@pytest.mark.parametrize("spec,cuts", SPLITS, ids=["entropy_3ranks", "bias_k3kl_2ranks", "gspo_2ranks",
                                                   "entropy_q0.5_2ranks"])
def test_sequence_split_matches_whole_batch(R, spec, cuts):
    """Threshold and entropy mask bit for bit, counts exact, loss, other
    metrics and dL/dlogp to fp32 rounding of the whole-batch loss stage; the
    loss within 1e-5 of the fp64 oracle."""
    case, cfg, _, fw, whole, dp = _whole_and_split(R, spec, cuts)
    wm = whole["metrics"].cpu().tolist()
    if spec.top_entropy_quantile < 1.0:
        assert np.float32(dp["thr"]) == np.float32(wm[4])
        kept = int(dp["emask"].sum())
        assert 0 < kept < int(case.inp.mask.sum()), "the mask must drop some but not all tokens"
    else:
        assert math.isnan(dp["metrics"][4]) and math.isnan(wm[4])
    assert torch.equal(dp["emask"], whole["emask"])
    for k in (1, 3, 5):
        assert dp["metrics"][k] == wm[k], k
    for k in (0, 2, 6, 7):
        assert dp["metrics"][k] == pytest.approx(wm[k], rel=2e-6, abs=1e-7), k
    wl = whole["loss"].item()
    assert dp["loss"] == pytest.approx(wl, rel=2e-6, abs=1e-9)
    torch.testing.assert_close(dp["dlogp"], whole["dlogp"], rtol=2e-6, atol=1e-12)
    # the whole batch's loss against the oracle (the oracle's own threshold and mask)
    ol = case.loss().loss
    assert abs(dp["loss"] - ol) <= 1e-5 * abs(ol), (dp["loss"], ol)


def test_sequence_split_gradients_sum_to_whole_batch(R):
    """Each rank's backward over its rows (whole vocabulary): its dX rows are
    the whole batch's, and dW, db summed over ranks are the whole batch's."""
    spec, cuts = SPLITS[1]
    case, cfg, (X, W, b, tg), fw, whole, dp = _whole_and_split(R, spec, cuts)
    T = spec.T
    wbw = R.backward_shard(cfg, X, W, b, tg, 0, fw["lse"], whole["dlogp"])
    dW = torch.zeros_like(wbw["dW"])
    db = torch.zeros_like(wbw["db"])
    for a, e in dp["ranks"]:
        cfg_r = cfg_of(R, spec.with_(B=e - a))
        o = R.backward_shard(cfg_r, X[a * T:e * T], W, b, tg[a * T:e * T], 0, fw["lse"][a * T:e * T],
                             dp["dlogp"][a * T:e * T])
        torch.testing.assert_close(o["dX"], wbw["dX"][a * T:e * T], rtol=1e-4, atol=1e-9)
        dW += o["dW"]                                                              # the all-reduce
        db += o["db"]
    torch.cuda.synchronize()
    rel = lambda x, y: float((x - y).norm() / y.norm())
    assert rel(dW, wbw["dW"]) <= 1e-5
    assert rel(db, wbw["db"]) <= 1e-5


def test_distributed_quantile_with_an_empty_rank(R):
    """A rank whose tokens are all masked contributes empty counts; the
    threshold is still the whole batch's, and with no active token anywhere
    it is NaN."""
    spec = Workload("dp_empty_rank", B=3, T=64, H=64, V=300, dtype="bf16", top_entropy_quantile=0.3,
                    prompt_len=8, seed=132)
    case = Case(spec)
    mask = case.inp.mask.clone()
    mask[:spec.T] = 0                                  # rank 0 holds one sequence with no active token
    ent = torch.from_numpy(case.ent.astype(np.float32)).cuda()
    m = mask.cuda()
    for mm, expect_nan in ((m, False), (torch.zeros_like(m), True)):
        ranks = [(0, 1), (1, 3)]
        states = [R.alloc_select_state() for _ in ranks]
        for pass_ in range(R.SELECT_PASSES):
            counts = [R.entropy_hist(ent[a * spec.T:e * spec.T], mm[a * spec.T:e * spec.T], pass_, st)
                      for (a, e), st in zip(ranks, states)]
            total = torch.stack(counts).sum(0, dtype=torch.int64).to(torch.int32)
            for st in states:
                R.entropy_select(pass_, total, 0.3, st)
        torch.cuda.synchronize()
        thr = R.rlloss_select_threshold(states[0])
        if expect_nan:
            assert math.isnan(thr)
        else:
            import oracle as O
            othr, _ = O.entropy_threshold(ent.double().cpu().numpy(), mm.cpu().numpy(), 0.3)
            assert np.float32(thr) == np.float32(othr)
