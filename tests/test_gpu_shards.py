"""Vocabulary-parallel form of the path on one GPU, through the C ABI.

W (and b) are cut into contiguous vocabulary shards of uneven sizes; each
shard's forward yields a row state, the states of all shards give the loss
and dL/dlogp, and each shard's backward gives its dW / db rows and its part
of dX.  The exchanges a multi-rank run makes (gather the states, sum the dX
parts) are done here with torch on the same device.  Everything is checked
against the fp64 oracle of the whole vocabulary and against the single-call
path.
"""
import numpy as np
import pytest
import torch

from lm_head_log_tma_gb300.workloads import GSPO_TOKEN, Workload

from parity import (Case, cfg_of, check_grads, check_loss_and_metrics, check_rows, reconcile_loss)
from test_gpu_parity import MID

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_log_tma_gb300 import rlloss
    return rlloss


def _shard_cfg(R, spec, V, **kw):
    cfg = cfg_of(R, spec, **kw)
    cfg.V = V
    return cfg


def _cuts(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(int)


def run_shards(R, case, sizes, bwd_flags=0, accumulate_dx=False, drop=()):
    """Steps 1-3 over shards of the given sizes; shards listed in drop are
    left out of the states (their vocabulary is then missing)."""
    spec, i = case.spec, case.inp
    assert sum(sizes) == spec.V
    cut = _cuts(sizes)
    dev = "cuda"
    X, W, tg = i.X.to(dev), i.W.to(dev), i.targets.to(dev)
    b = None if i.b is None else i.b.to(dev)
    shards = [(int(cut[k]), int(sizes[k])) for k in range(len(sizes))]
    states = []
    for k, (v0, vs) in enumerate(shards):
        if k in drop:
            continue
        Wk = W[v0:v0 + vs].contiguous()
        bk = None if b is None else b[v0:v0 + vs].contiguous()
        st, ws = R.forward_shard(_shard_cfg(R, spec, vs), X, Wk, bk, tg, v0)
        assert R.rlloss_get_device_status(ws) == 0
        states.append(st)
    states = torch.stack(states).contiguous()
    t = lambda x: None if x is None else x.to(dev)
    out = R.loss_from_shards(cfg_of(R, spec), states, tg, t(case.old), t(case.ref), t(i.adv), t(i.mask))
    torch.cuda.synchronize()
    out["status"] = R.rlloss_get_device_status(out["workspace"])
    out["states"] = states
    if drop:
        return out
    dX = torch.zeros(spec.N, spec.H, dtype=torch.float32, device=dev)
    dWs, dbs = [], []
    for k, (v0, vs) in enumerate(shards):
        Wk = W[v0:v0 + vs].contiguous()
        bk = None if b is None else b[v0:v0 + vs].contiguous()
        flags = bwd_flags | (R.FLAG_ACCUMULATE if accumulate_dx and k > 0 else 0)
        cfg = _shard_cfg(R, spec, vs, flags=flags)
        outs = dict(dX=dX if accumulate_dx else torch.empty_like(dX),
                    dW=torch.empty(vs, spec.H, dtype=torch.float32, device=dev),
                    db=None if bk is None else torch.empty(vs, dtype=torch.float32, device=dev))
        if accumulate_dx and k > 0:
            outs["dW"].zero_()
            if outs["db"] is not None:
                outs["db"].zero_()
        o = R.backward_shard(cfg, X, Wk, bk, tg, v0, out["lse"], out["dlogp"], outputs=outs)
        torch.cuda.synchronize()
        assert R.rlloss_get_device_status(o["workspace"]) == 0
        if not accumulate_dx:
            dX += o["dX"]
        dWs.append(o["dW"])
        dbs.append(o["db"])
    out["dX"] = dX
    out["dW"] = torch.cat(dWs)
    out["db"] = None if b is None else torch.cat(dbs)
    return out


SHARDED = [
    (MID[0], [400, 350, 250]),
    (MID[1], [300, 250, 227]),
    (MID[2], [650, 650]),
    (MID[3], [1, 599]),
    (MID[4], [100, 300, 115]),
    (Workload("many_shards", B=2, T=100, H=64, V=2000, dtype="bf16", prompt_len=5, seed=131),
     [256, 255, 257, 1, 511, 720]),
]


@pytest.mark.parametrize("spec,sizes", SHARDED, ids=[s.name for s, _ in SHARDED])
def test_vocab_shards_match_oracle(R, spec, sizes):
    case = Case(spec)
    out = run_shards(R, case, sizes)
    assert out["status"] == 0, hex(out["status"])
    check_rows(out, case)
    lse = out["lse"].double().cpu().numpy()
    assert np.all(np.abs(lse - case.lse) <= 2e-5 + 2e-6 * np.abs(case.lse))
    res = reconcile_loss(out, case)
    check_loss_and_metrics(out, case, res)
    dl = out["dlogp"].double().cpu().numpy()
    c = res.c
    assert np.all(np.abs(dl - c) <= 1e-5 * np.abs(c).max() + 1e-12)
    check_grads(out, case, res)


@pytest.mark.parametrize("spec", [MID[1], MID[4]], ids=["bf16_bias_k3kl", "fp32_bias"])
def test_one_shard_forward_is_bit_identical_to_scoring(R, spec):
    """A single shard over the whole vocabulary merges the same partial
    states in the same order as the scoring call: lse, logp and entropy
    come out with the same bits."""
    case = Case(spec)
    out = run_shards(R, case, [spec.V])
    i = case.inp
    b = None if i.b is None else i.b.cuda()
    ref = R.forward(cfg_of(R, spec), i.X.cuda(), i.W.cuda(), b, i.targets.cuda())
    torch.cuda.synchronize()
    for k in ("logp", "entropy", "lse"):
        assert torch.equal(out[k].view(torch.int32), ref[k].view(torch.int32)), k


@pytest.mark.parametrize("spec,sizes", [SHARDED[1], SHARDED[4]], ids=["bf16_bias_k3kl", "fp32_bias"])
def test_vocab_shards_agree_with_single_call(R, spec, sizes):
    """The sharded path and rlloss_fwd_bwd agree: loss to 1e-6, per-token
    values to a few fp32 ulps, gradients to fp32 summation order (against the
    single call's recomputing backward, which the shard backward also runs;
    the single call's default, stored-probability backward rounds elsewhere
    and is checked against the oracle in the parity tests)."""
    case = Case(spec)
    a = run_shards(R, case, sizes)
    b = case.run_gpu(R, flags=R.FLAG_RECOMPUTE)
    assert abs(a["loss"].item() - b["loss"].item()) <= 1e-6 * abs(b["loss"].item()) + 1e-9
    for k in ("logp", "entropy"):
        assert torch.allclose(a[k], b[k], rtol=1e-6, atol=1e-5), k
    for k in ("dX", "dW", "db"):
        if b.get(k) is None:
            continue
        x, y = a[k], b[k]
        assert torch.allclose(x, y, rtol=1e-3, atol=2e-3 * float(y.abs().max())), k


def test_dx_parts_accumulate_in_place(R):
    """Summing the shards' dX parts with RLLOSS_FLAG_ACCUMULATE into one
    buffer gives the torch sum of the parts, bit for bit (one fp32 addition
    per element per shard, in shard order)."""
    spec, sizes = SHARDED[1]
    case = Case(spec)
    a = run_shards(R, case, sizes)
    b = run_shards(R, case, sizes, accumulate_dx=True)
    assert torch.equal(a["dX"], b["dX"])
    assert torch.equal(a["dW"], b["dW"])


def test_dense_shard_backward_matches_compacted(R):
    spec, sizes = SHARDED[0]
    case = Case(spec)
    a = run_shards(R, case, sizes)
    b = run_shards(R, case, sizes, bwd_flags=R.FLAG_ALL_ROWS)
    for k in ("dX", "dW"):
        y = b[k]
        assert torch.allclose(a[k], y, rtol=1e-4, atol=1e-5 * float(y.abs().max())), k


def test_missing_shard_flags_bad_targets(R):
    """States from only some shards: rows whose target lies in the missing
    vocabulary get a NaN logp and the bad-target status bit; the others
    keep finite values."""
    spec, sizes = SHARDED[0]
    case = Case(spec)
    out = run_shards(R, case, sizes, drop=(1,))
    assert out["status"] & R.DEV_EBADTARGET
    cut = _cuts(sizes)
    tg = case.inp.targets.numpy()
    missing = (tg >= cut[1]) & (tg < cut[2])
    assert missing.any() and (~missing).any()
    lp = out["logp"].cpu().numpy()
    assert np.all(np.isnan(lp[missing]))
    assert np.all(np.isfinite(lp[~missing]))
