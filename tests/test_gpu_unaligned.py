"""The loss stage and the batch-split entropy steps on input arrays that do not
start on a 16-byte boundary.

The per-token kernels of the loss stage (the entropy radix histogram, the
entropy mask, the GMPO partial sums and coefficients) take four tokens a
thread with vector loads when the arrays allow it, and one token at a time
otherwise; a tensor sliced one element in takes the second route (fp32 arrays
4 bytes off, byte masks 1 byte off).  Both routes must give the same
decisions, the same entropy threshold bit for bit, and the loss and dL/dlogp
of the oracle ("Add GMPO to fused linear GRPO loss", Details: GMPO with K3 KL;
"support top_entropy_quantile in fused linear GRPO loss", Details: the
batch-global quantile and the mask on the policy term).
"""
import numpy as np
import pytest
import torch

import oracle as O
from lm_head_log_tma_gb300.workloads import random_entropies

pytestmark = pytest.mark.gpu

B, T = 3, 1001   # odd T: slices and sequences start at unaligned tokens
EPS_LOW, EPS_HIGH = 0.2, 0.3


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_log_tma_gb300 import rlloss
    return rlloss


def _inputs(seed):
    rng = np.random.default_rng(seed)
    N = B * T
    logp = (-11.9 + 0.5 * rng.standard_normal(N)).astype(np.float32)
    old = (logp + 0.3 * rng.standard_normal(N)).astype(np.float32)
    ref = (logp + 0.1 * rng.standard_normal(N)).astype(np.float32)
    adv = np.array([1.0, -0.7, 0.4], np.float32)
    mask = np.ones(N, np.uint8)
    for i, prompt in enumerate((37, 130, 5)):   # prompts of odd lengths
        mask[i * T:i * T + prompt] = 0
    ent = random_entropies(N, seed).numpy()
    return logp, old, ref, adv, mask, ent


def _aligned(x):
    return torch.as_tensor(x).cuda()


def _shifted(x):
    """A device copy of x whose data starts one element past an aligned allocation."""
    t = torch.as_tensor(x)
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    buf[1:] = t.cuda()
    out = buf[1:]
    assert out.data_ptr() % 16 != 0
    return out


@pytest.mark.parametrize("beta,q", [(0.0, 1.0), (0.0, 0.2), (0.04, 1.0), (0.04, 0.2)])
def test_loss_stage_on_unaligned_inputs(R, beta, q):
    """Aligned and shifted inputs: identical clip and kept counts, entropy
    threshold and mask; loss and dL/dlogp equal to fp32 summation order and to
    the oracle."""
    logp, old, ref, adv, mask, ent = _inputs(7)
    cfg = R.make_cfg(B, T, eps_low=EPS_LOW, eps_high=EPS_HIGH, beta=beta, top_entropy_quantile=q)
    outs = []
    for place in (_aligned, _shifted):
        o = R.loss_from_logp(cfg, place(logp), place(ent) if q < 1 else None, place(old),
                             place(ref) if beta else None, place(adv), place(mask))
        torch.cuda.synchronize()
        assert R.rlloss_get_device_status(o["workspace"]) == 0
        outs.append(o)
    a, s = outs
    ma, ms = a["metrics"].cpu().numpy(), s["metrics"].cpu().numpy()
    for k in (1, 3, 5):   # clip count, active tokens, kept tokens: exact
        assert ma[k] == ms[k], k
    assert np.array_equal(ma[4], ms[4]) or (np.isnan(ma[4]) and np.isnan(ms[4]))   # threshold
    if q < 1:
        assert torch.equal(a["emask"], s["emask"])
    assert s["loss"].item() == pytest.approx(a["loss"].item(), rel=1e-6)
    da, ds = a["dlogp"].cpu().numpy(), s["dlogp"].cpu().numpy()
    assert np.array_equal(da == 0, ds == 0)
    assert np.allclose(ds, da, rtol=1e-6, atol=0)

    f64 = lambda x: x.astype(np.float64)
    o = O.gmpo_loss(f64(logp), f64(old), f64(ref) if beta else None, f64(adv), mask, B, T, EPS_LOW, EPS_HIGH,
                    beta=beta, entropy=f64(ent) if q < 1 else None, q=float(np.float32(q)))
    assert ma[1] == o.metrics[1]
    for g in (a, s):
        assert g["loss"].item() == pytest.approx(o.loss, rel=1e-5)
        gd = g["dlogp"].cpu().numpy()
        assert np.array_equal(gd == 0, o.c == 0)
        assert np.allclose(gd, o.c, rtol=1e-5, atol=1e-12)


def test_entropy_select_steps_on_unaligned_inputs(R):
    """The batch-split radix select (per-pass counts, select step) gives the same
    counts in every pass and the same threshold from shifted arrays as from
    aligned ones, and exactly the oracle's threshold (sort, linear interpolation)."""
    _, _, _, _, mask, ent = _inputs(11)
    q = 0.2
    thr = []
    counts = []
    for place in (_aligned, _shifted):
        e, m = place(ent), place(mask)
        st = R.alloc_select_state()
        cs = []
        for p in range(R.SELECT_PASSES):
            c = R.entropy_hist(e, m, p, st)
            cs.append(c.clone())
            R.entropy_select(p, c, q, st)
        torch.cuda.synchronize()
        counts.append(cs)
        thr.append(R.rlloss_select_threshold(st))
    for ca, cb in zip(*counts):
        assert torch.equal(ca, cb)
    assert thr[0] == thr[1]
    # q crosses the C ABI as an fp32 value: the oracle takes that value, widened
    ref_thr, _ = O.entropy_threshold(ent.astype(np.float64), mask, float(np.float32(q)))
    assert thr[0] == ref_thr
