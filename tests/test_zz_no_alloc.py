"""The allocation-free loss entry point against the workspace-taking one.

rlloss_loss_from_logp_noalloc serves callers that cannot allocate device
memory — code running while another component captures a CUDA graph, plugins
handed only the tensors they read and write, runtimes whose memory pool is
reserved in full up front.  Its scratch is a fixed 4 MiB array inside the
library instead of a caller workspace.  Here it is called through the C ABI
twice in a row (different problem shapes, so stale contents of the shared
array would show) and checked against rlloss_loss_from_logp on the same inputs,
and once against the fp64 oracle, so that a fault the two entries share would
not go unseen.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O

from lm_head_log_tma_gb300.workloads import random_entropies

pytestmark = pytest.mark.gpu

LOSS_RTOL = 1e-5


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_log_tma_gb300 import rlloss
    return rlloss


def _entry(R):
    f = R.lib.rlloss_loss_from_logp_noalloc
    f.argtypes = [ctypes.POINTER(R.RllossCfg)] + [ctypes.c_void_p] * 12
    f.restype = ctypes.c_int
    return f


def _inputs(B, T, seed):
    g = torch.Generator().manual_seed(seed)
    N = B * T
    logp = -11.9 + 0.5 * torch.randn(N, generator=g)
    old = logp + 0.3 * torch.randn(N, generator=g)
    ref = logp + 0.1 * torch.randn(N, generator=g)
    adv = torch.randn(B, generator=g)
    mask = (torch.arange(T)[None, :] >= 7).expand(B, T).reshape(-1).to(torch.uint8).contiguous()
    ent = random_entropies(N, seed)
    return {k: v.cuda() for k, v in dict(logp=logp, old=old, ref=ref, adv=adv, mask=mask, ent=ent).items()}


def _call_noalloc(R, f, cfg, t):
    N = cfg.B * cfg.T
    o = dict(loss=torch.empty(1, device="cuda"), metrics=torch.empty(R.NMETRICS, device="cuda"),
             dlogp=torch.empty(N, device="cuda"), emask=torch.empty(N, dtype=torch.uint8, device="cuda"),
             status=torch.full((1,), -1, dtype=torch.int32, device="cuda"))
    p = lambda x: ctypes.c_void_p(x.data_ptr())
    rc = f(ctypes.byref(cfg), p(t["logp"]), p(t["ent"]), p(t["old"]), p(t["ref"]), p(t["adv"]), p(t["mask"]),
           p(o["loss"]), p(o["metrics"]), p(o["dlogp"]), p(o["emask"]), p(o["status"]),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, o


def test_noalloc_matches_workspace_entry_two_calls_in_a_row(R):
    f = _entry(R)
    cases = [(R.make_cfg(6, 700, eps_low=0.2, eps_high=0.3, beta=0.04, top_entropy_quantile=0.2), 21),
             (R.make_cfg(3, 517), 22)]
    for cfg, seed in cases:
        t = _inputs(cfg.B, cfg.T, seed)
        rc, a = _call_noalloc(R, f, cfg, t)
        assert rc == R.OK
        b = R.loss_from_logp(cfg, t["logp"], t["ent"], t["old"], t["ref"] if cfg.beta else None, t["adv"],
                             t["mask"])
        torch.cuda.synchronize()
        assert a["status"].item() == 0
        assert R.rlloss_get_device_status(b["workspace"]) == 0
        la, lb = a["loss"].item(), b["loss"].item()
        assert abs(la - lb) <= LOSS_RTOL * abs(lb)
        assert torch.allclose(a["dlogp"], b["dlogp"], rtol=LOSS_RTOL, atol=0)
        assert torch.equal(a["emask"], b["emask"])
        ma, mb = a["metrics"].cpu(), b["metrics"].cpu()
        assert torch.allclose(ma, mb, rtol=LOSS_RTOL, atol=0, equal_nan=True)
        assert ma[1] == mb[1] and ma[3] == mb[3] and ma[5] == mb[5]


def test_noalloc_rejects_problems_beyond_its_scratch(R):
    f = _entry(R)
    cfg = R.make_cfg(1, 1 << 22)          # 4 Mi tokens: needs more than the 4 MiB scratch
    rc = f(ctypes.byref(cfg), *([None] * 12))
    assert rc == 5                         # RLLOSS_ETOOLARGE


def test_noalloc_matches_the_oracle(R):
    """GMPO with K3 KL and the entropy mask at q = 0.2 against the fp64 oracle
    on the same fp32 inputs: the mask bit for bit, the loss within 1e-5."""
    f = _entry(R)
    B, T = 5, 600
    cfg = R.make_cfg(B, T, eps_low=0.2, eps_high=0.3, beta=0.04, top_entropy_quantile=0.2)
    t = _inputs(B, T, 23)
    rc, a = _call_noalloc(R, f, cfg, t)
    assert rc == R.OK
    torch.cuda.synchronize()
    assert a["status"].item() == 0
    h = {k: v.cpu().double().numpy() for k, v in t.items()}
    o = O.gmpo_loss(h["logp"], h["old"], h["ref"], h["adv"], h["mask"].astype(np.uint8), B, T, 0.2, 0.3,
                    beta=0.04, entropy=h["ent"], q=0.2)
    assert np.array_equal(a["emask"].cpu().numpy(), o.emask)
    assert abs(a["loss"].item() - o.loss) <= LOSS_RTOL * abs(o.loss)
    g = a["dlogp"].cpu().double().numpy()
    assert np.array_equal(g == 0, o.c == 0)
    assert np.allclose(g, o.c, rtol=1e-5, atol=1e-12)
    m = a["metrics"].cpu().double().numpy()
    assert m[1] == o.metrics[1] and m[3] == o.metrics[3] and m[5] == o.metrics[5]
