"""Shared helpers for GPU-vs-oracle parity tests.

Tolerances (derivations in DESIGN.md, "Parity bar"):
  loss                      relative 1e-5
  dX, dW, db                relative L2 <= 5e-3 and cosine >= 0.9999
  logp, entropy per token   |err| <= 2e-5 + 2e-6 |x|   (fp32 accumulation over K, fp32 row state)
  clip count, entropy mask  exact, except items within 1e-6 of their bound or threshold
                            ("knife-edge"); for those the GPU's decision is taken as
                            valid and the oracle recomputes with it.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from lm_head_log_tma_gb300.workloads import GMPO, GSPO_TOKEN, Inputs, Workload, make_inputs

LOSS_RTOL = 1e-5
GRAD_RELL2 = 5e-3
GRAD_COS = 0.9999
ROW_ATOL = 2e-5
ROW_RTOL = 2e-6
EDGE = 1e-6


def rel_l2(a, b):
    a = np.asarray(a, np.float64).ravel(); b = np.asarray(b, np.float64).ravel()
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel(); b = np.asarray(b, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def problem_of(spec: Workload) -> O.Problem:
    return O.Problem(spec.B, spec.T, spec.loss_type, spec.eps_low, spec.eps_high, spec.beta,
                     spec.temperature, spec.top_entropy_quantile)


def cfg_of(R, spec: Workload, **kw):
    return R.make_cfg(spec.B, spec.T, spec.H, spec.V, dtype=R.FP32 if spec.dtype == "fp32" else R.BF16,
                      loss_type=spec.loss_type, eps_low=spec.eps_low, eps_high=spec.eps_high,
                      beta=spec.beta, temperature=spec.temperature,
                      top_entropy_quantile=spec.top_entropy_quantile, has_bias=spec.has_bias, **kw)


class Case:
    """One workload: inputs, oracle forward, and (lazily) oracle loss/grads."""

    def __init__(self, spec: Workload, inp: Inputs | None = None, threads=None):
        self.spec = spec
        self.inp = inp if inp is not None else make_inputs(spec)
        self.prob = problem_of(spec)
        i = self.inp
        self.lse, self.logp, self.ent = O.row_stats(i.X, i.W, i.b, i.targets, spec.temperature,
                                                    threads=threads)
        pol = torch.from_numpy(self.logp)
        self.old = i.old_logp(pol)
        self.ref = i.ref_logp(pol)
        self.old64 = self.old.double().numpy()
        self.ref64 = None if self.ref is None else self.ref.double().numpy()
        self.adv64 = i.adv.double().numpy()
        self.mask = i.mask.numpy()

    def loss(self, emask_override=None, clip_override=None) -> O.LossResult:
        return O.loss_stage(self.prob, self.logp, self.ent, self.old64, self.ref64, self.adv64,
                            self.mask, emask_override=emask_override, clip_override=clip_override)

    def run_gpu(self, R, dev="cuda", per_token=True, **cfg_kw):
        i = self.inp
        cfg = cfg_of(R, self.spec, **cfg_kw)
        t = lambda x: None if x is None else x.to(dev)
        out = R.fwd_bwd(cfg, t(i.X), t(i.W), t(i.b), t(i.targets), t(self.old), t(self.ref), t(i.adv),
                        t(i.mask), per_token=per_token)
        torch.cuda.synchronize()
        out["status"] = R.rlloss_get_device_status(out["workspace"])
        return out

    # knife-edge items ------------------------------------------------------
    def gmpo_clip_edges(self):
        """Active tokens whose oracle log ratio is within EDGE of the active bound."""
        s = self.spec
        lr = (self.logp - self.old64).reshape(s.B, s.T)
        A = self.adv64[:, None]
        eh, el = O.f32(s.eps_high), O.f32(s.eps_low)
        near = ((A > 0) & (np.abs(lr - eh) <= EDGE)) | ((A < 0) & (np.abs(lr + el) <= EDGE))
        return (near & (self.mask.reshape(s.B, s.T) != 0)).reshape(-1)


def check_rows(out, case: Case, rows=None):
    """Per-token logp and entropy against the oracle; returns max errors."""
    gl = out["logp"].double().cpu().numpy()
    ge = out["entropy"].double().cpu().numpy()
    ol, oe = case.logp, case.ent
    if rows is not None:
        gl, ge, ol, oe = gl[rows], ge[rows], ol[rows], oe[rows]
    el = np.abs(gl - ol)
    ee = np.abs(ge - oe)
    assert np.all(el <= ROW_ATOL + ROW_RTOL * np.abs(ol)), f"logp max err {el.max():.3e}"
    assert np.all(ee <= ROW_ATOL + ROW_RTOL * np.abs(oe)), f"entropy max err {ee.max():.3e}"
    return float(el.max()), float(ee.max())


def reconcile_loss(out, case: Case):
    """Oracle loss stage with the GPU's decisions on knife-edge items only.

    Asserts that every entropy-mask bit away from the threshold matches the
    oracle, then returns the oracle LossResult recomputed with the GPU's bits
    on the knife-edge tokens."""
    s = case.spec
    res = case.loss()
    emask_override = None
    if s.top_entropy_quantile < 1.0:
        g = out["emask"].cpu().numpy().astype(np.uint8)
        thr = res.metrics[4]
        edge = np.abs(case.ent - thr) <= EDGE
        diff = g != res.emask
        assert not np.any(diff & ~edge), f"{int((diff & ~edge).sum())} mask bits differ away from the threshold"
        if np.any(diff):
            emask_override = np.where(edge, g, res.emask)
            res = case.loss(emask_override=emask_override)
    return res


def check_loss_and_metrics(out, case: Case, res: O.LossResult):
    gl = float(out["loss"].item())
    assert abs(gl - res.loss) <= LOSS_RTOL * abs(res.loss), f"loss {gl!r} vs oracle {res.loss!r}"
    gm = out["metrics"].double().cpu().numpy()
    om = res.metrics
    n_edge = int(case.gmpo_clip_edges().sum()) if case.spec.loss_type == GMPO else 0
    assert abs(gm[1] - om[1]) <= n_edge, f"clip count {gm[1]} vs {om[1]}"
    assert gm[3] == om[3]
    if case.spec.top_entropy_quantile < 1.0:
        assert abs(gm[4] - om[4]) <= 2e-6 * abs(om[4]) + 1e-6, (gm[4], om[4])
        assert gm[5] == om[5], (gm[5], om[5])
    else:
        assert np.isnan(gm[4])
    assert abs(gm[6] - om[6]) <= 1e-5 + 1e-5 * abs(om[6]), (gm[6], om[6])
    assert abs(gm[7] - om[7]) <= 1e-5 * abs(om[7]) + 1e-7, (gm[7], om[7])
    if case.spec.beta != 0:
        assert abs(gm[2] - om[2]) <= 1e-4 * abs(om[2]) + 1e-7, (gm[2], om[2])
    return gl, res.loss


def check_grads(out, case: Case, res: O.LossResult, dx_rows=None, dw_rows=None):
    i = case.inp
    s = case.spec
    dX, dW, db = O.grads(i.X, i.W, i.b, i.targets, s.temperature, case.lse, res.c, dx_rows, dw_rows,
                         want_db=i.b is not None)
    gdx = out["dX"].double().cpu().numpy()
    gdw = out["dW"].double().cpu().numpy()
    if dx_rows is not None:
        gdx = gdx[dx_rows]
    if dw_rows is not None:
        gdw = gdw[dw_rows]
    # rows of knife-edge clip tokens may legitimately differ: compare the rest
    edges = case.gmpo_clip_edges() if s.loss_type == GMPO else np.zeros(s.N, bool)
    keep = ~edges if dx_rows is None else ~edges[dx_rows]
    stats = {}
    for name, g, o in (("dX", gdx[keep], dX[keep]), ("dW", gdw, dW)):
        r, c = rel_l2(g, o), cosine(g, o)
        stats[name] = (r, c)
        assert r <= GRAD_RELL2 and c >= GRAD_COS, f"{name}: rel-L2 {r:.3e} cos {c:.7f}"
    if i.b is not None:
        gdb = out["db"].double().cpu().numpy()
        r, c = rel_l2(gdb, db), cosine(gdb, db)
        stats["db"] = (r, c)
        assert r <= GRAD_RELL2 and c >= GRAD_COS, f"db: rel-L2 {r:.3e} cos {c:.7f}"
    return stats
