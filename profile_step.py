"""Run a few fused forward+backward steps of the Qwen-0.5B LM-head workload
recipe at a chosen token count, for profilers (ncu) to attach to.

  python profile_step.py --T 2048 --steps 1 --warmup 2
  python profile_step.py --loss-only --B 16 --T 4194304 --q 0.2 --steps 1 --warmup 1

The inputs follow the workload recipe (H=896, V=151936, bf16, GMPO); the
sampler log-probs are the policy's plus noise, with the policy log-probs
taken from the library's own forward output of a first call.  --loss-only
runs the loss stage alone (rlloss_loss_from_logp: entropy quantile, loss,
dL/dlogp) on B*T synthetic tokens (log-probs near -11.9, entropies of the
large-vocabulary recipe, 1/8 of each sequence masked as prompt), for the
reduction kernels.
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

from lm_head_log_tma_gb300 import rlloss as R
from lm_head_log_tma_gb300.workloads import WORKLOADS, make_inputs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--steps", type=int, default=1)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--loss-only", action="store_true")
    ap.add_argument("--q", type=float, default=0.2, help="top-entropy quantile of --loss-only")
    ap.add_argument("--recompute", action="store_true", help="RLLOSS_FLAG_RECOMPUTE")
    a = ap.parse_args()
    if a.loss_only:
        return loss_only(a)
    spec = WORKLOADS[a.workload]
    kw = {}
    if a.B:
        kw["B"] = a.B
    if a.T:
        kw["T"] = a.T
        if not isinstance(spec.prompt_len, tuple):
            kw["prompt_len"] = min(spec.prompt_len, a.T // 8)
    spec = dataclasses.replace(spec, **kw)
    inp = make_inputs(spec, device="cuda")
    cfg = R.make_cfg(spec.B, spec.T, spec.H, spec.V, dtype=R.BF16 if spec.dtype == "bf16" else R.FP32,
                     loss_type=spec.loss_type, eps_low=spec.eps_low, eps_high=spec.eps_high, beta=spec.beta,
                     temperature=spec.temperature, top_entropy_quantile=spec.top_entropy_quantile,
                     has_bias=spec.has_bias, flags=R.FLAG_RECOMPUTE if a.recompute else 0)
    zeros = torch.zeros(spec.N, device="cuda")
    first = R.fwd_bwd(cfg, inp.X, inp.W, inp.b, inp.targets, zeros, zeros if spec.beta else None, inp.adv,
                      inp.mask)
    pol = first["logp"].clone()
    old, ref = inp.old_logp(pol), inp.ref_logp(pol)
    ws, outs = first["workspace"], None
    for _ in range(a.warmup + a.steps):   # a training step: no per-token outputs
        outs = R.fwd_bwd(cfg, inp.X, inp.W, inp.b, inp.targets, old, ref, inp.adv, inp.mask, workspace=ws,
                         outputs=outs, per_token=False)
    torch.cuda.synchronize()
    st = R.rlloss_get_device_status(ws)
    print(f"{spec.name} B={spec.B} T={spec.T}: loss {outs['loss'].item():.6g} status {st:#x}")
    return 0 if st == 0 else 1


def loss_only(a):
    from lm_head_log_tma_gb300.workloads import random_entropies
    B, T = a.B or 16, a.T or (1 << 22)
    N = B * T
    g = torch.Generator(device="cuda").manual_seed(5)
    logp = -11.9 + 0.5 * torch.randn(N, generator=g, device="cuda")
    old = logp + 0.3 * torch.randn(N, generator=g, device="cuda")
    adv = torch.randn(B, generator=g, device="cuda")
    mask = (torch.arange(T, device="cuda")[None, :] >= T // 8).expand(B, T).reshape(-1).to(torch.uint8).contiguous()
    ent = random_entropies(N, 5, device="cuda")
    cfg = R.make_cfg(B, T, top_entropy_quantile=a.q)
    o = None
    for _ in range(a.warmup + a.steps):
        o = R.loss_from_logp(cfg, logp, ent, old, None, adv, mask)
    torch.cuda.synchronize()
    st = R.rlloss_get_device_status(o["workspace"])
    print(f"loss stage B={B} T={T} q={a.q}: loss {o['loss'].item():.6g} threshold {o['metrics'][4].item():.6g} "
          f"status {st:#x}")
    return 0 if st == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
