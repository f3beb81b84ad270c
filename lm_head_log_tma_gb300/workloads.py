"""Seeded synthetic workloads for the fused LM-head RL policy loss.

This module only draws random numbers and lays them out; it holds none of the
loss arithmetic, so both the CUDA path and the fp64 CPU oracle can be fed from
it.  The recipes follow the workload table of the build (Qwen-0.5B LM-head
shape H=896, V=151936 from "Add GMPO to fused linear GRPO loss", section
"Forward and backward numerical comparison"; the GSPO clip range from the
Tinker "GSPO" page, section "Choosing clipping thresholds").

One input of the recipes needs the policy's own log-probabilities: the
"old" (sampler) and "ref" log-probs are defined as the policy log-prob plus
Gaussian noise.  The noise is drawn here; the policy log-prob is supplied by
the caller (the oracle in tests, a plain full-logits pass in the benchmark).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import torch

GMPO = 0
GSPO_TOKEN = 1


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    V: int
    dtype: str                 # "bf16" or "fp32" for X, W, b
    loss_type: int = GMPO
    has_bias: bool = False
    bias_std: float = 0.0
    temperature: float = 1.0
    eps_low: float = 0.4
    eps_high: float = 0.4
    beta: float = 0.0
    top_entropy_quantile: float = 1.0
    prompt_len: int | tuple = 0   # int, or (lo, hi) inclusive uniform range per sequence
    adv_kind: str = "normal"      # "normal", "pm1zero", or "fixed"
    adv_fixed: tuple = ()
    old_noise_std: float = 0.3
    ref_noise_std: float = 0.0    # 0 -> ref_logp absent
    seed: int = 0

    @property
    def N(self) -> int:
        return self.B * self.T

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five synthetic workloads.  Index = seed offset (seed 0 + index).
WORKLOADS: list[Workload] = [
    Workload("tiny_gmpo_fp32", B=2, T=16, H=64, V=512, dtype="fp32", prompt_len=4,
             adv_kind="fixed", adv_fixed=(1.0, -0.5), old_noise_std=0.3, seed=0),
    Workload("qwen05b_gmpo_b1_t4096", B=1, T=4096, H=896, V=151936, dtype="bf16",
             prompt_len=512, adv_kind="normal", old_noise_std=0.3, seed=1),
    Workload("qwen05b_gmpo_k3kl_bias_b8_t2048", B=8, T=2048, H=896, V=151936, dtype="bf16",
             has_bias=True, bias_std=0.01, eps_low=0.2, eps_high=0.3, beta=0.04,
             prompt_len=(64, 512), adv_kind="pm1zero", old_noise_std=0.3,
             ref_noise_std=0.1, seed=2),
    Workload("qwen05b_gmpo_entropy_q0.2_b16_t4096", B=16, T=4096, H=896, V=151936,
             dtype="bf16", temperature=0.7, top_entropy_quantile=0.2, prompt_len=512,
             adv_kind="normal", old_noise_std=0.3, seed=3),
    Workload("qwen05b_gspo_token_b16_t8192", B=16, T=8192, H=896, V=151936, dtype="bf16",
             loss_type=GSPO_TOKEN, eps_low=3e-4, eps_high=4e-4, prompt_len=256,
             adv_kind="normal", old_noise_std=0.02, seed=4),
]


@dataclass
class Inputs:
    """One batch.  Shapes: X [N,H], W [V,H], b [V] or None, targets int64 [N],
    mask uint8 [N], adv fp32 [B], old_noise / ref_noise fp32 [N]."""
    spec: Workload
    X: torch.Tensor
    W: torch.Tensor
    b: torch.Tensor | None
    targets: torch.Tensor
    mask: torch.Tensor
    adv: torch.Tensor
    old_noise: torch.Tensor
    ref_noise: torch.Tensor | None
    prompt_lens: list = field(default_factory=list)

    def old_logp(self, policy_logp: torch.Tensor) -> torch.Tensor:
        """Sampler log-probs: the supplied policy log-probs shifted by the drawn noise."""
        return (policy_logp.float().to(self.old_noise.device) + self.old_noise).contiguous()

    def ref_logp(self, policy_logp: torch.Tensor) -> torch.Tensor | None:
        if self.ref_noise is None:
            return None
        return (policy_logp.float().to(self.ref_noise.device) + self.ref_noise).contiguous()


def _torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def make_inputs(spec: Workload, device: str | torch.device = "cpu") -> Inputs:
    """Draw one batch of ``spec`` with a generator seeded by ``spec.seed``.

    X ~ N(0,1), W ~ N(0, 0.02^2), b ~ N(0, bias_std^2), targets uniform in [0,V),
    completion mask = 0 on each sequence's prompt, advantages per sequence.
    Draws happen in fp32 and are then rounded to the workload dtype.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(spec.seed))
    N, H, V, B, T = spec.N, spec.H, spec.V, spec.B, spec.T
    dt = _torch_dtype(spec.dtype)

    X = torch.randn(N, H, generator=g, device=dev, dtype=torch.float32).to(dt).contiguous()
    W = (torch.randn(V, H, generator=g, device=dev, dtype=torch.float32) * 0.02).to(dt).contiguous()
    b = None
    if spec.has_bias:
        b = (torch.randn(V, generator=g, device=dev, dtype=torch.float32) * spec.bias_std).to(dt).contiguous()
    targets = torch.randint(0, V, (N,), generator=g, device=dev, dtype=torch.int64)

    if isinstance(spec.prompt_len, tuple):
        lo, hi = spec.prompt_len
        pl = torch.randint(lo, hi + 1, (B,), generator=g, device=dev).tolist()
    else:
        pl = [int(spec.prompt_len)] * B
    t_idx = torch.arange(T, device=dev)
    mask = torch.stack([(t_idx >= p) for p in pl]).reshape(N).to(torch.uint8).contiguous()

    if spec.adv_kind == "fixed":
        adv = torch.tensor(spec.adv_fixed, dtype=torch.float32, device=dev)
        assert adv.numel() == B
    elif spec.adv_kind == "pm1zero":
        adv = (torch.randint(0, 3, (B,), generator=g, device=dev) - 1).to(torch.float32)
    else:
        adv = torch.randn(B, generator=g, device=dev, dtype=torch.float32)

    old_noise = torch.randn(N, generator=g, device=dev, dtype=torch.float32) * spec.old_noise_std
    ref_noise = None
    if spec.ref_noise_std > 0:
        ref_noise = torch.randn(N, generator=g, device=dev, dtype=torch.float32) * spec.ref_noise_std
    return Inputs(spec, X, W, b, targets, mask, adv.contiguous(), old_noise.contiguous(),
                  None if ref_noise is None else ref_noise.contiguous(), pl)


def random_entropies(n: int, seed: int, center: float = 11.56, std: float = 0.017,
                     device="cpu") -> torch.Tensor:
    """A narrow band of fp32 per-token entropies (the spread seen at V=151936,
    temperature 0.7), for exercising the batch-global quantile on its own."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return (center + std * torch.randn(n, generator=g, device=device, dtype=torch.float32)).contiguous()
