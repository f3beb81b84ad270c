"""GPU parity of the fused path against the fp64 oracle, through the C ABI.

Sizes here span several 128-row and 256-column tiles with ragged tails, so
every tail path of the kernels runs; the oracle finishes each in seconds.
"""
import numpy as np
import pytest
import torch

import oracle as O
from lm_head_log_tma_gb300.workloads import GMPO, GSPO_TOKEN, WORKLOADS, Workload, make_inputs, random_entropies

from parity import (EDGE, Case, cfg_of as parity_cfg, check_grads, check_loss_and_metrics, check_rows,
                    reconcile_loss)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_log_tma_gb300 import rlloss
    return rlloss


MID = [
    Workload("mid_gmpo_bf16", B=3, T=150, H=192, V=1000, dtype="bf16", prompt_len=20, seed=101),
    Workload("mid_gmpo_bias_k3kl", B=4, T=130, H=256, V=777, dtype="bf16", has_bias=True, bias_std=0.3,
             eps_low=0.2, eps_high=0.3, beta=0.04, prompt_len=(5, 40), adv_kind="pm1zero",
             ref_noise_std=0.1, seed=102),
    Workload("mid_entropy_q0.2_tau0.7", B=5, T=100, H=128, V=1300, dtype="bf16", temperature=0.7,
             top_entropy_quantile=0.2, prompt_len=10, seed=103),
    Workload("mid_gspo_token", B=6, T=97, H=64, V=600, dtype="bf16", loss_type=GSPO_TOKEN, eps_low=3e-4,
             eps_high=4e-4, prompt_len=8, old_noise_std=0.02, seed=104),
    Workload("mid_fp32_bias_odd", B=2, T=77, H=100, V=515, dtype="fp32", has_bias=True, bias_std=0.1,
             temperature=1.3, prompt_len=3, seed=105),
    Workload("mid_wide_logits", B=2, T=140, H=512, V=2000, dtype="bf16", prompt_len=12, seed=106),
]


def _full_check(R, case, **cfg_kw):
    out = case.run_gpu(R, **cfg_kw)
    assert out["status"] == 0, hex(out["status"])
    check_rows(out, case)
    res = reconcile_loss(out, case)
    gl, ol = check_loss_and_metrics(out, case, res)
    stats = check_grads(out, case, res)
    return out, res, stats


EDGE_SHAPES = [
    Workload("wide_h_2048", B=2, T=300, H=2048, V=3000, dtype="bf16", prompt_len=10, seed=121),
    Workload("ragged_h_1040_bias", B=3, T=100, H=1040, V=1500, dtype="bf16", has_bias=True, bias_std=0.2,
             prompt_len=5, seed=122),
    Workload("many_short_sequences", B=300, T=3, H=64, V=500, dtype="bf16", prompt_len=1, seed=123),
    Workload("many_short_gspo", B=257, T=4, H=64, V=300, dtype="bf16", loss_type=GSPO_TOKEN, eps_low=0.05,
             eps_high=0.05, prompt_len=1, old_noise_std=0.05, seed=124),
    Workload("one_token_sequence", B=1, T=1, H=64, V=257, dtype="bf16", prompt_len=0, seed=125),
    Workload("narrow_h_8", B=2, T=90, H=8, V=700, dtype="bf16", prompt_len=5, seed=126),
    Workload("large_vocab_70001", B=1, T=300, H=128, V=70001, dtype="bf16", prompt_len=20, seed=127),
]


@pytest.mark.parametrize("spec", EDGE_SHAPES, ids=[s.name for s in EDGE_SHAPES])
def test_edge_shapes(R, spec):
    """Hidden sizes that span several 448-wide dX/dW tiles (one ragged), many
    sequences of a few tokens, and a single one-token sequence."""
    case = Case(spec)
    _full_check(R, case)


def test_tiny_fp32_workload(R):
    case = Case(WORKLOADS[0])
    _full_check(R, case)


@pytest.mark.parametrize("spec", MID, ids=[s.name for s in MID])
def test_mid_workloads(R, spec):
    case = Case(spec)
    _full_check(R, case)


def test_backward_chunking_is_invariant(R):
    """Recompute chunks of 128 rows (several dW/db accumulation steps) give the
    same result as one chunk; with stored probabilities a 128-row buffer stores
    one row tile and recomputes the rest, which passes the oracle too."""
    spec = MID[1]
    case = Case(spec)
    _full_check(R, case, chunk_rows=128)
    a, _, _ = _full_check(R, case, flags=R.FLAG_RECOMPUTE)
    b, _, _ = _full_check(R, case, chunk_rows=128, flags=R.FLAG_RECOMPUTE)
    assert torch.equal(a["loss"], b["loss"])
    assert torch.allclose(a["dX"], b["dX"], rtol=1e-4, atol=1e-9)
    assert torch.allclose(a["dW"], b["dW"], rtol=1e-4, atol=1e-9)


def test_entropy_mask_non_vacuous_and_forced_path_bit_identical(R):
    spec = MID[2]
    case = Case(spec)
    out, res, _ = _full_check(R, case)
    m = out["metrics"].cpu().numpy()
    assert 0 < m[5] < m[3]           # drops some but not all active tokens
    # q = 1 with the quantile path forced is bit-identical to the path off
    spec1 = spec.with_(top_entropy_quantile=1.0)
    case1 = Case(spec1, case.inp)
    o1 = case1.run_gpu(R)
    o2 = case1.run_gpu(R, flags=R.FLAG_FORCE_ENTROPY_PATH)
    for k in ("loss", "dX", "dW"):
        assert torch.equal(o1[k], o2[k]), k
    assert torch.equal(o2["emask"], case.inp.mask.cuda())


@pytest.mark.parametrize("spec", [MID[1], MID[4], MID[5]], ids=["bf16_bias_k3kl", "fp32_bias_odd", "wide"])
def test_tile_shapes_agree(R, spec):
    """256-row CTA-pair tiles and 128-row single-CTA tiles give the same
    results (both with the recomputing backward, which single-CTA tiles use;
    the default call, which may take the stored-probability backward, passes
    the oracle as well)."""
    case = Case(spec)
    _full_check(R, case)
    a, _, _ = _full_check(R, case, flags=R.FLAG_RECOMPUTE)
    b, _, _ = _full_check(R, case, flags=R.FLAG_SINGLE_CTA_TILES)
    for k in ("loss", "logp", "entropy"):
        assert torch.allclose(a[k], b[k], rtol=1e-6, atol=1e-7), k
    for k in ("dX", "dW"):
        assert torch.allclose(a[k], b[k], rtol=1e-3, atol=1e-8), k


def test_repeated_calls_are_bit_identical(R):
    """Two calls give the same bits.  Every floating-point reduction has a fixed
    order, with one exception that is still order-free: the compacted backward
    adds each kept row's two dX halves (one per vocabulary half) into a zeroed
    dX with atomic adds, and two addends onto zero give the same fp32 sum in
    either order."""
    case = Case(MID[1])
    a = case.run_gpu(R)
    b = case.run_gpu(R)
    for k in ("loss", "metrics", "dX", "dW", "db", "logp", "entropy"):
        assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), k


def test_uniform_logits_closed_form(R):
    """W = 0: every logit is 0, so logp = -log V and H = log V on the GPU too."""
    spec = Workload("zeros", B=2, T=130, H=64, V=700, dtype="bf16", prompt_len=0, seed=7)
    inp = make_inputs(spec)
    inp.W.zero_()
    case = Case(spec, inp)
    out = case.run_gpu(R)
    assert out["status"] == 0
    assert np.allclose(out["logp"].cpu().numpy(), -np.log(700), atol=2e-6)
    assert np.allclose(out["entropy"].cpu().numpy(), np.log(700), atol=2e-6)


def test_rising_logits_move_the_reference(R):
    """A bias rising along the vocabulary (b_v = 0.048 v: logits climb about 90
    log2 units across V = 1300) puts every row's largest logits far above the
    first 32-column chunk the forward takes its reference from, so the
    reference has to move during the row (the rescale path); per-token logp,
    entropy, loss and gradients still match the oracle, on the stored path and
    the recompute."""
    spec = Workload("rising_logits", B=2, T=300, H=64, V=1300, dtype="bf16", has_bias=True, prompt_len=10,
                    seed=131)
    inp = make_inputs(spec)
    inp.b = (torch.arange(spec.V, dtype=torch.float32) * 0.048).to(torch.bfloat16)
    case = Case(spec, inp)
    assert np.all(case.lse * 1.4426950408889634 < 96)   # inside the stored range
    _full_check(R, case)
    _full_check(R, case, flags=R.FLAG_RECOMPUTE)


def test_bad_target_sets_status(R):
    spec = Workload("badtarget", B=1, T=128, H=64, V=300, dtype="bf16", seed=8)
    case = Case(spec)
    case.inp.targets[5] = 300
    out = case.run_gpu(R)
    assert out["status"] & R.DEV_EBADTARGET
    assert np.isnan(out["logp"][5].item())


def test_bounded_wait_times_out_cleanly(R):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert R.rlloss_selftest_bounded_wait(ws, 2_000_000) == R.OK
    torch.cuda.synchronize()
    assert R.rlloss_get_device_status(ws) & R.DEV_ETIMEOUT
    # the context is still usable afterwards
    assert torch.ones(4, device="cuda").sum().item() == 4


def test_forward_only_scoring_matches_oracle_and_full_call(R):
    """rlloss_forward: per-token logp, entropy and lse against the oracle, and
    bit-identical logp / entropy to the full call."""
    spec = MID[1]
    case = Case(spec)
    i = case.inp
    cfg = R.make_cfg(spec.B, spec.T, spec.H, spec.V, dtype=R.BF16, temperature=0.7, has_bias=True)
    f = R.forward(cfg, i.X.cuda(), i.W.cuda(), i.b.cuda(), i.targets.cuda())
    torch.cuda.synchronize()
    assert R.rlloss_get_device_status(f["workspace"]) == 0
    lse, logp, ent = O.row_stats(i.X, i.W, i.b, i.targets, 0.7)
    for k, ref in (("logp", logp), ("entropy", ent), ("lse", lse)):
        g = f[k].double().cpu().numpy()
        assert np.all(np.abs(g - ref) <= 2e-5 + 2e-6 * np.abs(ref)), k
    case07 = Case(spec.with_(temperature=0.7), i)
    full = case07.run_gpu(R)
    assert torch.equal(full["logp"], f["logp"]) and torch.equal(full["entropy"], f["entropy"])


def _e4m3_rows(x):
    """Per-row absmax scaling into e4m3 (the caller's quantizer; any would do):
    returns (e4m3 tensor, fp32 scales, fp64 dequantized values)."""
    x = x.float()
    scale = (x.abs().amax(dim=1) / 448.0).clamp(min=1e-30)
    q = (x / scale[:, None]).to(torch.float8_e4m3fn)
    return q, scale, q.to(torch.float64) * scale.double()[:, None]


@pytest.mark.parametrize("shape", [(2, 150, 192, 1000, True, 0.7), (3, 77, 64, 515, False, 1.0),
                                   (1, 300, 896, 2000, False, 1.0)], ids=["h192_bias", "h64", "h896"])
def test_e4m3_scoring_matches_oracle(R, shape):
    """Forward-only scoring with e4m3 operands and per-row scales: logp,
    entropy and lse equal the oracle's on the dequantized inputs to the same
    bar as the bf16 path (the e4m3 products and their fp32 sums are exact up
    to fp32 rounding)."""
    B, T, H, V, bias, tau = shape
    g = torch.Generator().manual_seed(H + V)
    X = torch.randn(B * T, H, generator=g)
    W = torch.randn(V, H, generator=g) * 0.02
    b = torch.randn(V, generator=g) * 0.05 if bias else None
    y = torch.randint(0, V, (B * T,), generator=g)
    X8, xs, Xd = _e4m3_rows(X)
    W8, ws, Wd = _e4m3_rows(W)
    cfg = R.make_cfg(B, T, H, V, dtype=R.FP8_E4M3, temperature=tau, has_bias=bias)
    c = lambda t: None if t is None else t.cuda()
    f = R.forward_e4m3(cfg, c(X8), c(xs), c(W8), c(ws), c(b), c(y))
    torch.cuda.synchronize()
    assert R.rlloss_get_device_status(f["workspace"]) == 0
    lse, logp, ent = O.row_stats(Xd, Wd, None if b is None else b.double(), y, tau)
    for k, ref in (("logp", logp), ("entropy", ent), ("lse", lse)):
        gk = f[k].double().cpu().numpy()
        err = np.abs(gk - ref)
        assert np.all(err <= 2e-5 + 2e-6 * np.abs(ref)), (k, float(err.max()))


def test_gspo_per_token_advantages_full_path(R):
    """GSPO with per-token advantages (nonzero also outside the ratio mask)
    through the fused path, against the oracle."""
    spec = MID[3]
    case = Case(spec)
    i = case.inp
    g = torch.Generator().manual_seed(77)
    An = torch.randn(spec.N, generator=g)
    cfg = R.make_cfg(spec.B, spec.T, spec.H, spec.V, dtype=R.BF16, loss_type=R.GSPO_TOKEN, eps_low=spec.eps_low,
                     eps_high=spec.eps_high, flags=R.FLAG_ADV_PER_TOKEN)
    c = lambda x: x.cuda()
    out = R.fwd_bwd(cfg, c(i.X), c(i.W), None, c(i.targets), c(case.old), None, c(An), c(i.mask))
    torch.cuda.synchronize()
    assert R.rlloss_get_device_status(out["workspace"]) == 0
    prob = O.Problem(spec.B, spec.T, O.GSPO_TOKEN, spec.eps_low, spec.eps_high, per_token_adv=True)
    res = O.loss_stage(prob, case.logp, case.ent, case.old64, None, An.double().numpy(), case.mask)
    gl = out["loss"].item()
    assert abs(gl - res.loss) <= 1e-5 * abs(res.loss), (gl, res.loss)
    assert out["metrics"][1].item() == res.metrics[1]
    dX, dW, _ = O.grads(i.X, i.W, None, i.targets, spec.temperature, case.lse, res.c)
    from parity import rel_l2, cosine
    for name, gx, ox in (("dX", out["dX"], dX), ("dW", out["dW"], dW)):
        gx = gx.double().cpu().numpy()
        assert rel_l2(gx, ox) <= 5e-3 and cosine(gx, ox) >= 0.9999, name


@pytest.mark.parametrize("q", [0.5, 0.8])
def test_entropy_mask_other_quantiles_full_path(R, q):
    """The batch-global mask at q = 0.5 and 0.8 through the fused path: it
    drops some but not all active tokens, and everything matches the oracle."""
    case = Case(MID[2].with_(top_entropy_quantile=q))
    out, _, _ = _full_check(R, case)
    m = out["metrics"].cpu().numpy()
    assert 0 < m[5] < m[3]


@pytest.mark.parametrize("spec", [MID[0], MID[3]], ids=["gmpo", "gspo"])
def test_extreme_log_ratios_full_path(R, spec):
    """Sampler log-probs 30 nats away from the policy's (alternating sign by
    sequence): GMPO's log-space clip keeps every ratio finite, GSPO's
    sequence ratios are e^(+-30)-sized and clipped; loss and gradients stay
    finite and match the oracle."""
    case = Case(spec)
    sign = torch.tensor([(-1.0) ** i for i in range(spec.B)]).repeat_interleave(spec.T)
    case.old = (case.old.double() + 30.0 * sign).float()
    case.old64 = case.old.double().numpy()
    out, _, _ = _full_check(R, case)
    assert np.isfinite(out["loss"].item())
    for k in ("dX", "dW"):
        assert torch.isfinite(out[k]).all(), k


def test_nonfinite_logp_sets_status(R):
    """A NaN log-prob on an active token makes the loss NaN and sets the
    non-finite bit in the device status word (no trap)."""
    n = 64
    logp = np.full(n, -2.0, np.float32)
    logp[5] = np.nan
    g = _loss_gpu(R, R.make_cfg(1, n), logp, np.full(n, -2.0, np.float32), np.ones(1, np.float32),
                  np.ones(n, np.uint8))
    assert g["status"] & R.DEV_ENONFINITE
    assert np.isnan(g["loss"].item())


# ------------------------------------------------------------------ backward row compaction
def _grads_close(a, b):
    for k in ("dX", "dW", "db"):
        if a.get(k) is None:
            continue
        x, y = a[k], b[k]
        tol = 1e-5 * float(y.abs().max()) + 1e-12
        assert torch.allclose(x, y, rtol=1e-4, atol=tol), k


@pytest.mark.parametrize("spec", [MID[0], MID[1], MID[3], MID[4]], ids=["gmpo", "bias_k3kl", "gspo", "fp32_bias_odd"])
def test_compacted_backward_matches_dense(R, spec):
    """By default rows with c_n = 0 are dropped before the backward; the dense
    backward over every row gives the same gradients up to fp32 summation
    order, the same forward and loss bits, and both pass the oracle."""
    case = Case(spec)
    _full_check(R, case)   # default call (stored probabilities where they apply)
    a, res, _ = _full_check(R, case, flags=R.FLAG_RECOMPUTE)
    b, _, _ = _full_check(R, case, flags=R.FLAG_ALL_ROWS)
    keep = res.c != 0
    assert 0 < keep.sum() < spec.N, "the workload must both keep and drop rows"
    assert R.rlloss_get_backward_rows(a["workspace"]) == int(keep.sum())
    assert R.rlloss_get_backward_rows(b["workspace"]) == spec.N
    for k in ("loss", "metrics", "logp", "entropy"):
        assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), k
    assert torch.count_nonzero(a["dX"][torch.from_numpy(~keep).cuda()]) == 0
    _grads_close(a, b)


def test_misaligned_gradient_buffer_is_rejected(R):
    """dX must start on a 16-byte boundary (its rows leave through TMA maps
    and float4 adds): a dX one float past such a boundary is rejected before
    any launch, and the buffer is left as it was."""
    spec = MID[1]
    case = Case(spec)
    a = case.run_gpu(R, per_token=False)
    assert a["status"] == 0, hex(a["status"])
    i = case.inp
    N, H = spec.N, spec.H
    buf = torch.full((N * H + 8,), float("nan"), device="cuda")
    dX = buf[1:1 + N * H].view(N, H)
    assert dX.data_ptr() % 16 == 4
    outs = dict(a)
    outs["dX"] = dX
    cfg = parity_cfg(R, spec)
    t = lambda x: None if x is None else x.cuda()
    with pytest.raises(R.RllossError) as e:
        R.fwd_bwd(cfg, t(i.X), t(i.W), t(i.b), t(i.targets), t(case.old), t(case.ref), t(i.adv), t(i.mask),
                  workspace=a["workspace"], outputs=outs, per_token=False)
    assert e.value.code == R.EINVAL
    torch.cuda.synchronize()
    assert torch.isnan(buf).all()


def test_backward_without_gradient_rows(R):
    """All advantages 0 and no KL: every c_n is 0, nothing is kept, and dX,
    dW, db come out exactly zero, in one chunk and in several."""
    spec = MID[1].with_(beta=0.0)
    case = Case(spec)
    case.inp.adv.zero_()
    for chunk in (0, 128):
        out = case.run_gpu(R, chunk_rows=chunk)
        assert out["status"] == 0, hex(out["status"])
        assert out["loss"].item() == 0.0
        for k in ("dX", "dW", "db"):
            assert torch.count_nonzero(out[k]) == 0, (chunk, k)


def test_compaction_with_empty_later_chunks(R):
    """Most rows are prompt: the kept rows fit in the first 256-row chunk and
    the later chunks have none.  Matches the dense backward and the oracle."""
    spec = Workload("mostly_prompt", B=2, T=640, H=128, V=900, dtype="bf16", prompt_len=560, seed=109)
    case = Case(spec)
    _full_check(R, case, chunk_rows=256)   # default call (stored probabilities where they apply)
    a, res, _ = _full_check(R, case, chunk_rows=256, flags=R.FLAG_RECOMPUTE)
    assert 0 < (res.c != 0).sum() <= 160
    b, _, _ = _full_check(R, case, chunk_rows=256, flags=R.FLAG_ALL_ROWS)
    _grads_close(a, b)


def _run_into(R, case, outs, **cfg_kw):
    i = case.inp
    cfg = parity_cfg(R, case.spec, **cfg_kw)
    t = lambda x: None if x is None else x.cuda()
    out = R.fwd_bwd(cfg, t(i.X), t(i.W), t(i.b), t(i.targets), t(case.old), t(case.ref), t(i.adv), t(i.mask),
                    outputs=outs)
    torch.cuda.synchronize()
    assert R.rlloss_get_device_status(out["workspace"]) == 0
    return out


@pytest.mark.parametrize("spec,all_rows,chunk", [(MID[1], False, 0), (MID[1], False, 128), (MID[1], True, 0),
                                                 (MID[4], False, 0), (MID[4], True, 128), (MID[3], False, 0)],
                         ids=["bias_k3kl", "bias_k3kl_chunks", "bias_k3kl_all_rows", "fp32_bias",
                              "fp32_bias_all_rows_chunks", "gspo"])
def test_accumulate_adds_gradients(R, spec, all_rows, chunk):
    """FLAG_ACCUMULATE adds the call's gradients to what dX, dW, db hold.
    The result is the initial values plus the overwriting call's gradients:
    bit for bit where each element gets a single addition (kept dX rows of
    the compacted backward; dW and db with one chunk), within fp32 rounding
    otherwise.  Rows without gradient keep their initial bits, and the same
    initial values give the same bits on every call."""
    case = Case(spec)
    # the overwriting call runs the same (recomputing) backward as ACCUMULATE
    base, res, _ = _full_check(R, case, chunk_rows=chunk,
                               flags=R.FLAG_ALL_ROWS if all_rows else R.FLAG_RECOMPUTE)
    g = torch.Generator().manual_seed(7)
    init = {k: torch.randn(base[k].shape, generator=g).cuda() for k in ("dX", "dW", "db") if base.get(k) is not None}
    flags = R.FLAG_ACCUMULATE | (R.FLAG_ALL_ROWS if all_rows else 0)
    runs = []
    for _ in range(2):
        outs = {k: v.clone() for k, v in base.items() if isinstance(v, torch.Tensor)}
        outs.update({k: v.clone() for k, v in init.items()})
        runs.append(_run_into(R, case, outs, chunk_rows=chunk, flags=flags))
    a, b = runs
    for k in init:
        assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), k
    for k in ("loss", "metrics"):
        assert torch.equal(a[k].view(torch.int32), base[k].view(torch.int32)), k
    one_chunk = chunk == 0
    exact = {"dX": not all_rows, "dW": one_chunk, "db": one_chunk}
    for k, v0 in init.items():
        want = v0 + base[k]
        if exact[k]:
            assert torch.equal(a[k].view(torch.int32), want.view(torch.int32)), k
        else:
            tol = 1e-6 * float(want.abs().max())
            assert torch.allclose(a[k], want, rtol=1e-5, atol=tol), k
    dropped = torch.from_numpy(res.c == 0).cuda()
    assert dropped.any()
    assert torch.equal(a["dX"][dropped], init["dX"][dropped])
    # the added part against the oracle
    added = dict(a)
    for k, v0 in init.items():
        added[k] = (a[k].double() - v0.double()).float()
    check_grads(added, case, res)


SKIP = [
    Workload("long_prompt_gmpo", B=2, T=640, H=128, V=900, dtype="bf16", prompt_len=560, seed=111),
    Workload("long_prompt_entropy", B=3, T=512, H=128, V=700, dtype="bf16", prompt_len=300, temperature=0.7,
             top_entropy_quantile=0.3, seed=112),
    Workload("long_prompt_gspo", B=4, T=512, H=64, V=600, dtype="bf16", loss_type=GSPO_TOKEN, eps_low=3e-4,
             eps_high=4e-4, prompt_len=280, old_noise_std=0.02, seed=113),
    Workload("long_prompt_fp32_bias", B=2, T=600, H=100, V=515, dtype="fp32", has_bias=True, bias_std=0.1,
             prompt_len=520, seed=114),
]


@pytest.mark.parametrize("spec", SKIP, ids=[s.name for s in SKIP])
def test_forward_skips_fully_masked_tiles(R, spec):
    """Without per-token outputs the forward runs only over row tiles that
    hold an unmasked row; loss, metrics and gradients match the oracle and the
    run with per-token outputs (which computes every tile)."""
    case = Case(spec)
    a = case.run_gpu(R, per_token=False)
    assert a["status"] == 0, hex(a["status"])
    tiles = -(-spec.N // 256)
    assert R.rlloss_get_forward_tiles(a["workspace"]) < tiles
    res = reconcile_loss(a, case)
    check_loss_and_metrics(a, case, res)
    check_grads(a, case, res)
    b, _, _ = _full_check(R, case)
    assert R.rlloss_get_forward_tiles(b["workspace"]) == tiles
    assert abs(a["loss"].item() - b["loss"].item()) <= 1e-6 * abs(b["loss"].item()) + 1e-9
    _grads_close(a, b)


@pytest.mark.parametrize("spec", [MID[1], MID[2]], ids=["bias_k3kl", "entropy_mask"])
def test_cuda_graph_capture_and_replay(R, spec):
    """A fwd_bwd call captured in a CUDA graph (every operation of the call is
    stream-ordered and allocation-free) replays to the eager call's bits, and
    picks up new input values written in place between replays."""
    case = Case(spec)
    i = case.inp
    c = lambda x: None if x is None else x.cuda()
    X, W, b, y, old, ref, adv, mask = map(c, (i.X, i.W, i.b, i.targets, case.old, case.ref, i.adv, i.mask))
    cfg = parity_cfg(R, spec)
    ws = R.alloc_workspace(R.rlloss_workspace_bytes(cfg), "cuda")
    eager = R.fwd_bwd(cfg, X, W, b, y, old, ref, adv, mask, workspace=ws, per_token=False)
    ref_out = {k: v.clone() for k, v in eager.items() if k != "workspace" and v is not None}
    outs = {k: v for k, v in eager.items() if k != "workspace"}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        R.fwd_bwd(cfg, X, W, b, y, old, ref, adv, mask, workspace=ws, outputs=outs, per_token=False)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        R.fwd_bwd(cfg, X, W, b, y, old, ref, adv, mask, workspace=ws, outputs=outs, per_token=False)
    for v in outs.values():
        if v is not None:
            v.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert R.rlloss_get_device_status(ws) == 0
    for k, v in ref_out.items():
        assert torch.equal(outs[k].view(torch.int32) if outs[k].dtype == torch.float32 else outs[k],
                           v.view(torch.int32) if v.dtype == torch.float32 else v), k
    adv.neg_()                                   # new advantages, same buffers
    g.replay()
    torch.cuda.synchronize()
    fresh = R.fwd_bwd(cfg, X, W, b, y, old, ref, adv, mask, per_token=False)
    for k in ("loss", "dX", "dW"):
        assert torch.equal(outs[k], fresh[k]), k


# ------------------------------------------------------------------ loss stage only
def _loss_gpu(R, cfg, logp, old, adv, mask, entropy=None, ref=None):
    c = lambda x: None if x is None else torch.as_tensor(x).cuda()
    o = R.loss_from_logp(cfg, c(logp), c(entropy), c(old), c(ref), c(adv), c(mask))
    torch.cuda.synchronize()
    o["status"] = R.rlloss_get_device_status(o["workspace"])
    return o


@pytest.mark.parametrize("side", ["high", "low"])
def test_exact_clip_boundaries_loss_stage(R, side):
    """lr == bound exactly (Sterbenz: logp = -b, old = -2b) is unclipped with full
    gradient; the next fp32 value outward clips.  Decisions and gradients are
    compared exactly, the loss to the oracle's value rounded to fp32."""
    eps = 0.4
    ef = np.float32(eps)
    A = 1.0 if side == "high" else -1.0
    bound = ef if A > 0 else -ef
    old = np.float32(-2 * ef) if A > 0 else np.float32(-ef)
    on = np.float32(old + bound)
    assert float(on) - float(old) == float(bound)
    out_v = np.nextafter(on, np.float32(np.inf if A > 0 else -np.inf))
    in_v = np.nextafter(on, np.float32(-np.inf if A > 0 else np.inf))
    logp = np.array([on, out_v, in_v, on], np.float32)
    oldv = np.full(4, old, np.float32)
    adv = np.array([A], np.float32)
    mask = np.ones(4, np.uint8)
    cfg = R.make_cfg(1, 4, eps_low=eps, eps_high=eps)
    g = _loss_gpu(R, cfg, logp, oldv, adv, mask)
    o = O.gmpo_loss(logp.astype(np.float64), oldv.astype(np.float64), None, adv.astype(np.float64), mask, 1, 4,
                    eps, eps)
    assert g["status"] == 0
    assert g["metrics"][1].item() == o.metrics[1] == 1
    gd = g["dlogp"].cpu().numpy()
    assert np.array_equal(gd == 0, o.c == 0)
    assert np.allclose(gd, o.c, rtol=1e-6, atol=0)
    assert g["loss"].item() == pytest.approx(np.float32(o.loss), rel=1e-7)


def test_gspo_clip_bounds_loss_stage(R):
    """GSPO: sequence ratios exactly on each fp32 clip bound and one fp64 ulp
    either side, under both advantage signs (Tinker "GSPO", objective formula
    and "Choosing clipping thresholds").  The log ratios are fp32 pieces whose
    masked mean is, exactly, the fp64 preimage of the target ratio.  Clip
    decisions, the zero pattern of dL/dlogp and its values must equal the
    oracle's; the oracle's ratios are asserted to sit on the targets."""
    from exact_bounds import gspo_sequences_on_bounds
    lo, hi = O.f32(1 - 3e-4), O.f32(1 + 4e-4)
    targets, lp1, old1, m1 = gspo_sequences_on_bounds(lo, hi)
    k, T = lp1.shape
    B = 2 * k
    logp = np.concatenate([lp1, lp1]).reshape(-1)
    old = np.concatenate([old1, old1]).reshape(-1)
    mask = np.concatenate([m1, m1]).reshape(-1)
    adv = np.concatenate([np.full(k, 1.0), np.full(k, -1.0)]).astype(np.float32)
    o = O.gspo_token_loss(logp.astype(np.float64), old.astype(np.float64), adv.astype(np.float64), mask, B, T)
    assert np.array_equal(np.exp(o.seq_log_ratio), np.concatenate([targets, targets]))
    assert o.metrics[1] == 4
    cfg = R.make_cfg(B, T, loss_type=R.GSPO_TOKEN, eps_low=3e-4, eps_high=4e-4)
    g = _loss_gpu(R, cfg, logp, old, adv, mask)
    assert g["status"] == 0
    assert g["metrics"][1].item() == o.metrics[1]
    gd = g["dlogp"].cpu().numpy()
    assert np.array_equal(gd == 0, o.c == 0)
    assert np.array_equal(gd, o.c.astype(np.float32))
    assert g["loss"].item() == pytest.approx(o.loss, rel=1e-6)
    # one sequence at a time: the ratio the GPU formed is the target itself
    for i in (1, 4):
        sl = slice(i * T, (i + 1) * T)
        g1 = _loss_gpu(R, R.make_cfg(1, T, loss_type=R.GSPO_TOKEN, eps_low=3e-4, eps_high=4e-4),
                       logp[sl], old[sl], adv[i:i + 1], mask[sl])
        assert g1["metrics"][7].item() == np.float32(targets[i]) and g1["metrics"][1].item() == 0


def test_quantile_beyond_2_24_elements_exact(R):
    """2^24 + 1 active entropies (past torch.quantile's cap): threshold and mask
    against a sort of the same fp32 values ("support top_entropy_quantile",
    Details: the sort fallback beyond the 2^24-element cap)."""
    n = (1 << 24) + 1
    H = random_entropies(n, seed=11)
    mask = torch.ones(n, dtype=torch.uint8)
    mask[::7] = 0
    logp = torch.full((n,), -11.0)
    old = logp.clone()
    adv = torch.ones(1)
    cfg = R.make_cfg(1, n, top_entropy_quantile=0.2)
    g = _loss_gpu(R, cfg, logp, old, adv, mask, entropy=H)
    thr, e = O.entropy_threshold(H.double().numpy(), mask.numpy(), 0.2)
    assert g["status"] == 0
    assert g["metrics"][4].item() == np.float32(thr)
    assert np.array_equal(g["emask"].cpu().numpy(), e)
    assert g["metrics"][5].item() == e.sum()


def test_quantile_small_cases_exact(R):
    rng = np.random.default_rng(12)
    for n, q in ((1, 0.2), (2, 0.5), (5, 0.0), (5, 1.0), (1000, 0.37), (4097, 0.8)):
        H = rng.normal(3.0, 1.0, n).astype(np.float32)
        H[: n // 3] = H[0]                       # ties
        mask = (rng.uniform(size=n) < 0.9).astype(np.uint8)
        cfg = R.make_cfg(1, n, top_entropy_quantile=q, flags=R.FLAG_FORCE_ENTROPY_PATH)
        g = _loss_gpu(R, cfg, np.full(n, -2.0, np.float32), np.full(n, -2.0, np.float32),
                      np.ones(1, np.float32), mask, entropy=H)
        thr, e = O.entropy_threshold(H.astype(np.float64), mask, q)
        assert np.array_equal(g["emask"].cpu().numpy(), e), (n, q)
        if mask.sum():
            assert g["metrics"][4].item() == np.float32(thr), (n, q)


def test_empty_active_set(R):
    n = 64
    cfg = R.make_cfg(2, 32, top_entropy_quantile=0.3)
    g = _loss_gpu(R, cfg, np.full(n, -2.0, np.float32), np.full(n, -2.0, np.float32), np.ones(2, np.float32),
                  np.zeros(n, np.uint8), entropy=np.ones(n, np.float32))
    assert g["status"] == 0
    assert np.isnan(g["metrics"][4].item())
    assert g["emask"].sum().item() == 0
    assert g["loss"].item() == 0.0


def test_gspo_empty_sequence_flags_status(R):
    cfg = R.make_cfg(2, 4, loss_type=R.GSPO_TOKEN, eps_low=3e-4, eps_high=4e-4)
    mask = np.array([1, 1, 1, 1, 0, 0, 0, 0], np.uint8)
    g = _loss_gpu(R, cfg, np.full(8, -2.0, np.float32), np.full(8, -2.0, np.float32), np.ones(2, np.float32), mask)
    assert g["status"] & R.DEV_EEMPTYSEQ
