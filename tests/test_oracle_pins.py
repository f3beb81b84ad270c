"""Pins for the fp64 oracle against what the pages and the mathematics fix.

Each test ties one part of the oracle to something other than itself: a closed
form, a brute-force evaluation, a library routine computing the same textbook
quantity, finite differences, or autograd of an independent full-logits
restatement.  A dropped term, a wrong sign or index, or a transposed operand
in the oracle fails at least one of these.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand_problem(rng, N, H, V, bias=True):
    X = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H)) * 0.3
    b = rng.standard_normal(V) * 0.1 if bias else None
    y = rng.integers(0, V, N)
    return X, W, b, y


# --- per-row stats ------------------------------------------------------------

def test_uniform_logits_closed_form():
    """W = 0, b = 0: every logit is 0, so lse = H = log V and logp = -log V."""
    V, H, N = 37, 5, 4
    X = np.random.default_rng(0).standard_normal((N, H))
    lse, logp, ent = O.row_stats(X, np.zeros((V, H)), np.zeros(V), np.arange(N) % V, 0.7)
    assert np.allclose(lse, math.log(V), atol=1e-14, rtol=0)
    assert np.allclose(logp, -math.log(V), atol=1e-14, rtol=0)
    assert np.allclose(ent, math.log(V), atol=1e-14, rtol=0)


def test_one_hot_logit_has_zero_entropy():
    """One logit 1000 above the rest: p is one-hot in fp64, so H = 0, logp(hot) = 0."""
    V, H = 9, 3
    X = np.zeros((2, H)); W = np.zeros((V, H)); b = np.zeros(V); b[4] = 1000.0
    lse, logp, ent = O.row_stats(X, W, b, np.array([4, 2]), 1.0)
    assert ent[0] == pytest.approx(0.0, abs=1e-300)
    assert logp[0] == pytest.approx(0.0, abs=1e-12)
    assert logp[1] == pytest.approx(-1000.0, abs=1e-9)


def test_row_stats_brute_force():
    """A tiny case evaluated with scalar loops and math.fsum."""
    rng = np.random.default_rng(1)
    X, W, b, y = _rand_problem(rng, 3, 4, 6)
    tau = 0.8
    lse, logp, ent = O.row_stats(X, W, b, y, tau)
    for n in range(3):
        z = [(math.fsum(X[n, h] * W[v, h] for h in range(4)) + b[v]) / tau for v in range(6)]
        Z = math.fsum(math.exp(t) for t in z)
        p = [math.exp(t) / Z for t in z]
        assert lse[n] == pytest.approx(math.log(Z), abs=1e-13)
        assert logp[n] == pytest.approx(z[y[n]] - math.log(Z), abs=1e-13)
        assert ent[n] == pytest.approx(-math.fsum(pi * math.log(pi) for pi in p), abs=1e-13)


def test_row_stats_match_library_routines():
    """Entropy vs torch Categorical.entropy and vs -sum p log p; logp vs log_softmax."""
    rng = np.random.default_rng(2)
    X, W, b, y = _rand_problem(rng, 70, 16, 300)
    tau = 0.7
    lse, logp, ent = O.row_stats(X, W, b, y, tau)
    z = O.logits_rows(X, W, b, tau, np.arange(70))
    zt = torch.from_numpy(z)
    ref_ent = torch.distributions.Categorical(logits=zt).entropy().numpy()
    ref_logp = torch.log_softmax(zt, -1)[torch.arange(70), torch.from_numpy(y)].numpy()
    assert np.allclose(ent, ref_ent, atol=1e-12, rtol=0)
    assert np.allclose(ent, O.entropy_direct(z), atol=1e-12, rtol=0)
    assert np.allclose(logp, ref_logp, atol=1e-12, rtol=0)
    assert np.allclose(lse, torch.logsumexp(zt, -1).numpy(), atol=1e-12, rtol=0)


def test_row_stats_threaded_equals_serial():
    rng = np.random.default_rng(3)
    X, W, b, y = _rand_problem(rng, 300, 8, 50)
    a = O.row_stats(X, W, b, y, 1.0, threads=1)
    c = O.row_stats(X, W, b, y, 1.0, threads=4)
    for u, v in zip(a, c):
        assert np.array_equal(u, v)


# --- GMPO ---------------------------------------------------------------------

def test_gmpo_zero_log_ratio_closed_form():
    """All lr = 0 with constant A: r_i = 1 exactly, so L = -A (beta = 0)."""
    B, T = 3, 7
    logp = np.random.default_rng(4).uniform(-12, -1, B * T)
    mask = np.ones(B * T, np.uint8); mask[:2] = 0
    for A in (1.0, -0.5, 2.25):
        r = O.gmpo_loss(logp, logp.copy(), None, np.full(B, A), mask, B, T, 0.4, 0.4)
        assert r.loss == -A
        assert np.all(r.metrics[7] == 1.0)
        assert r.metrics[1] == 0


def test_gmpo_kl_vanishes_when_ref_equals_policy():
    B, T = 2, 5
    rng = np.random.default_rng(5)
    logp = rng.uniform(-5, -1, B * T)
    old = logp + rng.normal(0, 0.1, B * T)
    mask = np.ones(B * T, np.uint8)
    a = O.gmpo_loss(logp, old, logp.copy(), np.array([1.0, -1.0]), mask, B, T, 0.2, 0.3, beta=0.04)
    z = O.gmpo_loss(logp, old, None, np.array([1.0, -1.0]), mask, B, T, 0.2, 0.3, beta=0.0)
    assert a.metrics[2] == 0.0
    assert a.loss == z.loss
    assert np.array_equal(a.c, z.c)


def test_gmpo_geometric_mean_by_hand():
    """One sequence, A = +1, eps_high = 0.25: clr = [0.25, -0.1, 0.2] (first clipped)."""
    eh = O.f32(0.25)
    logp = np.array([-1.0, -2.0, -3.0]); old = logp - np.array([0.5, -0.1, 0.2])
    r = O.gmpo_loss(logp, old, None, np.array([1.0]), np.ones(3, np.uint8), 1, 3, 0.25, 0.25)
    lr = logp - old
    expect_r = math.exp((eh + lr[1] + lr[2]) / 3)
    assert r.loss == pytest.approx(-expect_r, rel=1e-15)
    assert r.metrics[1] == 1 and r.metrics[0] == pytest.approx(1 / 3)
    assert r.c[0] == 0.0
    assert r.c[1] == pytest.approx(-expect_r / 3, rel=1e-15)


@pytest.mark.parametrize("side", ["high", "low"])
def test_gmpo_exact_clip_boundary_and_neighbours(side):
    """lr == bound exactly is unclipped with gradient 1; the next float outward clips.

    Mirrors the pages' exact-boundary tests ("Add GMPO ...", Details: exact
    clipping boundaries and adjacent torch.nextafter values)."""
    eps = 0.4
    ef = np.float32(eps)
    A = 1.0 if side == "high" else -1.0
    bound = ef if side == "high" else -ef
    # old = logp - bound exactly: with logp = -bound... choose logp = -(2|b|)*sign so lr = bound
    old = np.float32(-2 * ef) if side == "high" else np.float32(-ef)
    logp_on = np.float32(old + bound)
    assert float(logp_on) - float(old) == float(bound)
    outward = np.nextafter(logp_on, np.float32(np.inf if side == "high" else -np.inf))
    inward = np.nextafter(logp_on, np.float32(-np.inf if side == "high" else np.inf))
    res = {}
    for name, lp in (("on", logp_on), ("out", outward), ("in", inward)):
        r = O.gmpo_loss(np.array([lp], np.float64), np.array([old], np.float64), None,
                        np.array([A]), np.ones(1, np.uint8), 1, 1, eps, eps)
        res[name] = r
    assert res["on"].metrics[1] == 0 and res["in"].metrics[1] == 0 and res["out"].metrics[1] == 1
    assert res["on"].c[0] != 0.0 and res["in"].c[0] != 0.0 and res["out"].c[0] == 0.0
    # clipped loss equals the loss at the bound
    assert res["out"].loss == res["on"].loss


def test_gmpo_extreme_clipped_ratios_are_finite():
    B, T = 2, 4
    logp = np.full(B * T, -3.0)
    old = logp.copy(); old[:T] -= 50.0; old[T:] += 50.0     # seq0 lr=+50 (A>0), seq1 lr=-50 (A<0)
    r = O.gmpo_loss(logp, old, None, np.array([1.0, -1.0]), np.ones(B * T, np.uint8), B, T, 0.4, 0.4)
    assert np.isfinite(r.loss) and np.all(np.isfinite(r.c))
    assert r.metrics[1] == B * T
    assert np.all(r.c == 0.0)


def test_gmpo_zero_advantage_never_clips():
    logp = np.array([-1.0, -1.0]); old = logp - np.array([5.0, -5.0])
    r = O.gmpo_loss(logp, old, None, np.array([0.0]), np.ones(2, np.uint8), 1, 2, 0.4, 0.4)
    assert r.metrics[1] == 0 and r.loss == 0.0 and np.all(r.c == 0.0)


def test_gmpo_empty_sequence_contributes_zero_and_counts_in_B():
    B, T = 2, 3
    logp = np.full(6, -2.0); old = logp.copy()
    mask = np.array([0, 0, 0, 1, 1, 1], np.uint8)
    r = O.gmpo_loss(logp, old, None, np.array([1.0, 1.0]), mask, B, T, 0.4, 0.4)
    assert r.loss == pytest.approx(-0.5)
    assert np.all(r.c[:3] == 0)


# --- entropy quantile ---------------------------------------------------------

def test_quantile_matches_torch_quantile():
    rng = np.random.default_rng(6)
    H = rng.normal(11.56, 0.017, 5000)
    m = (rng.uniform(size=5000) < 0.8).astype(np.uint8)
    for q in (0.0, 0.2, 0.5, 0.8, 1.0, 0.37):
        thr, e = O.entropy_threshold(H, m, q)
        ref = torch.quantile(torch.from_numpy(H[m != 0]), 1 - q, interpolation="linear").item()
        assert thr == pytest.approx(ref, abs=1e-12)
        assert np.array_equal(e, (m != 0) & (H >= thr))


def test_quantile_one_keeps_every_active_token_and_is_a_noop():
    """q = 1 is bit-identical to the mask being off ("support top_entropy_quantile", Details)."""
    rng = np.random.default_rng(7)
    B, T = 3, 50
    H = rng.normal(11.5, 0.02, B * T)
    mask = (rng.uniform(size=B * T) < 0.7).astype(np.uint8)
    thr, e = O.entropy_threshold(H, mask, 1.0)
    assert thr == H[mask != 0].min()
    assert np.array_equal(e, mask)
    logp = rng.uniform(-12, -10, B * T); old = logp + rng.normal(0, 0.3, B * T)
    adv = rng.normal(size=B)
    a = O.gmpo_loss(logp, old, None, adv, mask, B, T, 0.4, 0.4, entropy=H, q=1.0)
    b_ = O.gmpo_loss(logp, old, None, adv, mask, B, T, 0.4, 0.4)
    assert a.loss == b_.loss and np.array_equal(a.c, b_.c)
    assert np.array_equal(a.metrics[:4], b_.metrics[:4])


def test_quantile_is_batch_global_not_per_chunk():
    rng = np.random.default_rng(8)
    B, T = 4, 64
    H = rng.normal(11.5, 0.02, (B, T)) + np.arange(B)[:, None] * 0.01
    m = np.ones((B, T), np.uint8)
    thr_all, e_all = O.entropy_threshold(H.reshape(-1), m.reshape(-1), 0.2)
    # permuting the batch (any chunking order) leaves the threshold unchanged
    perm = rng.permutation(B)
    thr_perm, _ = O.entropy_threshold(H[perm].reshape(-1), m[perm].reshape(-1), 0.2)
    assert thr_perm == thr_all
    # per-chunk thresholds differ, so a chunked quantile would not be equivalent
    per_chunk = [O.entropy_threshold(H[i], m[i], 0.2)[0] for i in range(B)]
    assert any(t != thr_all for t in per_chunk)
    # non-vacuous: some but not all active tokens are dropped
    assert 0 < e_all.sum() < m.sum()


def test_quantile_empty_active_set():
    thr, e = O.entropy_threshold(np.ones(5), np.zeros(5, np.uint8), 0.2)
    assert math.isnan(thr) and e.sum() == 0


def test_quantile_range_validation():
    with pytest.raises(ValueError):
        O.entropy_threshold(np.ones(3), np.ones(3), 1.5)
    with pytest.raises(ValueError):
        O.gmpo_loss(np.ones(2), np.ones(2), None, np.ones(1), np.ones(2), 1, 2, 0.4, 0.4,
                    entropy=np.ones(2), q=-0.1)


def test_entropy_mask_scales_policy_term():
    """Reading R7: with a kept fraction ebar_i, the sequence term is -A_i r_i ebar_i."""
    B, T = 1, 4
    logp = np.full(4, -2.0); old = logp.copy()
    H = np.array([1.0, 2.0, 3.0, 4.0])
    r = O.gmpo_loss(logp, old, None, np.array([2.0]), np.ones(4, np.uint8), B, T, 0.4, 0.4,
                    entropy=H, q=0.25)
    # pos = 0.75 * 3 = 2.25 -> thr = 3.25 -> keep only H=4 -> ebar = 1/4
    assert r.metrics[4] == pytest.approx(3.25)
    assert r.metrics[5] == 1
    assert r.loss == pytest.approx(-2.0 * 1.0 * 0.25)


# --- GSPO ---------------------------------------------------------------------

def test_gspo_zero_log_ratio_closed_form():
    """All lr = 0: s_i = 1 (inside the clip range), so L = -sum_n A_n."""
    B, T = 3, 6
    rng = np.random.default_rng(9)
    logp = rng.uniform(-12, -1, B * T)
    mask = np.ones(B * T, np.uint8); mask[::4] = 0
    adv = rng.normal(size=B)
    r = O.gspo_token_loss(logp, logp.copy(), adv, mask, B, T)
    An = (adv[:, None] * mask.reshape(B, T)).reshape(-1)
    assert r.loss == pytest.approx(-An.sum(), rel=1e-15)
    assert r.metrics[6] == 0.0 and r.metrics[7] == 1.0 and r.metrics[1] == 0
    assert np.allclose(r.c, -An, rtol=1e-15)


def test_gspo_default_clip_range_matches_page():
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))
    lo, hi = g["gspo_default_clip"]["low"], g["gspo_default_clip"]["high"]
    import inspect
    sig = inspect.signature(O.gspo_token_loss)
    assert 1 - sig.parameters["eps_low"].default == pytest.approx(lo, abs=1e-15)
    assert 1 + sig.parameters["eps_high"].default == pytest.approx(hi, abs=1e-15)


def _torch_gspo(logp, old, adv, mask, B, T, lo, hi, per_token=False):
    """Independent autograd statement of GSPO-token: stop-gradient via detach."""
    lp = logp.reshape(B, T); m = mask.reshape(B, T)
    seq = ((lp.detach() - old.reshape(B, T)) * m).sum(1) / m.sum(1)
    ratio = torch.exp(seq[:, None] + lp - lp.detach())
    An = adv.reshape(B, T) if per_token else adv[:, None] * m
    obj = torch.minimum(ratio * An, torch.clamp(ratio, lo, hi) * An)
    return -obj.sum()


def test_gspo_gradient_matches_autograd():
    rng = np.random.default_rng(10)
    B, T = 4, 9
    logp = rng.uniform(-3, -1, B * T)
    mask = np.ones(B * T, np.uint8); mask[:2] = 0
    adv = np.array([1.0, -1.0, 0.7, -0.3])
    # sequence ratios well away from the bounds: two clipped high, one low, one inside
    shift = np.repeat([3e-3, 3e-3, -3e-3, 1e-5], T)
    old = logp - shift
    r = O.gspo_token_loss(logp, old, adv, mask, B, T)
    lp_t = torch.tensor(logp, requires_grad=True)
    L = _torch_gspo(lp_t, torch.tensor(old), torch.tensor(adv), torch.tensor(mask, dtype=torch.float64),
                    B, T, O.f32(1 - 3e-4), O.f32(1 + 4e-4))
    L.backward()
    assert r.loss == pytest.approx(L.item(), rel=1e-14)
    assert np.allclose(r.c, lp_t.grad.numpy(), rtol=1e-14, atol=0)
    assert r.metrics[1] == 3


def test_gspo_per_token_advantages_match_autograd_and_reduce_to_per_sequence():
    rng = np.random.default_rng(14)
    B, T = 3, 8
    logp = rng.uniform(-3, -1, B * T)
    mask = np.ones(B * T, np.uint8); mask[[0, 1, 8]] = 0
    old = logp - np.repeat([3e-3, -3e-3, 1e-5], T)
    An = rng.normal(size=B * T)                 # per-token, including some outside the ratio mask
    r = O.gspo_token_loss(logp, old, An, mask, B, T, per_token_adv=True)
    lp_t = torch.tensor(logp, requires_grad=True)
    L = _torch_gspo(lp_t, torch.tensor(old), torch.tensor(An), torch.tensor(mask, dtype=torch.float64), B, T,
                    O.f32(1 - 3e-4), O.f32(1 + 4e-4), per_token=True)
    L.backward()
    assert r.loss == pytest.approx(L.item(), rel=1e-14)
    assert np.allclose(r.c, lp_t.grad.numpy(), rtol=1e-14, atol=0)
    # per-sequence advantages broadcast on the mask are the special case A_n = A_i m_n
    adv = rng.normal(size=B)
    a = O.gspo_token_loss(logp, old, adv, mask, B, T)
    b_ = O.gspo_token_loss(logp, old, (adv[:, None] * mask.reshape(B, T)).reshape(-1), mask, B, T,
                           per_token_adv=True)
    assert a.loss == b_.loss and np.array_equal(a.c, b_.c)


def test_gspo_exact_bounds_and_neighbours_match_autograd():
    """Sequence ratios exactly on the fp32 clip bounds and one fp64 ulp either side.

    Tinker "GSPO", objective formula and "Choosing clipping thresholds": the
    objective is min(s A, clip(s, lo, hi) A).  Autograd of that formula decides
    the gradient at the bound itself: the clamp's gradient is inclusive and the
    minimum ties, so the gradient passes in full (reading R12).  The clip
    diagnostic counts ratios strictly outside the range (reading R17)."""
    from exact_bounds import gspo_sequences_on_bounds
    lo, hi = O.f32(1 - 3e-4), O.f32(1 + 4e-4)
    targets, lp1, old1, m1 = gspo_sequences_on_bounds(lo, hi)
    k, T = lp1.shape
    # every ratio under both advantage signs: sequences 0..k-1 with A = +1, k..2k-1 with A = -1
    logp = np.concatenate([lp1, lp1]).astype(np.float64).reshape(-1)
    old = np.concatenate([old1, old1]).astype(np.float64).reshape(-1)
    mask = np.concatenate([m1, m1]).reshape(-1)
    B = 2 * k
    adv = np.concatenate([np.ones(k), -np.ones(k)])
    r = O.gspo_token_loss(logp, old, adv, mask, B, T)
    s = np.exp(r.seq_log_ratio)
    assert np.array_equal(s, np.concatenate([targets, targets]))        # on the bound, exactly
    lp_t = torch.tensor(logp, requires_grad=True)
    L = _torch_gspo(lp_t, torch.tensor(old), torch.tensor(adv), torch.tensor(mask, dtype=torch.float64),
                    B, T, lo, hi)
    L.backward()
    seq_t = ((torch.tensor(logp) - torch.tensor(old)).reshape(B, T) * torch.tensor(m1.astype(np.float64)).repeat(2, 1)
             ).sum(1) / 4.0
    assert np.array_equal(torch.exp(seq_t).numpy(), s)                  # autograd sees the same ratios
    g = lp_t.grad.numpy()
    assert r.loss == pytest.approx(L.item(), rel=1e-15)
    assert np.array_equal(r.c == 0, g == 0)
    assert np.allclose(r.c, g, rtol=1e-15, atol=0)
    # the gradient stops only on the flat side of the clamp, strictly past the bound
    flat = np.zeros(B, bool)
    flat[5] = True          # A > 0, s = next(hi)
    flat[k + 0] = True      # A < 0, s = prev(lo)
    active = mask.reshape(B, T) != 0
    assert np.array_equal((g.reshape(B, T) == 0) & active, flat[:, None] & active)
    # strict "outside": prev(lo) and next(hi) count, the bounds themselves do not
    out = (s < lo) | (s > hi)
    assert out.sum() == 4 and not out[[1, 4, k + 1, k + 4]].any()
    assert r.metrics[1] == 4 and np.array_equal(r.clipped, out)


def test_gspo_requires_active_token_per_sequence():
    with pytest.raises(ValueError):
        O.gspo_token_loss(np.ones(4), np.ones(4), np.ones(2), np.array([1, 1, 0, 0]), 2, 2)


# --- gradients ------------------------------------------------------------------

def _torch_gmpo_full(X, W, b, y, old, ref, adv, mask, B, T, tau, el, eh, beta, keep=None):
    """Independent full-logits autograd statement of GMPO.  ``keep`` is a fixed
    0/1 entropy-mask vector (no gradient flows through a threshold decision);
    it scales each sequence's policy term by its kept fraction."""
    z = (X @ W.T + b) / tau
    logp = torch.log_softmax(z, -1).gather(1, y[:, None])[:, 0].reshape(B, T)
    m = mask.reshape(B, T)
    lr = logp - old.reshape(B, T)
    A = adv[:, None]
    clr = torch.where(A > 0, torch.clamp(lr, max=eh), torch.where(A < 0, torch.clamp(lr, min=-el), lr))
    n = m.sum(1)
    r = torch.exp((clr * m).sum(1) / n)
    ebar = torch.ones_like(n) if keep is None else (keep.reshape(B, T) * m).sum(1) / n
    d = ref.reshape(B, T) - logp
    kl = torch.exp(d) - d - 1
    return (-adv * r * ebar + beta * (kl * m).sum(1) / n).mean()


def _small_gmpo_case(seed):
    rng = np.random.default_rng(seed)
    B, T, H, V = 2, 5, 6, 11
    X, W, b, y = _rand_problem(rng, B * T, H, V)
    tau = 0.7
    _, logp, _ = O.row_stats(X, W, b, y, tau)
    # log ratios placed at least 0.05 away from the clip bounds
    lr = rng.choice([-0.6, -0.1, 0.05, 0.15, 0.7], size=B * T)
    old = logp - lr
    ref = logp + rng.normal(0, 0.1, B * T)
    mask = np.ones(B * T, np.uint8); mask[[0, 5]] = 0
    adv = np.array([1.0, -0.5])
    return B, T, X, W, b, y, tau, old, ref, mask, adv


def test_gradients_match_autograd_of_full_logits():
    B, T, X, W, b, y, tau, old, ref, mask, adv = _small_gmpo_case(11)
    prob = O.Problem(B, T, O.GMPO, 0.2, 0.3, 0.04, tau)
    out = O.fwd_bwd(prob, X, W, b, y, old, ref, adv, mask)
    Xt, Wt, bt = (torch.tensor(a, requires_grad=True) for a in (X, W, b))
    L = _torch_gmpo_full(Xt, Wt, bt, torch.tensor(y), torch.tensor(old), torch.tensor(ref),
                         torch.tensor(adv), torch.tensor(mask, dtype=torch.float64), B, T, tau,
                         O.f32(0.2), O.f32(0.3), 0.04)
    L.backward()
    assert out["loss"] == pytest.approx(L.item(), rel=1e-13)
    assert np.allclose(out["dX"], Xt.grad.numpy(), rtol=1e-10, atol=1e-14)
    assert np.allclose(out["dW"], Wt.grad.numpy(), rtol=1e-10, atol=1e-14)
    assert np.allclose(out["db"], bt.grad.numpy(), rtol=1e-10, atol=1e-14)


@pytest.mark.parametrize("loss_type", [O.GMPO, O.GSPO_TOKEN])
def test_gradients_match_central_finite_differences(loss_type):
    B, T, X, W, b, y, tau, old, ref, mask, adv = _small_gmpo_case(12)
    if loss_type == O.GMPO:
        prob = O.Problem(B, T, O.GMPO, 0.2, 0.3, 0.04, tau)
    else:
        # sequence ratios far from the clip bounds in both directions
        _, logp, _ = O.row_stats(X, W, b, y, tau)
        old = logp - np.repeat([2e-2, -3e-5], T)
        prob = O.Problem(B, T, O.GSPO_TOKEN, 3e-4, 4e-4, 0.0, tau)
        ref = None
    out = O.fwd_bwd(prob, X, W, b, y, old, ref, adv, mask)

    def L(X_, W_, b_):
        _, lp, ent = O.row_stats(X_, W_, b_, y, tau)
        return O.loss_stage(prob, lp, ent, old, ref, adv, mask).loss

    h = 1e-6
    for name, arr, g in (("X", X, out["dX"]), ("W", W, out["dW"]), ("b", b, out["db"])):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            save = arr[idx]
            arr[idx] = save + h; up = L(X, W, b)
            arr[idx] = save - h; dn = L(X, W, b)
            arr[idx] = save
            fd[idx] = (up - dn) / (2 * h)
        assert np.allclose(g, fd, rtol=1e-6, atol=1e-9), name


def _masked_gmpo_case():
    """B=2, T=8, seven active tokens a sequence, q = 0.2 keeps 2 and 1 of them;
    every active entropy lies at least 7e-3 from the threshold and from its
    neighbours, and every log ratio at least 0.05 from a clip bound."""
    rng = np.random.default_rng(0)
    B, T, H, V = 2, 8, 6, 11
    X, W, b, y = _rand_problem(rng, B * T, H, V)
    tau = 0.7
    _, logp, _ = O.row_stats(X, W, b, y, tau)
    lr = np.random.default_rng(100).choice([-0.6, -0.1, 0.05, 0.15, 0.7], size=B * T)
    old = logp - lr
    ref = logp + np.random.default_rng(101).normal(0, 0.1, B * T)
    mask = np.ones(B * T, np.uint8); mask[[0, T]] = 0
    adv = np.array([1.0, -0.5])
    return B, T, X, W, b, y, tau, old, ref, mask, adv


def _torch_entropy_mask(X, W, b, tau, mask, q):
    """The entropy mask from torch alone: Categorical entropy of the logits and
    torch.quantile (linear) of the active entropies at 1 - q; keep H >= thr."""
    z = (torch.tensor(X) @ torch.tensor(W).T + torch.tensor(b)) / tau
    Hs = torch.distributions.Categorical(logits=z).entropy()
    act = torch.tensor(mask) != 0
    thr = torch.quantile(Hs[act], 1 - q, interpolation="linear")
    return (act & (Hs >= thr)).to(torch.float64), Hs.numpy(), thr.item()


def test_entropy_masked_gradients_match_autograd():
    """GMPO with the entropy mask at q = 0.2 and beta != 0 ("support
    top_entropy_quantile ...", Details: the mask multiplies the policy term
    after the loss-type branch, before the KL penalty).  Every entry of dX, dW,
    db and of c = dL/dlogp against autograd, with the mask taken from torch."""
    B, T, X, W, b, y, tau, old, ref, mask, adv = _masked_gmpo_case()
    q = 0.2
    keep, Hs, thr = _torch_entropy_mask(X, W, b, tau, mask, q)
    kept = keep.numpy().reshape(B, T).sum(1)
    assert kept.tolist() == [2, 1]                                  # the kept fractions differ
    act = np.sort(Hs[mask != 0])
    assert np.abs(act - thr).min() > 5e-3 and np.diff(act).min() > 5e-3
    prob = O.Problem(B, T, O.GMPO, 0.2, 0.3, 0.04, tau, q)
    out = O.fwd_bwd(prob, X, W, b, y, old, ref, adv, mask)
    assert np.array_equal(out["emask"], keep.numpy().astype(np.uint8))
    assert out["metrics"][4] == pytest.approx(thr, abs=1e-12)
    Xt, Wt, bt = (torch.tensor(a, requires_grad=True) for a in (X, W, b))
    z = (Xt @ Wt.T + bt) / tau
    lp_t = torch.log_softmax(z, -1).gather(1, torch.tensor(y)[:, None])[:, 0]
    lp_t.retain_grad()
    L = _torch_gmpo_full(Xt, Wt, bt, torch.tensor(y), torch.tensor(old), torch.tensor(ref),
                         torch.tensor(adv), torch.tensor(mask, dtype=torch.float64), B, T, tau,
                         O.f32(0.2), O.f32(0.3), 0.04, keep=keep)
    L.backward()
    assert out["loss"] == pytest.approx(L.item(), rel=1e-13)
    assert np.allclose(out["dX"], Xt.grad.numpy(), rtol=1e-10, atol=1e-14)
    assert np.allclose(out["dW"], Wt.grad.numpy(), rtol=1e-10, atol=1e-14)
    assert np.allclose(out["db"], bt.grad.numpy(), rtol=1e-10, atol=1e-14)
    # c itself: the gradient of the same statement with logp as the leaf
    lp_leaf = torch.tensor(out["logp"], requires_grad=True)
    m = torch.tensor(mask, dtype=torch.float64).reshape(B, T)
    lr = lp_leaf.reshape(B, T) - torch.tensor(old).reshape(B, T)
    A = torch.tensor(adv)[:, None]
    clr = torch.where(A > 0, torch.clamp(lr, max=O.f32(0.3)), torch.clamp(lr, min=-O.f32(0.2)))
    n = m.sum(1)
    r = torch.exp((clr * m).sum(1) / n)
    ebar = (keep.reshape(B, T) * m).sum(1) / n
    d = torch.tensor(ref).reshape(B, T) - lp_leaf.reshape(B, T)
    Lc = (-torch.tensor(adv) * r * ebar + 0.04 * ((torch.exp(d) - d - 1) * m).sum(1) / n).mean()
    Lc.backward()
    assert np.allclose(out["c"], lp_leaf.grad.numpy(), rtol=1e-12, atol=1e-16)
    # non-vacuous: the masked coefficient differs from the unmasked one on every unclipped active token
    nomask = O.gmpo_loss(out["logp"], old, ref, adv, mask, B, T, 0.2, 0.3, 0.04)
    live = (mask != 0) & (out["c"] != nomask.c)
    assert live.sum() == (mask != 0).sum() - out["clipped"].sum()


def test_entropy_masked_gradients_match_central_finite_differences():
    """The same masked case against central differences of the whole oracle
    (h = 1e-6; the mask is recomputed at every point and does not change,
    since no entropy lies within 5e-3 of the threshold or of another)."""
    B, T, X, W, b, y, tau, old, ref, mask, adv = _masked_gmpo_case()
    prob = O.Problem(B, T, O.GMPO, 0.2, 0.3, 0.04, tau, 0.2)
    out = O.fwd_bwd(prob, X, W, b, y, old, ref, adv, mask)
    base_mask = out["emask"].copy()

    def L(X_, W_, b_):
        _, lp, ent = O.row_stats(X_, W_, b_, y, tau)
        res = O.loss_stage(prob, lp, ent, old, ref, adv, mask)
        assert np.array_equal(res.emask, base_mask)
        return res.loss

    h = 1e-6
    for name, arr, g in (("X", X, out["dX"]), ("W", W, out["dW"]), ("b", b, out["db"])):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            save = arr[idx]
            arr[idx] = save + h; up = L(X, W, b)
            arr[idx] = save - h; dn = L(X, W, b)
            arr[idx] = save
            fd[idx] = (up - dn) / (2 * h)
        assert np.allclose(g, fd, rtol=1e-6, atol=1e-9), name


def test_db_sums_to_zero_and_sampled_rows_agree():
    B, T, X, W, b, y, tau, old, ref, mask, adv = _small_gmpo_case(13)
    prob = O.Problem(B, T, O.GMPO, 0.2, 0.3, 0.04, tau)
    out = O.fwd_bwd(prob, X, W, b, y, old, ref, adv, mask)
    assert abs(out["db"].sum()) < 1e-13
    rows = np.array([7, 1]); vs = np.array([3, 10, 0])
    dX, dW, db = O.grads(X, W, b, y, tau, out["lse"], out["c"], rows, vs)
    assert np.allclose(dX, out["dX"][rows], rtol=1e-13, atol=1e-15)
    assert np.allclose(dW, out["dW"][vs], rtol=1e-13, atol=1e-15)
    assert np.allclose(db, out["db"], rtol=1e-13, atol=1e-15)


# --- vocabulary shards ------------------------------------------------------

def _shard_bounds(sizes):
    cut = np.concatenate([[0], np.cumsum(sizes)]).astype(int)
    return [(int(cut[k]), int(cut[k + 1])) for k in range(len(sizes))]


def test_shard_states_merge_to_library_logsumexp_and_entropy():
    """States of uneven shards (one of a single row, one whose logits sit 60
    above the rest) merge, in any order, to scipy's logsumexp, the entropy
    -sum p log p of scipy's softmax, and the target log-prob."""
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(41)
    X, W, b, y = _rand_problem(rng, 40, 16, 300)
    b[150:151] += 60.0
    tau = 0.8
    sizes = [37, 113, 1, 149]
    states = [O.shard_state(X, W[v0:v1], b[v0:v1], y, tau, v0) for v0, v1 in _shard_bounds(sizes)]
    z = (X @ W.T + b) / tau
    lse_ref = logsumexp(z, axis=1)
    p = softmax(z, axis=1)
    ent_ref = -(p * np.log(p, where=p > 0, out=np.zeros_like(p))).sum(axis=1)
    for order in (states, states[::-1], [states[2], states[0], states[3], states[1]]):
        lse, logp, ent = O.merge_states(order, y, 300)
        assert np.allclose(lse, lse_ref, rtol=0, atol=1e-12)
        assert np.allclose(logp, z[np.arange(40), y] - lse_ref, rtol=0, atol=1e-12)
        assert np.allclose(ent, ent_ref, rtol=0, atol=1e-10)


def test_missing_shard_leaves_its_targets_without_logp():
    rng = np.random.default_rng(42)
    X, W, b, y = _rand_problem(rng, 30, 8, 90)
    bounds = _shard_bounds([30, 30, 30])
    states = [O.shard_state(X, W[v0:v1], b[v0:v1], y, 1.0, v0) for v0, v1 in bounds]
    _, logp, _ = O.merge_states([states[0], states[2]], y, 90)
    missing = (y >= 30) & (y < 60)
    assert missing.any() and (~missing).any()
    assert np.all(np.isnan(logp[missing])) and np.all(np.isfinite(logp[~missing]))
    y_bad = y.copy(); y_bad[0] = 90
    _, logp, _ = O.merge_states(states, y_bad, 90)
    assert np.isnan(logp[0]) and np.all(np.isfinite(logp[1:]))


def test_shard_gradients_sum_to_the_full_vocabulary_gradients():
    """dX is the sum of the shards' parts; dW and db are the shards' rows
    stacked (the full gradients are pinned to autograd above)."""
    B, T, X, W, b, y, tau, old, ref, mask, adv = _small_gmpo_case(14)
    prob = O.Problem(B, T, O.GMPO, 0.2, 0.3, 0.04, tau)
    out = O.fwd_bwd(prob, X, W, b, y, old, ref, adv, mask)
    V = W.shape[0]
    sizes = [V // 3, 1, V - V // 3 - 1]
    dX = np.zeros_like(out["dX"]); dWs = []; dbs = []
    for v0, v1 in _shard_bounds(sizes):
        px, pw, pb = O.shard_grads(X, W[v0:v1], b[v0:v1], y, tau, v0, out["lse"], out["c"])
        dX += px; dWs.append(pw); dbs.append(pb)
    assert np.allclose(dX, out["dX"], rtol=1e-11, atol=1e-15)
    assert np.allclose(np.concatenate(dWs), out["dW"], rtol=1e-11, atol=1e-15)
    assert np.allclose(np.concatenate(dbs), out["db"], rtol=1e-11, atol=1e-15)


# --- invariances the definitions imply -------------------------------------------

def test_row_stats_shift_invariance():
    """Softmax is unchanged when a constant is added to every logit of a row:
    lse moves by exactly that constant, logp and entropy do not move."""
    rng = np.random.default_rng(41)
    X, W, b, y = _rand_problem(rng, 12, 9, 70)
    tau = 0.8
    lse0, lp0, h0 = O.row_stats(X, W, b, y, tau)
    lse1, lp1, h1 = O.row_stats(X, W, b + 3.0 * tau, y, tau)
    np.testing.assert_allclose(lse1 - lse0, 3.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lp1, lp0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(h1, h0, rtol=0, atol=1e-12)


def test_temperature_folds_into_the_weights():
    """z = (X W^T + b) / tau: scaling W and b by 1/tau at tau = 1 gives the
    same row statistics and the same gradient coefficients' G (the 1/tau of
    dlogits included)."""
    rng = np.random.default_rng(42)
    X, W, b, y = _rand_problem(rng, 10, 7, 50)
    tau = 0.55
    a = O.row_stats(X, W, b, y, tau)
    c = O.row_stats(X, W / tau, b / tau, y, 1.0)
    for u, v in zip(a, c):
        np.testing.assert_allclose(u, v, rtol=1e-12, atol=1e-12)
    cn = rng.standard_normal(10)
    g_a = O.dlogits_rows(X, W, b, y, tau, a[0], cn, np.arange(10))
    g_c = O.dlogits_rows(X, W / tau, b / tau, y, 1.0, c[0], cn / tau, np.arange(10))
    np.testing.assert_allclose(g_a, g_c, rtol=1e-12, atol=1e-15)


def test_gmpo_common_shift_of_logp_and_old_changes_nothing():
    """The log ratio lr = logp - old is all GMPO (beta = 0) sees: shifting both
    by the same amount leaves loss, clip decisions and dL/dlogp unchanged."""
    rng = np.random.default_rng(43)
    B, T = 3, 9
    lp = rng.normal(-4, 1, B * T)
    old = lp + rng.normal(0, 0.4, B * T)
    m = (rng.random(B * T) > 0.2).astype(np.uint8)
    A = np.array([0.9, -1.3, 0.4])
    r0 = O.gmpo_loss(lp, old, None, A, m, B, T, 0.2, 0.3)
    r1 = O.gmpo_loss(lp + 1.75, old + 1.75, None, A, m, B, T, 0.2, 0.3)
    assert r1.loss == pytest.approx(r0.loss, rel=1e-13)
    assert np.array_equal(r0.clipped, r1.clipped)
    np.testing.assert_allclose(r1.c, r0.c, rtol=1e-12, atol=1e-18)


def test_batch_duplication_pins_the_reductions():
    """Stacking the batch on itself: GMPO's loss is a mean over sequences, so
    it stays and each token's dL/dlogp halves; GSPO-token's loss is a sum over
    tokens, so it doubles and dL/dlogp stays (readings R6 and R8)."""
    rng = np.random.default_rng(44)
    B, T = 3, 8
    lp = rng.normal(-4, 1, B * T)
    old = lp + rng.normal(0, 0.3, B * T)
    ref = lp + rng.normal(0, 0.1, B * T)
    m = (rng.random(B * T) > 0.2).astype(np.uint8)
    m[::T] = 1
    A = np.array([1.0, -0.6, 0.3])
    d = lambda x: np.concatenate([x, x])
    g1 = O.gmpo_loss(lp, old, ref, A, m, B, T, 0.2, 0.3, beta=0.04)
    g2 = O.gmpo_loss(d(lp), d(old), d(ref), d(A), d(m), 2 * B, T, 0.2, 0.3, beta=0.04)
    assert g2.loss == pytest.approx(g1.loss, rel=1e-13)
    np.testing.assert_allclose(g2.c, d(g1.c) / 2, rtol=1e-12, atol=1e-18)
    s1 = O.gspo_token_loss(lp, old, A, m, B, T, 0.05, 0.05)
    s2 = O.gspo_token_loss(d(lp), d(old), d(A), d(m), 2 * B, T, 0.05, 0.05)
    assert s2.loss == pytest.approx(2 * s1.loss, rel=1e-13)
    np.testing.assert_allclose(s2.c, d(s1.c), rtol=1e-12, atol=1e-18)
