"""fp64 CPU oracle for the fused LM-head RL policy loss.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module.  It shares no
code with the CUDA library (``lm_head_log_tma_gb300``) and imports nothing
from it.

It is the plain definition of what the fused path computes, written in fp64
with numpy.  The one library primitive it leans on is a matrix product
(``X @ W.T`` and friends); everything else is the textbook formula, evaluated
row by row (rows are independent by definition, so rows are taken in groups
only to bound memory and to spread them over host threads).

Notation: sequences i = 0..B-1, tokens n = i*T + t, N = B*T; m_n in {0,1} is
the completion mask, n_i = sum_t m_n, A_i the per-sequence advantage.
  l = X W^T + b,  z = l / tau,  lse_n = logsumexp(z_n),
  logp_n = z_{n,y_n} - lse_n,   H_n = lse_n - sum_v p_nv z_nv,  p = softmax(z).

Sources (page, section):
  * "Add GMPO to fused linear GRPO loss" (Liger-Kernel PR #1320), Summary and
    Details: one-sided, advantage-dependent clipping of each token's log ratio
    in log space to [-eps_low, +eps_high]; per-sequence geometric mean
    exp(masked_mean(clipped log ratio)); per-sample reduction; K3 KL; clipping
    metric; sequence-level importance sampling rejected.
  * "support top_entropy_quantile in fused linear GRPO loss" (Liger-Kernel PR
    #1558), Summary and Details: entropy H = log_z - sum_exp_z / sum_exp from
    the streamed accumulators; threshold = quantile(active entropies, 1 - q)
    over the whole batch; mask multiplies the policy term after the loss-type
    branch and before the KL penalty; q = 1 is a no-op; q outside [0,1] raises.
  * Tinker "GSPO": sequence ratio s = exp(mean over the masked tokens of
    log p - log q); token ratio carries s's value and its own log-prob's
    gradient; objective -sum_t min(s_t A_t, clip(s_t, lo, hi) A_t); default
    clip range [1 - 3e-4, 1 + 4e-4]; diagnostics loss:sum,
    gspo_sequence_log_ratio:mean, gspo_clipped_fraction:mean.

Readings taken where the pages are silent (each also listed in the design doc):
  R1 GMPO clip metric counts strict excursions (lr > eps_high for A>0,
     lr < -eps_low for A<0); at lr == bound the token is unclipped and passes
     gradient 1 (inclusive clamp gradient).
  R2 A_i == 0: never clipped (its policy term is zero anyway).
  R3 quantile = linear interpolation between order statistics (torch.quantile's
     default), position (1-q)(n_act-1).
  R4 entropy mask keeps H_n >= threshold (ties kept); with q = 1 every active
     token is kept.
  R5 no active token -> empty mask, threshold NaN.
  R6 GMPO reduction: per-sequence masked mean, then mean over the B sequences;
     a sequence with no active token contributes 0 and still counts in B.
  R7 the entropy mask scales the per-token policy term -A_i r_i (so the
     sequence term becomes -A_i r_i mean_t(e_t)); it does not enter r_i.
  R8 GSPO reduction is a sum over tokens; advantages are A_i on completion
     tokens and 0 on the prompt.
  R9 the Tinker page calls the sampler log-probs "ref_logprobs"; here they are
     old_logp.  ref_logp is the KL reference model's log-probs.
  R10 entropy is taken on temperature-scaled logits.
  R11 GSPO's clip bounds are applied as the fp32 values of 1-eps_low, 1+eps_high;
     GMPO's eps are compared as their fp32 values widened to fp64.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

GMPO = 0
GSPO_TOKEN = 1

ROW_BLOCK = 64


def as_f64(x):
    """Widen an array (numpy, or a CPU torch tensor of any float dtype) to fp64 exactly."""
    if x is None:
        return None
    if hasattr(x, "detach"):           # torch tensor: widen through torch (bf16 has no numpy dtype)
        import torch
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def as_i64(x):
    if hasattr(x, "detach"):
        return x.detach().to("cpu").numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


def f32(x: float) -> float:
    """The fp32 value of x, widened back to fp64."""
    return float(np.float32(x))


# ---------------------------------------------------------------------------
# Per-row quantities: log-softmax, target log-prob and entropy.
# "support top_entropy_quantile ...", Details (entropy from the streamed
# log-sum-exp accumulators; the plain two-pass definition is used here).
# ---------------------------------------------------------------------------

def logits_rows(X, W, b, tau, rows):
    """z for the given rows: (X[rows] W^T + b) / tau, fp64 [len(rows), V]."""
    z = X[rows] @ W.T
    if b is not None:
        z = z + b[None, :]
    return z / tau


def _stats_block(z, y):
    zmax = z.max(axis=1)
    s = np.exp(z - zmax[:, None]).sum(axis=1)
    lse = zmax + np.log(s)
    p = np.exp(z - lse[:, None])
    ent = lse - (p * z).sum(axis=1)
    logp = z[np.arange(z.shape[0]), y] - lse
    return lse, logp, ent


def row_stats(X, W, b, targets, tau, rows=None, threads=None):
    """Returns (lse, logp, entropy) in fp64 for ``rows`` (default: all rows)."""
    X = as_f64(X); W = as_f64(W); b = as_f64(b); y = as_i64(targets)
    if rows is None:
        rows = np.arange(X.shape[0])
    rows = np.asarray(rows, dtype=np.int64)
    lse = np.empty(rows.size); logp = np.empty(rows.size); ent = np.empty(rows.size)

    def work(k0):
        r = rows[k0:k0 + ROW_BLOCK]
        z = logits_rows(X, W, b, tau, r)
        lse[k0:k0 + r.size], logp[k0:k0 + r.size], ent[k0:k0 + r.size] = _stats_block(z, y[r])

    starts = range(0, rows.size, ROW_BLOCK)
    nt = threads or os.cpu_count() or 1
    if nt == 1 or rows.size <= ROW_BLOCK:
        for k0 in starts:
            work(k0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(work, starts))
    return lse, logp, ent


def entropy_direct(z):
    """-sum_v p log p for one block of logits (used to pin the lse - E[z] form)."""
    zmax = z.max(axis=1, keepdims=True)
    lp = z - zmax - np.log(np.exp(z - zmax).sum(axis=1, keepdims=True))
    return -(np.exp(lp) * lp).sum(axis=1)


# ---------------------------------------------------------------------------
# Batch-global entropy quantile and mask.
# "support top_entropy_quantile ...", Details: threshold = quantile(active
# entropies, 1 - q) over the whole batch; readings R3, R4, R5.
# ---------------------------------------------------------------------------

def entropy_threshold(entropy, mask, q):
    """Returns (thr, e): thr fp64 (NaN if no active token), e uint8 [N]."""
    if not (0.0 <= q <= 1.0):
        raise ValueError("top_entropy_quantile must lie in [0, 1]")
    H = np.asarray(entropy, dtype=np.float64)
    m = np.asarray(mask) != 0
    act = np.sort(H[m])
    n_act = act.size
    if n_act == 0:
        return float("nan"), np.zeros(H.shape, np.uint8)
    pos = (1.0 - q) * (n_act - 1)
    lo = int(math.floor(pos))
    hi = min(lo + 1, n_act - 1)
    frac = pos - lo
    thr = act[lo] + frac * (act[hi] - act[lo])
    e = (m & (H >= thr)).astype(np.uint8)
    return float(thr), e


# ---------------------------------------------------------------------------
# Loss stage.  Metrics vector layout (8 entries):
#   0 clip fraction, 1 clip count, 2 KL mean over active tokens,
#   3 n_active, 4 entropy threshold, 5 tokens kept by the entropy mask,
#   6 mean over sequences of the sequence log ratio, 7 mean sequence ratio.
# ---------------------------------------------------------------------------

@dataclass
class LossResult:
    loss: float
    metrics: np.ndarray        # fp64 [8]
    c: np.ndarray              # dL/dlogp_n, fp64 [N]
    clipped: np.ndarray        # GMPO: per-token clip flag; GSPO: per-sequence flag
    emask: np.ndarray          # entropy-mask bits actually used (uint8 [N])
    seq_log_ratio: np.ndarray  # [B]
    kl: np.ndarray | None = None


def gmpo_loss(logp, old_logp, ref_logp, adv, mask, B, T, eps_low, eps_high, beta=0.0,
              entropy=None, q=1.0, emask_override=None, clip_override=None):
    """GMPO objective ("Add GMPO to fused linear GRPO loss", Summary/Details).

    Per token:  lr = logp - old.  A_i > 0: clr = min(lr, eps_high);  A_i < 0:
    clr = max(lr, -eps_low);  A_i = 0: clr = lr.  Per sequence:
    r_i = exp(sum_t m clr / n_i), ebar_i = sum_t m e / n_i,
    l_i = -A_i r_i ebar_i + beta sum_t m kl / n_i  with  kl = e^(ref-logp) - (ref-logp) - 1.
    L = mean_i l_i.  Returns the loss, metrics, and c_n = dL/dlogp_n.

    ``emask_override`` / ``clip_override`` let a caller impose decisions on
    tokens that sit on a knife edge (used only by parity tests, which first
    check that every overridden token is within the stated distance of its
    bound or threshold).
    """
    lp = np.asarray(logp, np.float64).reshape(B, T)
    old = np.asarray(old_logp, np.float64).reshape(B, T)
    m = (np.asarray(mask).reshape(B, T) != 0)
    A = np.asarray(adv, np.float64).reshape(B)
    el, eh = f32(eps_low), f32(eps_high)
    if eps_low < 0 or eps_high < 0:
        raise ValueError("eps must be >= 0")

    thr = float("nan")
    if q < 1.0:
        if entropy is None:
            raise ValueError("entropy needed when q < 1")
        thr, e = entropy_threshold(np.asarray(entropy, np.float64).reshape(-1), m.reshape(-1), q)
    elif not (0.0 <= q <= 1.0):
        raise ValueError("top_entropy_quantile must lie in [0, 1]")
    else:
        e = m.reshape(-1).astype(np.uint8)
    if emask_override is not None:
        e = np.asarray(emask_override, np.uint8).reshape(-1)
    e2 = e.reshape(B, T).astype(np.float64)

    lr = lp - old
    Ab = A[:, None]
    pos, neg = Ab > 0, Ab < 0
    clipped = (pos & (lr > eh)) | (neg & (lr < -el))
    if clip_override is not None:
        clipped = np.asarray(clip_override, bool).reshape(B, T)
    clr = np.where(clipped, np.where(pos, eh, -el), lr)
    clipped = clipped & m

    n_i = m.sum(axis=1).astype(np.float64)
    has = n_i > 0
    safe_n = np.where(has, n_i, 1.0)
    mean_clr = np.where(has, (m * clr).sum(axis=1) / safe_n, 0.0)
    r = np.where(has, np.exp(mean_clr), 0.0)
    ebar = np.where(has, (m * e2).sum(axis=1) / safe_n, 0.0)

    kl = None
    kl_term = np.zeros(B)
    if beta != 0.0:
        ref = np.asarray(ref_logp, np.float64).reshape(B, T)
        d = ref - lp
        kl = np.exp(d) - d - 1.0
        kl_term = np.where(has, (m * kl).sum(axis=1) / safe_n, 0.0)
    l_i = np.where(has, -A * r * ebar + beta * kl_term, 0.0)
    loss = l_i.sum() / B

    g = (~clipped).astype(np.float64)
    c = (-Ab * (r * ebar)[:, None] * g) * m / (B * safe_n[:, None])
    if beta != 0.0:
        c = c + beta * (1.0 - np.exp(d)) * m / (B * safe_n[:, None])
    c = np.where(has[:, None], c, 0.0)

    n_act = float(m.sum())
    metrics = np.zeros(8)
    metrics[1] = float(clipped.sum())
    metrics[0] = metrics[1] / n_act if n_act > 0 else 0.0
    metrics[2] = float((m * kl).sum() / n_act) if (beta != 0.0 and n_act > 0) else 0.0
    metrics[3] = n_act
    metrics[4] = thr
    metrics[5] = float((e2 * m).sum())
    nh = has.sum()
    metrics[6] = float(mean_clr[has].sum() / nh) if nh else 0.0
    metrics[7] = float(r[has].sum() / nh) if nh else 0.0
    return LossResult(float(loss), metrics, c.reshape(-1), clipped.reshape(-1),
                      e.reshape(-1), mean_clr, None if kl is None else kl.reshape(-1))


def gspo_token_loss(logp, old_logp, adv, mask, B, T, eps_low=3e-4, eps_high=4e-4,
                    clip_override=None, per_token_adv=False):
    """GSPO-token objective (Tinker "GSPO").

    s_i = exp(sum_t m (logp - old) / n_i) (taken on detached log-probs); each
    token's ratio s_t has s_i's value and the gradient of its own logp, so
    ds_t/dlogp_t = s_i.  Advantages: per sequence ([B]) gives A_n = A_i m_n
    (reading R8); with ``per_token_adv`` ([N]) A_n is given directly (the
    page's per-token advantages input).  obj_n = min(s A_n, clip(s, lo, hi) A_n),
    L = -sum_n obj_n.  c_n = -A_n s_i g_n, where g_n = 0 exactly when the
    clipped branch is the strictly smaller one with a flat clamp:
    (A_n > 0 and s_i > hi) or (A_n < 0 and s_i < lo).  At s_i == lo or hi the
    clamp is inclusive and the minimum ties, so the gradient passes in full.
    """
    lp = np.asarray(logp, np.float64).reshape(B, T)
    old = np.asarray(old_logp, np.float64).reshape(B, T)
    m = (np.asarray(mask).reshape(B, T) != 0)
    A = np.asarray(adv, np.float64)
    lo, hi = f32(1.0 - eps_low), f32(1.0 + eps_high)
    n_i = m.sum(axis=1).astype(np.float64)
    if np.any(n_i == 0):
        raise ValueError("sequence_ratio_mask must mark at least one token per sequence")
    slr = (m * (lp - old)).sum(axis=1) / n_i
    s = np.exp(slr)
    if per_token_adv:
        An = A.reshape(B, T)
    else:
        An = A.reshape(B)[:, None] * m
    sc = np.clip(s, lo, hi)
    obj = np.minimum(s[:, None] * An, sc[:, None] * An)
    loss = -obj.sum()
    out = (s < lo) | (s > hi)
    if clip_override is not None:
        out = np.asarray(clip_override, bool).reshape(B)
        flat_hi, flat_lo = out & (s >= 1.0), out & (s < 1.0)
    else:
        flat_hi, flat_lo = s > hi, s < lo
    gate = ~((An > 0) & flat_hi[:, None] | (An < 0) & flat_lo[:, None])
    c = -An * s[:, None] * gate
    metrics = np.zeros(8)
    metrics[1] = float(out.sum())
    metrics[0] = metrics[1] / B
    metrics[3] = float(m.sum())
    metrics[4] = float("nan")
    metrics[5] = float(m.sum())
    metrics[6] = float(slr.mean())
    metrics[7] = float(s.mean())
    return LossResult(float(loss), metrics, c.reshape(-1), out, m.reshape(-1).astype(np.uint8), slr)


# ---------------------------------------------------------------------------
# Gradients through the LM head.  With c_n = dL/dlogp_n and
# dlogp_n/dl_nv = (delta_{v,y_n} - p_nv) / tau:
#   G = dL/dl = c (onehot - p) / tau,   dX = G W,   dW = G^T X,   db = sum_n G_n.
# ---------------------------------------------------------------------------

def dlogits_rows(X, W, b, targets, tau, lse, c, rows):
    """G for the given rows, fp64 [len(rows), V]."""
    z = logits_rows(X, W, b, tau, rows)
    p = np.exp(z - lse[rows][:, None])
    G = -p
    G[np.arange(len(rows)), targets[rows]] += 1.0
    return G * (c[rows] / tau)[:, None]


def grads(X, W, b, targets, tau, lse, c, dx_rows=None, dw_rows=None, want_db=True,
          threads=None):
    """dX for ``dx_rows`` (default all), dW for vocab rows ``dw_rows`` (default all)
    and db (full) if ``want_db``.  lse and c are fp64 [N]."""
    X = as_f64(X); W = as_f64(W); b = as_f64(b); y = as_i64(targets)
    N, V = X.shape[0], W.shape[0]
    lse = np.asarray(lse, np.float64); c = np.asarray(c, np.float64)
    dx_rows = np.arange(N) if dx_rows is None else np.asarray(dx_rows, np.int64)
    all_v = dw_rows is None
    dw_rows = np.arange(V) if all_v else np.asarray(dw_rows, np.int64)

    dX = np.zeros((dx_rows.size, X.shape[1]))
    for k0 in range(0, dx_rows.size, ROW_BLOCK):
        r = dx_rows[k0:k0 + ROW_BLOCK]
        dX[k0:k0 + r.size] = dlogits_rows(X, W, b, y, tau, lse, c, r) @ W

    # dW rows and db need every token's G restricted to the chosen vocab rows.
    dW = np.zeros((dw_rows.size, X.shape[1]))
    db = np.zeros(V) if want_db else None
    nz = np.nonzero(c)[0]
    nt = threads or os.cpu_count() or 1
    chunks = [nz[k:k + ROW_BLOCK] for k in range(0, nz.size, ROW_BLOCK)]

    def work(r):
        zr = X[r] @ W[dw_rows].T
        if b is not None:
            zr = zr + b[dw_rows][None, :]
        zr = zr / tau
        G = -np.exp(zr - lse[r][:, None])
        hit = (y[r][:, None] == dw_rows[None, :])
        G = (G + hit) * (c[r] / tau)[:, None]
        part_db = None
        if want_db:
            if all_v:
                part_db = G.sum(axis=0)
            else:
                Gf = dlogits_rows(X, W, b, y, tau, lse, c, r)
                part_db = Gf.sum(axis=0)
        return G.T @ X[r], part_db

    if nt == 1 or len(chunks) <= 1:
        results = [work(r) for r in chunks]
    else:
        with ThreadPoolExecutor(nt) as ex:
            results = list(ex.map(work, chunks))
    for pdw, pdb in results:
        dW += pdw
        if want_db:
            db += pdb
    return dX, dW, db


# ---------------------------------------------------------------------------
# Vocabulary shards.  The streamed accumulators of "support
# top_entropy_quantile ...", Details (the log-sum-exp accumulator and a second
# online accumulator for the entropy) combine over disjoint vocabulary
# ranges: for a shard with reference m, s = sum e^(z-m), w = sum e^(z-m)(z-m),
# and with M = max_k m_k over the shards,
#   S = sum_k e^(m_k-M) s_k,   Wt = sum_k e^(m_k-M) (w_k + (m_k-M) s_k),
#   lse = M + log S,           H = lse - E_p[z] = log S - Wt / S.
# The gradient terms restrict to the shard's columns: G_shard = G[:, shard],
# dX = sum over shards of G_shard W_shard, dW and db are the shard's rows.
# ---------------------------------------------------------------------------

def shard_state(X, W_shard, b_shard, targets, tau, v_begin):
    """fp64 per-row state of the vocabulary rows [v_begin, v_begin + len(W_shard))."""
    X = as_f64(X); Ws = as_f64(W_shard); bs = as_f64(b_shard); y = as_i64(targets)
    N, Vs = X.shape[0], Ws.shape[0]
    m = np.empty(N); s = np.empty(N); w = np.empty(N); zy = np.full(N, np.nan)
    for k0 in range(0, N, ROW_BLOCK):
        r = np.arange(k0, min(N, k0 + ROW_BLOCK))
        z = logits_rows(X, Ws, bs, tau, r)
        mm = z.max(axis=1)
        e = np.exp(z - mm[:, None])
        m[r] = mm
        s[r] = e.sum(axis=1)
        w[r] = (e * (z - mm[:, None])).sum(axis=1)
        yl = y[r] - v_begin
        inside = (yl >= 0) & (yl < Vs)
        zy[r[inside]] = z[np.nonzero(inside)[0], yl[inside]]
    return dict(m=m, s=s, w=w, zy=zy)


def merge_states(states, targets=None, V=None):
    """(lse, logp, entropy) fp64 from the states of disjoint shards.  logp is
    NaN where no shard holds the target (or the target lies outside [0, V))."""
    M = np.max([st["m"] for st in states], axis=0)
    S = np.zeros_like(M); Wt = np.zeros_like(M)
    zy = np.full_like(M, np.nan)
    for st in states:
        f = np.exp(st["m"] - M)
        S += f * st["s"]
        Wt += f * (st["w"] + (st["m"] - M) * st["s"])
        have = ~np.isnan(st["zy"])
        zy[have] = st["zy"][have]
    lse = M + np.log(S)
    ent = np.log(S) - Wt / S
    logp = zy - lse
    if targets is not None and V is not None:
        y = as_i64(targets)
        logp[(y < 0) | (y >= V)] = np.nan
    return lse, logp, ent


def shard_grads(X, W_shard, b_shard, targets, tau, v_begin, lse, c):
    """This shard's part of dX, its dW rows and its db rows (fp64), from the
    whole vocabulary's lse and c = dL/dlogp."""
    X = as_f64(X); Ws = as_f64(W_shard); bs = as_f64(b_shard); y = as_i64(targets)
    N, Vs = X.shape[0], Ws.shape[0]
    lse = np.asarray(lse, np.float64); c = np.asarray(c, np.float64)
    dX = np.zeros((N, X.shape[1])); dW = np.zeros((Vs, X.shape[1]))
    db = np.zeros(Vs) if bs is not None else None
    for k0 in range(0, N, ROW_BLOCK):
        r = np.arange(k0, min(N, k0 + ROW_BLOCK))
        z = logits_rows(X, Ws, bs, tau, r)
        G = -np.exp(z - lse[r][:, None])
        yl = y[r] - v_begin
        inside = np.nonzero((yl >= 0) & (yl < Vs))[0]
        G[inside, yl[inside]] += 1.0
        G *= (c[r] / tau)[:, None]
        dX[r] = G @ Ws
        dW += G.T @ X[r]
        if db is not None:
            db += G.sum(axis=0)
    return dX, dW, db


# ---------------------------------------------------------------------------
# Whole pipeline.
# ---------------------------------------------------------------------------

@dataclass
class Problem:
    B: int
    T: int
    loss_type: int = GMPO
    eps_low: float = 0.4
    eps_high: float = 0.4
    beta: float = 0.0
    temperature: float = 1.0
    top_entropy_quantile: float = 1.0
    is_level_sequence: bool = False
    per_token_adv: bool = False


def loss_stage(prob: Problem, logp, entropy, old_logp, ref_logp, adv, mask,
               emask_override=None, clip_override=None) -> LossResult:
    if prob.loss_type == GMPO:
        if prob.is_level_sequence:
            raise ValueError("GMPO clips at token level; sequence-level importance sampling is rejected")
        return gmpo_loss(logp, old_logp, ref_logp, adv, mask, prob.B, prob.T, prob.eps_low,
                         prob.eps_high, prob.beta, entropy, prob.top_entropy_quantile,
                         emask_override, clip_override)
    if prob.loss_type == GSPO_TOKEN:
        return gspo_token_loss(logp, old_logp, adv, mask, prob.B, prob.T, prob.eps_low,
                               prob.eps_high, clip_override, prob.per_token_adv)
    if prob.per_token_adv:
        raise ValueError("per-token advantages are defined for GSPO-token only")
    raise ValueError("unknown loss type")


def fwd_bwd(prob: Problem, X, W, b, targets, old_logp, ref_logp, adv, mask,
            dx_rows=None, dw_rows=None, threads=None):
    """Full oracle: per-row stats, loss, and gradients.  Returns a dict."""
    lse, logp, ent = row_stats(X, W, b, targets, prob.temperature, threads=threads)
    res = loss_stage(prob, logp, ent, as_f64(old_logp).reshape(-1),
                     None if ref_logp is None else as_f64(ref_logp).reshape(-1),
                     as_f64(adv), as_i64(mask))
    dX, dW, db = grads(X, W, b, targets, prob.temperature, lse, res.c, dx_rows, dw_rows,
                       want_db=b is not None, threads=threads)
    return dict(lse=lse, logp=logp, entropy=ent, loss=res.loss, metrics=res.metrics,
                c=res.c, clipped=res.clipped, emask=res.emask, dX=dX, dW=dW, db=db, res=res)
