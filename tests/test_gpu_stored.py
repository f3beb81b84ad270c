"""The stored-probability backward against the recompute and the oracle.

With bf16 operands and no bias the forward also writes every logit's
unnormalised probability 2^t (bf16) for the row tiles that fit the chunk
buffer, and dX, dW of those rows come from it without a second logits GEMM:
G = (c/tau)(onehot(y) - p) with p = 2^(t - lse2) ("Add GMPO to fused linear
GRPO loss", Details: the input and weight gradients are sums over tokens of
c_n times the softmax terms).  Rows outside the stored tiles, and rows whose
log-sum-exp lies outside the stored range, are recomputed.  Both paths must
pass the oracle; they differ only in where bf16 rounding enters.
"""
import numpy as np
import pytest
import torch

from lm_head_log_tma_gb300.workloads import GSPO_TOKEN, Workload, make_inputs
from parity import GRAD_COS, GRAD_RELL2, Case, check_grads, check_loss_and_metrics, check_rows, cosine, \
    reconcile_loss, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_log_tma_gb300 import rlloss
    return rlloss


SPECS = [
    Workload("stored_gmpo", B=3, T=150, H=192, V=1000, dtype="bf16", prompt_len=20, seed=201),
    Workload("stored_entropy_q0.2_tau0.7", B=5, T=100, H=128, V=1300, dtype="bf16", temperature=0.7,
             top_entropy_quantile=0.2, prompt_len=10, seed=202),
    Workload("stored_gspo", B=6, T=97, H=64, V=600, dtype="bf16", loss_type=GSPO_TOKEN, eps_low=3e-4,
             eps_high=4e-4, prompt_len=8, old_noise_std=0.02, seed=203),
    Workload("stored_k3kl_asym", B=4, T=130, H=256, V=777, dtype="bf16", eps_low=0.2, eps_high=0.3, beta=0.04,
             prompt_len=(5, 40), adv_kind="pm1zero", ref_noise_std=0.1, seed=204),
    Workload("stored_wide_h_2048", B=2, T=300, H=2048, V=3000, dtype="bf16", prompt_len=10, seed=205),
    Workload("stored_many_short", B=300, T=3, H=64, V=500, dtype="bf16", prompt_len=1, seed=206),
    # with a bias, db comes out of dW's GEMM as one more column (k2 in column H of
    # the scaled X rows): inside the last tile's second half (H=256), in a
    # widened last half (H=448, a multiple of the 448-column tile), inside the
    # last tile's first half (H=1040, H=512)
    Workload("stored_bias_k3kl", B=4, T=130, H=256, V=777, dtype="bf16", has_bias=True, bias_std=0.3,
             eps_low=0.2, eps_high=0.3, beta=0.04, prompt_len=(5, 40), adv_kind="pm1zero", ref_noise_std=0.1,
             seed=207),
    Workload("stored_bias_h448", B=2, T=200, H=448, V=1500, dtype="bf16", has_bias=True, bias_std=0.2,
             prompt_len=16, seed=208),
    Workload("stored_bias_h1040", B=3, T=100, H=1040, V=1500, dtype="bf16", has_bias=True, bias_std=0.2,
             temperature=0.7, prompt_len=5, seed=209),
    Workload("stored_bias_h512", B=2, T=160, H=512, V=1100, dtype="bf16", has_bias=True, bias_std=0.2,
             prompt_len=12, seed=210),
]


def _check(R, case, **kw):
    out = case.run_gpu(R, **kw)
    assert out["status"] == 0, hex(out["status"])
    if out.get("logp") is not None:   # per-token outputs requested
        check_rows(out, case)
    res = reconcile_loss(out, case)
    check_loss_and_metrics(out, case, res)
    check_grads(out, case, res)
    return out, res


def _taken_rows(c, block=128):
    """Rows the stored-probability dX, dW run over: the 128-row blocks (of the
    forward's 256-row tiles, so 128-aligned in row order) holding a row with
    c_n != 0, taken whole."""
    nz = np.asarray(c) != 0
    pad = (-len(nz)) % block
    nz = np.concatenate([nz, np.zeros(pad, bool)])
    return int(nz.reshape(-1, block).any(axis=1).sum()) * block


def _close(a, b):
    for k in ("dX", "dW", "db"):
        if a.get(k) is None:
            continue
        x, y = a[k].double().cpu().numpy(), b[k].double().cpu().numpy()
        assert rel_l2(x, y) <= GRAD_RELL2 and cosine(x, y) >= GRAD_COS, k


@pytest.mark.parametrize("spec", SPECS, ids=[s.name for s in SPECS])
def test_stored_backward_matches_recompute_and_oracle(R, spec):
    """Default (stored) and FLAG_RECOMPUTE both pass the oracle; the forward,
    loss and metrics are bit-identical; every kept row went through the stored
    path when all row tiles fit the buffer."""
    case = Case(spec)
    a, res = _check(R, case, per_token=False)
    b, _ = _check(R, case, per_token=False, flags=R.FLAG_RECOMPUTE)
    for k in ("loss", "metrics"):
        assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), k
    kept = int((res.c != 0).sum())
    assert R.rlloss_get_stored_rows(a["workspace"]) == kept
    assert R.rlloss_get_stored_positions(a["workspace"]) == _taken_rows(res.c)
    assert R.rlloss_get_backward_rows(a["workspace"]) == 0
    assert R.rlloss_get_stored_rows(b["workspace"]) == 0
    assert R.rlloss_get_backward_rows(b["workspace"]) == kept
    assert torch.count_nonzero(a["dX"][torch.from_numpy(res.c == 0).cuda()]) == 0
    _close(a, b)


def test_stored_with_per_token_outputs_runs_every_tile(R):
    """Per-token outputs run the forward over every row tile (no tile list):
    the stored rows are then every tile's, and the result still matches."""
    case = Case(SPECS[0])
    a, res = _check(R, case, per_token=True)
    assert R.rlloss_get_stored_rows(a["workspace"]) == int((res.c != 0).sum())
    assert R.rlloss_get_stored_positions(a["workspace"]) == _taken_rows(res.c)


def test_stored_and_recomputed_rows_in_one_call(R):
    """A chunk buffer of 256 rows holds one of the two forward row tiles: the
    first tile's rows come from the stored probabilities, the second's are
    recomputed, and the sum passes the oracle and matches FLAG_RECOMPUTE."""
    spec = SPECS[0]
    case = Case(spec)
    a, res = _check(R, case, per_token=False, chunk_rows=256)
    c = res.c != 0
    assert R.rlloss_get_stored_rows(a["workspace"]) == int(c[:256].sum())
    assert R.rlloss_get_backward_rows(a["workspace"]) == int(c[256:].sum()) > 0
    b, _ = _check(R, case, per_token=False, chunk_rows=256, flags=R.FLAG_RECOMPUTE)
    _close(a, b)


def test_rows_outside_the_stored_range_are_recomputed(R):
    """Rows whose log-sum-exp is far above the stored range (X rows scaled by
    600: logits of hundreds of nats) go to the recompute; the others stay on
    the stored path, and every gradient passes the oracle."""
    spec = SPECS[0]
    inp = make_inputs(spec)
    big = np.array([21, 40, 77, 260, 301, 449])
    inp.X[torch.from_numpy(big)] *= 600
    case = Case(spec, inp)
    assert np.all(case.lse[big] * 1.4426950408889634 > 96)
    assert np.all(case.lse[np.setdiff1d(np.arange(spec.N), big)] * 1.4426950408889634 < 96)
    a, res = _check(R, case, per_token=False)
    kept_big = int((res.c[big] != 0).sum())
    assert kept_big > 0
    assert R.rlloss_get_backward_rows(a["workspace"]) == kept_big
    rows = torch.from_numpy(big[res.c[big] != 0]).cuda()
    assert torch.count_nonzero(a["dX"][rows]) > 0


BLOCKS = [
    # prompt of 200 rows: in the first 256-row tile the first 128-row block has
    # no kept row (left out), the second has some; three blocks taken, so the
    # last dX tile is half tail
    Workload("blocks_prompt200", B=1, T=512, H=192, V=900, dtype="bf16", prompt_len=200, seed=221),
    # whole sequences clipped (GSPO, tight bounds): their blocks are left out
    Workload("blocks_gspo_clipped", B=4, T=256, H=128, V=700, dtype="bf16", loss_type=GSPO_TOKEN,
             eps_low=3e-4, eps_high=4e-4, prompt_len=130, old_noise_std=0.02, seed=222),
    # with a bias (db through dW's GEMM): one taken block per sequence, three in all
    Workload("blocks_bias_prompt330", B=3, T=384, H=256, V=800, dtype="bf16", has_bias=True, bias_std=0.2,
             prompt_len=330, seed=223),
]


@pytest.mark.parametrize("spec", BLOCKS, ids=[s.name for s in BLOCKS])
def test_blocks_without_kept_rows_are_left_out(R, spec):
    """The stored-probability dX and dW skip 128-row blocks whose rows all have
    c_n = 0 and run a taken block whole, its other rows with zero factors
    (positions past the last taken block read the first one against zero X
    rows); the result passes the oracle and matches the recompute, and the
    rows run over are exactly the taken blocks'."""
    case = Case(spec)
    a, res = _check(R, case, per_token=False)
    b, _ = _check(R, case, per_token=False, flags=R.FLAG_RECOMPUTE)
    taken = _taken_rows(res.c)
    assert taken < spec.N
    assert R.rlloss_get_stored_positions(a["workspace"]) == taken
    assert R.rlloss_get_stored_rows(a["workspace"]) == int((res.c != 0).sum())
    assert torch.count_nonzero(a["dX"][torch.from_numpy(res.c == 0).cuda()]) == 0
    _close(a, b)


def test_stored_calls_are_bit_identical(R):
    """Two calls give the same bits: dX rows get two addends onto zero (one
    per vocabulary half), dW one store."""
    case = Case(SPECS[1])
    a = case.run_gpu(R, per_token=False)
    b = case.run_gpu(R, per_token=False)
    for k in ("loss", "metrics", "dX", "dW"):
        assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), k


GROUPED = [
    Workload("grouped_gmpo_k3kl_bias", B=6, T=256, H=128, V=1000, dtype="bf16", has_bias=True, bias_std=0.2,
             eps_low=0.2, eps_high=0.3, beta=0.04, prompt_len=(5, 40), adv_kind="pm1zero", ref_noise_std=0.1,
             seed=211),
    Workload("grouped_gspo", B=5, T=512, H=64, V=700, dtype="bf16", loss_type=GSPO_TOKEN, eps_low=3e-4,
             eps_high=4e-4, prompt_len=16, old_noise_std=0.02, seed=212),
]


@pytest.mark.parametrize("spec", GROUPED, ids=[s.name for s in GROUPED])
def test_sequence_groups(R, spec):
    """Without an entropy mask the batch runs in groups of whole sequences that
    each fit the stored-probability buffer (a buffer of two sequences here:
    groups of 2, 2 and 1 or 2): per group the forward with stores, the loss
    stage's additive sums (with the whole batch's B: GMPO's mean over
    sequences, GSPO's clipped fraction) and the stored backward; dW and db add
    up over the groups.  Against the oracle, the one-pass call, and the
    recompute; per-token outputs through the groups; repeated calls bit-identical."""
    case = Case(spec)
    chunk = 2 * spec.T
    a, res = _check(R, case, per_token=False, chunk_rows=chunk)
    tiles = R.rlloss_get_forward_tiles(a["workspace"])
    assert tiles == spec.N // 256
    assert R.rlloss_get_stored_rows(a["workspace"]) == int((res.c != 0).sum())
    assert R.rlloss_get_stored_positions(a["workspace"]) == _taken_rows(res.c)   # groups start 128-aligned
    assert R.rlloss_get_backward_rows(a["workspace"]) == 0
    b, _ = _check(R, case, per_token=False)   # one pass: the whole batch fits the default buffer
    c, _ = _check(R, case, per_token=False, chunk_rows=chunk, flags=R.FLAG_RECOMPUTE)
    for o in (b, c):
        assert abs(a["loss"].item() - o["loss"].item()) <= 1e-6 * abs(o["loss"].item()) + 1e-9
        assert torch.allclose(a["metrics"], o["metrics"], rtol=1e-6, atol=1e-7, equal_nan=True)
        _close(a, o)
    d, _ = _check(R, case, per_token=True, chunk_rows=chunk)
    a2 = case.run_gpu(R, per_token=False, chunk_rows=chunk)
    for k in ("loss", "metrics", "dX", "dW") + (("db",) if spec.has_bias else ()):
        assert torch.equal(a[k].view(torch.int32), a2[k].view(torch.int32)), k
