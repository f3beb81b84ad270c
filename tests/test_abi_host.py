"""Host-side tests of the C ABI: the library loads, exports every function the
header declares, and rejects invalid requests synchronously (no GPU needed:
validation happens before any CUDA call)."""
import ctypes
import json
import math
import os

import numpy as np
import pytest

from lm_head_log_tma_gb300 import build as B

if not os.path.exists(B.LIB):
    B.build()
from lm_head_log_tma_gb300 import rlloss as R  # noqa: E402


def test_library_exports_every_declared_function():
    names = R.declared_functions()
    assert "rlloss_fwd_bwd" in names and "rlloss_loss_from_logp" in names
    lib = ctypes.CDLL(R.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    for code in (R.OK, R.EINVAL, R.EUNSUPPORTED, R.EWORKSPACE, R.ECUDA, R.DEV_ETIMEOUT):
        assert R.status_str(code) != "unknown status"


def _cfg(**kw):
    base = dict(B=2, T=16, H=64, V=512, dtype=R.BF16)
    base.update(kw)
    return R.make_cfg(**base)


def test_workspace_bytes_positive_and_zero_for_invalid():
    assert R.rlloss_workspace_bytes(_cfg()) > 0
    assert R.rlloss_workspace_bytes(_cfg(top_entropy_quantile=1.5)) == 0
    assert R.rlloss_workspace_bytes(_cfg(temperature=0.0)) == 0
    assert R.rlloss_loss_workspace_bytes(_cfg(H=0, V=0)) > 0


def test_workspace_grows_with_fp32_split_and_bias():
    # against the recompute backward, which the fp32 and bias forms use too
    a = R.rlloss_workspace_bytes(_cfg(flags=R.FLAG_RECOMPUTE))
    assert R.rlloss_workspace_bytes(_cfg(dtype=R.FP32)) > a
    assert R.rlloss_workspace_bytes(_cfg(has_bias=True)) > a


def test_stored_probabilities_need_at_most_one_tile_more_and_a_flag_byte_per_row():
    # the chunk buffer holds whole 256-row tiles when the forward stores into it
    for T in (16, 2048):
        st = R.rlloss_workspace_bytes(_cfg(T=T))
        rc = R.rlloss_workspace_bytes(_cfg(T=T, flags=R.FLAG_RECOMPUTE))
        assert rc <= st <= rc + 256 * 576 * 2 + 2 * T + 512


def test_workspace_grows_only_by_row_state_beyond_the_chunk():
    """Past the chunk buffer the workspace grows by O(N) row state only, not by
    O(N*H): doubling a batch whose sequences do not fit a group (T = 32768, one
    pass) adds at most about 128 bytes per added token, whether the backward
    stores probabilities or recomputes (each chunk gathers its own X rows)."""
    for flags in (0, R.FLAG_RECOMPUTE):
        for H in (896, 4096):
            small = R.rlloss_workspace_bytes(R.make_cfg(64, 32768, H, 151936, flags=flags))
            big = R.rlloss_workspace_bytes(R.make_cfg(128, 32768, H, 151936, flags=flags))
            added = 64 * 32768
            assert 0 < big - small <= 128 * added, (flags, H, (big - small) / added)


def test_small_chunks_bound_the_workspace():
    """RLLOSS_FLAG_RECOMPUTE with 256-row chunks keeps the workspace below the
    pages' fused-path peaks at every shape of the GMPO page's H100 memory
    comparison (1.34-29.44 GiB), and the default stays within a few GiB."""
    gib = 2 ** 30
    for B, T in ((1, 512), (8, 2048), (16, 4096), (2, 32768), (128, 32768)):
        cfg = R.make_cfg(B, T, 896, 151936, flags=R.FLAG_RECOMPUTE)
        cfg.chunk_rows = 256
        assert R.rlloss_workspace_bytes(cfg) < 0.6 * gib, (B, T)
        assert R.rlloss_workspace_bytes(R.make_cfg(B, T, 896, 151936)) < 3.5 * gib, (B, T)


class _Null:
    def data_ptr(self):
        return 0


def _call(cfg):
    """fwd_bwd with null tensors: must be rejected before touching the GPU."""
    return R.lib.rlloss_fwd_bwd(ctypes.byref(cfg), *([None] * 16), None, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(is_level=R.IS_SEQUENCE), R.EINVAL),          # GMPO rejects sequence-level IS
    (dict(top_entropy_quantile=1.0001), R.EINVAL),     # q outside [0, 1]
    (dict(top_entropy_quantile=-0.01), R.EINVAL),
    (dict(top_entropy_quantile=float("nan")), R.EINVAL),
    (dict(temperature=0.0), R.EINVAL),
    (dict(temperature=-1.0), R.EINVAL),
    (dict(eps_low=-0.1), R.EINVAL),
    (dict(B=0), R.EINVAL),
    (dict(V=0), R.EINVAL),
    (dict(loss_type=7), R.EINVAL),
    (dict(dtype=3), R.EINVAL),
    (dict(H=60), R.EUNSUPPORTED),                       # bf16 rows must be 16-byte multiples
    (dict(loss_type=R.GSPO_TOKEN, beta=0.1), R.EUNSUPPORTED),
    (dict(loss_type=R.GSPO_TOKEN, top_entropy_quantile=0.5), R.EUNSUPPORTED),
    (dict(flags=R.FLAG_ADV_PER_TOKEN), R.EUNSUPPORTED),  # per-token advantages: GSPO only
    (dict(flags=0x80), R.EINVAL),                       # unknown flag
    (dict(dtype=R.FP8_E4M3), R.EUNSUPPORTED),            # e4m3 operands: forward-only scoring
    (dict(), R.EINVAL),                                 # valid cfg, null pointers
])
def test_invalid_requests_rejected_synchronously(kw, code):
    assert _call(_cfg(**kw)) == code


def test_accumulate_flag_is_accepted_and_needs_no_extra_workspace():
    # accumulation runs the recompute backward
    assert R.rlloss_workspace_bytes(_cfg(flags=R.FLAG_ACCUMULATE)) == \
        R.rlloss_workspace_bytes(_cfg(flags=R.FLAG_RECOMPUTE))
    assert R.rlloss_workspace_bytes(_cfg(flags=R.FLAG_ACCUMULATE | R.FLAG_ALL_ROWS)) > 0
    assert R.rlloss_workspace_bytes(_cfg(flags=0x40)) == 0


def test_vocab_shard_entries_validate_before_any_launch():
    cfg = _cfg()
    full = R.rlloss_workspace_bytes(cfg)
    assert 0 < R.rlloss_shard_loss_workspace_bytes(cfg) < full
    assert 0 < R.rlloss_backward_shard_workspace_bytes(cfg) <= full
    assert R.rlloss_shard_loss_workspace_bytes(_cfg(V=0)) == 0
    assert R.rlloss_backward_shard_workspace_bytes(_cfg(temperature=0.0)) == 0
    P = [None] * 13
    assert R.lib.rlloss_loss_from_shards(ctypes.byref(cfg), 0, *P, None, 0, None) == R.EINVAL
    assert R.lib.rlloss_loss_from_shards(ctypes.byref(cfg), R.MAX_SHARDS + 1, *P, None, 0, None) == R.EINVAL
    assert R.lib.rlloss_loss_from_shards(ctypes.byref(cfg), 2, *P, None, 0, None) == R.EINVAL
    assert R.lib.rlloss_forward_shard(ctypes.byref(cfg), None, None, None, None, 0, None, None, 0, None) == R.EINVAL
    assert R.lib.rlloss_backward_shard(ctypes.byref(cfg), *([None] * 4), 0, *([None] * 6), 0, None) == R.EINVAL
    e4 = _cfg(dtype=R.FP8_E4M3, H=896)
    assert R.lib.rlloss_forward_shard(ctypes.byref(e4), None, None, None, None, 0, None, None, 0, None) == \
        R.EUNSUPPORTED


def test_gmpo_sequence_is_rejection_matches_page():
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))
    assert g["gmpo_rejects_sequence_level_is"]["value"] is True
    assert _call(_cfg(is_level=R.IS_SEQUENCE)) == R.EINVAL
    # GSPO is a sequence-level ratio by construction and ignores the level
    assert _call(_cfg(loss_type=R.GSPO_TOKEN, is_level=R.IS_SEQUENCE)) == R.EINVAL  # still null pointers
    assert R.rlloss_workspace_bytes(_cfg(loss_type=R.GSPO_TOKEN, is_level=R.IS_SEQUENCE)) > 0


def test_quantile_range_matches_page():
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))["top_entropy_quantile"]
    assert R.rlloss_workspace_bytes(_cfg(top_entropy_quantile=g["valid_min"])) > 0
    assert R.rlloss_workspace_bytes(_cfg(top_entropy_quantile=g["valid_max"])) > 0
    assert R.rlloss_workspace_bytes(_cfg(top_entropy_quantile=float(np.nextafter(np.float32(g["valid_max"]), np.float32(2))))) == 0


def test_forward_only_workspace_is_smaller_and_validated():
    full = R.rlloss_workspace_bytes(_cfg())
    fwd = R.rlloss_forward_workspace_bytes(_cfg())
    assert 0 < fwd < full
    assert R.rlloss_forward_workspace_bytes(_cfg(temperature=0.0)) == 0
    # loss fields do not matter for the scoring pass
    assert R.rlloss_forward_workspace_bytes(_cfg(top_entropy_quantile=7.0)) == fwd
    cfg = _cfg()
    assert R.lib.rlloss_forward(ctypes.byref(cfg), *([None] * 7), None, 0, None) == R.EINVAL


def test_loss_from_logp_validation():
    cfg = _cfg(top_entropy_quantile=0.5)
    rc = R.lib.rlloss_loss_from_logp(ctypes.byref(cfg), *([None] * 10), None, 0, None)
    assert rc == R.EINVAL


@pytest.mark.parametrize("kw,code", [
    (dict(loss_type=R.GSPO_TOKEN, beta=0.1), R.EUNSUPPORTED),
    (dict(loss_type=R.GSPO_TOKEN, top_entropy_quantile=0.5), R.EUNSUPPORTED),
    (dict(flags=R.FLAG_ADV_PER_TOKEN), R.EUNSUPPORTED),
    (dict(top_entropy_quantile=1.5), R.EINVAL),
    (dict(is_level=R.IS_SEQUENCE), R.EINVAL),
    (dict(B=0), R.EINVAL),
])
def test_noalloc_and_workspace_loss_entries_agree_on_rejections(kw, code):
    """The allocation-free loss entry returns the workspace entry's code for a
    configuration that entry rejects (validation runs before any CUDA call)."""
    cfg = _cfg(**kw)
    ws = R.lib.rlloss_loss_from_logp(ctypes.byref(cfg), *([None] * 10), None, 0, None)
    f = R.lib.rlloss_loss_from_logp_noalloc
    f.argtypes = [ctypes.POINTER(R.RllossCfg)] + [ctypes.c_void_p] * 12
    f.restype = ctypes.c_int
    na = f(ctypes.byref(cfg), *([None] * 12))
    assert ws == na == code


def test_noalloc_scratch_limit_is_exported():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "rlloss.h")).read()
    assert "#define RLLOSS_NOALLOC_SCRATCH_BYTES (4u << 20)" in text


def test_e4m3_scoring_validation():
    """e4m3 operands: only through rlloss_forward_e4m3, rows of 16-byte
    multiples, CTA-pair tiles only; the plain forward refuses them."""
    ok = _cfg(dtype=R.FP8_E4M3, H=896)
    assert R.rlloss_forward_workspace_bytes(ok) > 0
    assert R.rlloss_workspace_bytes(ok) == 0                       # no fwd+bwd with e4m3
    assert R.rlloss_forward_workspace_bytes(_cfg(dtype=R.FP8_E4M3, H=904)) == 0   # 904 % 16 != 0
    assert R.rlloss_forward_workspace_bytes(_cfg(dtype=R.FP8_E4M3, H=896, flags=R.FLAG_SINGLE_CTA_TILES)) == 0
    assert R.lib.rlloss_forward(ctypes.byref(ok), *([None] * 7), None, 0, None) == R.EINVAL
    assert R.lib.rlloss_forward_e4m3(ctypes.byref(ok), *([None] * 9), None, 0, None) == R.EINVAL
    bf = _cfg()
    assert R.lib.rlloss_forward_e4m3(ctypes.byref(bf), *([None] * 9), None, 0, None) == R.EINVAL


def test_sequence_split_entries_validate_before_any_launch():
    cfg = _cfg(top_entropy_quantile=0.2)
    assert R.rlloss_select_state_bytes() == 256
    c = ctypes.c_void_p
    # bad pass, missing counts, missing state after pass 0, negative N, bad q
    assert R.lib.rlloss_entropy_hist(None, None, 0, 4, None, c(256), None) == R.EINVAL
    assert R.lib.rlloss_entropy_hist(None, None, 0, 0, None, None, None) == R.EINVAL
    assert R.lib.rlloss_entropy_hist(None, None, 0, 1, None, c(256), None) == R.EINVAL
    assert R.lib.rlloss_entropy_hist(None, None, -1, 0, None, c(256), None) == R.EINVAL
    assert R.lib.rlloss_entropy_hist(None, None, 10, 0, None, c(256), None) == R.EINVAL
    assert R.lib.rlloss_entropy_select(0, c(256), 1.5, c(256), None) == R.EINVAL
    assert R.lib.rlloss_entropy_select(-1, c(256), 0.2, c(256), None) == R.EINVAL
    assert R.lib.rlloss_entropy_select(0, None, 0.2, c(256), None) == R.EINVAL
    assert R.lib.rlloss_entropy_select(0, c(256), 0.2, c(264), None) == R.EINVAL   # state not 16-byte aligned
    P = [None] * 10
    assert R.lib.rlloss_loss_from_logp_dp(ctypes.byref(cfg), cfg.B - 1, *P, None, 0, None) == R.EINVAL
    assert R.lib.rlloss_loss_from_logp_dp(ctypes.byref(cfg), cfg.B, *P, None, 0, None) == R.EINVAL
    gs = _cfg(loss_type=R.GSPO_TOKEN, beta=0.1)
    assert R.lib.rlloss_loss_from_logp_dp(ctypes.byref(gs), gs.B, *P, None, 0, None) == R.EUNSUPPORTED
    with pytest.raises(R.RllossError):
        R.rlloss_metrics_from_sums(cfg, 0, [0.0] * R.NSUMS, 0.0)


def test_metrics_from_sums_follow_the_oracle_definitions():
    """The host finisher turns the batch sums into the loss and the metric
    vector exactly as the oracle defines them (GMPO with K3 KL and the
    entropy mask, and GSPO-token)."""
    import oracle as O
    rng = np.random.default_rng(21)
    B, T = 4, 30
    N = B * T
    mask = (rng.random(N) > 0.3).astype(np.uint8)
    mask[2 * T:3 * T] = 0                                       # a sequence without active tokens
    logp = rng.normal(-3.0, 1.0, N)
    old = logp + rng.normal(0, 0.3, N)
    ref = logp + rng.normal(0, 0.1, N)
    ent = rng.normal(4.0, 1.0, N)
    adv = np.array([1.0, -0.5, 0.8, -1.2])
    r = O.gmpo_loss(logp, old, ref, adv, mask, B, T, 0.2, 0.3, beta=0.04, entropy=ent, q=0.3)
    nh = float(((mask.reshape(B, T) != 0).sum(axis=1) > 0).sum())
    n_act = r.metrics[3]
    sums = [r.loss * B, n_act, r.metrics[1], r.metrics[2] * n_act, r.metrics[5], r.metrics[6] * nh,
            r.metrics[7] * nh, nh]
    cfg = _cfg(B=B, T=T, eps_low=0.2, eps_high=0.3, beta=0.04, top_entropy_quantile=0.3)
    loss, m = R.rlloss_metrics_from_sums(cfg, B, sums, r.metrics[4])
    assert np.float32(loss) == np.float32(r.loss)
    assert np.allclose(m, np.float32(r.metrics), rtol=1e-6)
    # GSPO: the loss is a sum, the clip fraction is over sequences
    mask[2 * T] = 1
    g = O.gspo_token_loss(logp, old, adv, mask, B, T, 0.05, 0.05)
    gs = [g.loss, g.metrics[3], g.metrics[1], 0.0, g.metrics[5], g.metrics[6] * B, g.metrics[7] * B, float(B)]
    gcfg = _cfg(B=B, T=T, loss_type=R.GSPO_TOKEN, eps_low=0.05, eps_high=0.05)
    loss, m = R.rlloss_metrics_from_sums(gcfg, B, gs, float("nan"))
    assert np.float32(loss) == np.float32(g.loss)
    assert np.allclose(m, np.float32(g.metrics), rtol=1e-6, equal_nan=True)


def test_header_is_plain_c():
    """include/rlloss.h compiles as strict C99 (no C++ in the ABI), and every
    declared function is referenced from C."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    names = R.declared_functions()
    body = "\n".join(f"  (void)&{n};" for n in names)
    src = f'#include <stddef.h>\n#include "rlloss.h"\nint main(void) {{\n{body}\n  return 0;\n}}\n'
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "abi.c")
        open(path, "w").write(src)
        r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                            "-I", inc, path], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_debug_build_compiles_and_exports_the_same_functions(tmp_path):
    """The -DRLLOSS_DEBUG variant (device index and TMA-coordinate checks that
    record RLLOSS_DEV_EBOUNDS instead of faulting) builds for sm_103a and
    exports every declared function.  nvcc cross-compiles without a GPU."""
    import shutil
    import subprocess
    from lm_head_log_tma_gb300 import build as B
    try:
        B.nvcc()
    except RuntimeError:
        pytest.skip("no nvcc")
    lib = B.build(debug=True, out=str(tmp_path / "librlloss_debug.so"))
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("no nm")
    out = subprocess.run([nm, "-D", "--defined-only", lib], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in R.declared_functions() if n not in exported]
    assert not missing, missing
    assert R.DEV_EBOUNDS == 0x100
