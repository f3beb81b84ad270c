"""ctypes binding of librlloss.so (include/rlloss.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library.  torch supplies device memory and streams.  Importing
this module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re
from ctypes import c_float, c_int, c_int32, c_size_t, c_uint32, c_uint64, c_void_p

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librlloss.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "rlloss.h")

OK, EINVAL, EUNSUPPORTED, EWORKSPACE, ECUDA = 0, 1, 2, 3, 4
DEV_ETIMEOUT, DEV_ENONFINITE, DEV_EBADTARGET, DEV_EEMPTYSEQ = 0x10, 0x20, 0x40, 0x80
DEV_EBOUNDS = 0x100     # builds with -DRLLOSS_DEBUG only
BF16, FP32, FP8_E4M3 = 0, 1, 2
GMPO, GSPO_TOKEN = 0, 1
IS_TOKEN, IS_SEQUENCE = 0, 1
FLAG_FORCE_ENTROPY_PATH = 0x1
FLAG_SINGLE_CTA_TILES = 0x2
FLAG_ADV_PER_TOKEN = 0x4
FLAG_ALL_ROWS = 0x8
FLAG_ACCUMULATE = 0x10
FLAG_RECOMPUTE = 0x20
NMETRICS = 8
STATE_FLOATS = 8        # floats per token of a vocabulary shard's row state
MAX_SHARDS = 4096
SELECT_PASSES = 4       # passes of the distributed entropy quantile
SELECT_COUNTS = 512     # uint32 counts per pass
NSUMS = 8               # doubles of batch sums (sequence-split batches)


class RllossCfg(ctypes.Structure):
    _fields_ = [("B", c_int32), ("T", c_int32), ("H", c_int32), ("V", c_int32),
                ("dtype", c_int32), ("loss_type", c_int32), ("is_level", c_int32),
                ("eps_low", c_float), ("eps_high", c_float), ("beta", c_float),
                ("temperature", c_float), ("top_entropy_quantile", c_float),
                ("has_bias", c_int32), ("flags", c_uint32), ("chunk_rows", c_int32)]


def make_cfg(B, T, H=0, V=0, dtype=BF16, loss_type=GMPO, is_level=IS_TOKEN, eps_low=0.4,
             eps_high=0.4, beta=0.0, temperature=1.0, top_entropy_quantile=1.0, has_bias=False,
             flags=0, chunk_rows=0) -> RllossCfg:
    return RllossCfg(B, T, H, V, dtype, loss_type, is_level, eps_low, eps_high, beta, temperature,
                     top_entropy_quantile, int(bool(has_bias)), flags, chunk_rows)


class RllossError(RuntimeError):
    def __init__(self, code, where=""):
        super().__init__(f"{where}: {status_str(code)} ({code})")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"librlloss.so is not built ({LIB_PATH}); run lm_head_log_tma_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    cfgp = ctypes.POINTER(RllossCfg)
    lib.rlloss_workspace_bytes.argtypes = [cfgp]
    lib.rlloss_workspace_bytes.restype = c_size_t
    lib.rlloss_loss_workspace_bytes.argtypes = [cfgp]
    lib.rlloss_loss_workspace_bytes.restype = c_size_t
    lib.rlloss_fwd_bwd.argtypes = [cfgp] + [P] * 16 + [P, c_size_t, P]
    lib.rlloss_fwd_bwd.restype = c_int
    lib.rlloss_forward_workspace_bytes.argtypes = [cfgp]
    lib.rlloss_forward_workspace_bytes.restype = c_size_t
    lib.rlloss_forward.argtypes = [cfgp] + [P] * 7 + [P, c_size_t, P]
    lib.rlloss_forward.restype = c_int
    lib.rlloss_forward_e4m3.argtypes = [cfgp] + [P] * 9 + [P, c_size_t, P]
    lib.rlloss_forward_e4m3.restype = c_int
    lib.rlloss_loss_from_logp.argtypes = [cfgp] + [P] * 10 + [P, c_size_t, P]
    lib.rlloss_loss_from_logp.restype = c_int
    lib.rlloss_forward_shard.argtypes = [cfgp, P, P, P, P, ctypes.c_int64, P, P, c_size_t, P]
    lib.rlloss_forward_shard.restype = c_int
    lib.rlloss_shard_loss_workspace_bytes.argtypes = [cfgp]
    lib.rlloss_shard_loss_workspace_bytes.restype = c_size_t
    lib.rlloss_loss_from_shards.argtypes = [cfgp, c_int32] + [P] * 13 + [P, c_size_t, P]
    lib.rlloss_loss_from_shards.restype = c_int
    lib.rlloss_backward_shard_workspace_bytes.argtypes = [cfgp]
    lib.rlloss_backward_shard_workspace_bytes.restype = c_size_t
    lib.rlloss_backward_shard.argtypes = [cfgp, P, P, P, P, ctypes.c_int64, P, P, P, P, P, P, c_size_t, P]
    lib.rlloss_backward_shard.restype = c_int
    lib.rlloss_select_state_bytes.argtypes = []
    lib.rlloss_select_state_bytes.restype = c_size_t
    lib.rlloss_entropy_hist.argtypes = [P, P, ctypes.c_int64, c_int32, P, P, P]
    lib.rlloss_entropy_hist.restype = c_int
    lib.rlloss_entropy_select.argtypes = [c_int32, P, c_float, P, P]
    lib.rlloss_entropy_select.restype = c_int
    lib.rlloss_select_threshold.argtypes = [P, ctypes.POINTER(ctypes.c_double)]
    lib.rlloss_select_threshold.restype = c_int
    lib.rlloss_loss_from_logp_dp.argtypes = [cfgp, c_int32] + [P] * 10 + [P, c_size_t, P]
    lib.rlloss_loss_from_logp_dp.restype = c_int
    lib.rlloss_metrics_from_sums.argtypes = [cfgp, c_int32, ctypes.POINTER(ctypes.c_double), ctypes.c_double,
                                             ctypes.POINTER(c_float), ctypes.POINTER(c_float)]
    lib.rlloss_metrics_from_sums.restype = c_int
    lib.rlloss_get_device_status.argtypes = [P, ctypes.POINTER(c_int32)]
    lib.rlloss_get_device_status.restype = c_int
    lib.rlloss_get_backward_rows.argtypes = [P, ctypes.POINTER(c_int32)]
    lib.rlloss_get_backward_rows.restype = c_int
    lib.rlloss_get_stored_rows.argtypes = [P, ctypes.POINTER(c_int32)]
    lib.rlloss_get_stored_rows.restype = c_int
    lib.rlloss_get_stored_positions.argtypes = [P, ctypes.POINTER(c_int32)]
    lib.rlloss_get_stored_positions.restype = c_int
    lib.rlloss_get_forward_tiles.argtypes = [P, ctypes.POINTER(c_int32)]
    lib.rlloss_get_forward_tiles.restype = c_int
    lib.rlloss_selftest_bounded_wait.argtypes = [P, c_uint64, P]
    lib.rlloss_selftest_bounded_wait.restype = c_int
    lib.rlloss_phase_timing.argtypes = [c_int]
    lib.rlloss_phase_timing.restype = c_int
    lib.rlloss_phase_times.argtypes = [ctypes.POINTER(c_float), ctypes.POINTER(c_int32), c_int]
    lib.rlloss_phase_times.restype = c_int
    lib.rlloss_kernel_launches.argtypes = []
    lib.rlloss_kernel_launches.restype = c_uint64
    lib.rlloss_status_str.argtypes = [c_int]
    lib.rlloss_status_str.restype = ctypes.c_char_p
    return lib


lib = _load()


def declared_functions() -> list[str]:
    """Function names declared in include/rlloss.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:size_t|int|uint64_t|const char\s*\*)\s*(rlloss_\w+)\s*\(", text, re.M)))


def status_str(code: int) -> str:
    return lib.rlloss_status_str(int(code)).decode()


def _p(t):
    if t is None:
        return None
    return c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------- raw entry points
def rlloss_workspace_bytes(cfg: RllossCfg) -> int:
    return int(lib.rlloss_workspace_bytes(ctypes.byref(cfg)))


def rlloss_loss_workspace_bytes(cfg: RllossCfg) -> int:
    return int(lib.rlloss_loss_workspace_bytes(ctypes.byref(cfg)))


def rlloss_fwd_bwd(cfg, X, W, b, targets, old_logp, ref_logp, adv, mask, out_loss, out_metrics, dX, dW,
                   db, out_logp, out_entropy, out_entropy_mask, workspace, stream=None) -> int:
    return lib.rlloss_fwd_bwd(ctypes.byref(cfg), _p(X), _p(W), _p(b), _p(targets), _p(old_logp),
                              _p(ref_logp), _p(adv), _p(mask), _p(out_loss), _p(out_metrics), _p(dX),
                              _p(dW), _p(db), _p(out_logp), _p(out_entropy), _p(out_entropy_mask),
                              _p(workspace), c_size_t(0 if workspace is None else workspace.numel()),
                              _stream(stream))


def rlloss_forward_workspace_bytes(cfg: RllossCfg) -> int:
    return int(lib.rlloss_forward_workspace_bytes(ctypes.byref(cfg)))


def rlloss_forward(cfg, X, W, b, targets, out_logp, out_entropy, out_lse, workspace, stream=None) -> int:
    return lib.rlloss_forward(ctypes.byref(cfg), _p(X), _p(W), _p(b), _p(targets), _p(out_logp),
                              _p(out_entropy), _p(out_lse), _p(workspace),
                              c_size_t(0 if workspace is None else workspace.numel()), _stream(stream))


def rlloss_forward_e4m3(cfg, X8, x_scale, W8, w_scale, b, targets, out_logp, out_entropy, out_lse, workspace,
                        stream=None) -> int:
    return lib.rlloss_forward_e4m3(ctypes.byref(cfg), _p(X8), _p(x_scale), _p(W8), _p(w_scale), _p(b), _p(targets),
                                   _p(out_logp), _p(out_entropy), _p(out_lse), _p(workspace),
                                   c_size_t(0 if workspace is None else workspace.numel()), _stream(stream))


def rlloss_loss_from_logp(cfg, logp, entropy, old_logp, ref_logp, adv, mask, out_loss, out_metrics,
                          out_dlogp, out_entropy_mask, workspace, stream=None) -> int:
    return lib.rlloss_loss_from_logp(ctypes.byref(cfg), _p(logp), _p(entropy), _p(old_logp),
                                     _p(ref_logp), _p(adv), _p(mask), _p(out_loss), _p(out_metrics),
                                     _p(out_dlogp), _p(out_entropy_mask), _p(workspace),
                                     c_size_t(0 if workspace is None else workspace.numel()),
                                     _stream(stream))


def rlloss_forward_shard(cfg, X, W, b, targets, v_begin, out_state, workspace, stream=None) -> int:
    return lib.rlloss_forward_shard(ctypes.byref(cfg), _p(X), _p(W), _p(b), _p(targets), ctypes.c_int64(v_begin),
                                    _p(out_state), _p(workspace),
                                    c_size_t(0 if workspace is None else workspace.numel()), _stream(stream))


def rlloss_shard_loss_workspace_bytes(cfg: RllossCfg) -> int:
    return int(lib.rlloss_shard_loss_workspace_bytes(ctypes.byref(cfg)))


def rlloss_loss_from_shards(cfg, nshards, states, targets, old_logp, ref_logp, adv, mask, out_loss, out_metrics,
                            out_lse, out_dlogp, out_logp, out_entropy, out_entropy_mask, workspace,
                            stream=None) -> int:
    return lib.rlloss_loss_from_shards(ctypes.byref(cfg), c_int32(nshards), _p(states), _p(targets), _p(old_logp),
                                       _p(ref_logp), _p(adv), _p(mask), _p(out_loss), _p(out_metrics), _p(out_lse),
                                       _p(out_dlogp), _p(out_logp), _p(out_entropy), _p(out_entropy_mask),
                                       _p(workspace), c_size_t(0 if workspace is None else workspace.numel()),
                                       _stream(stream))


def rlloss_backward_shard_workspace_bytes(cfg: RllossCfg) -> int:
    return int(lib.rlloss_backward_shard_workspace_bytes(ctypes.byref(cfg)))


def rlloss_backward_shard(cfg, X, W, b, targets, v_begin, lse, dlogp, dX, dW, db, workspace, stream=None) -> int:
    return lib.rlloss_backward_shard(ctypes.byref(cfg), _p(X), _p(W), _p(b), _p(targets), ctypes.c_int64(v_begin),
                                     _p(lse), _p(dlogp), _p(dX), _p(dW), _p(db), _p(workspace),
                                     c_size_t(0 if workspace is None else workspace.numel()), _stream(stream))


def rlloss_select_state_bytes() -> int:
    return int(lib.rlloss_select_state_bytes())


def rlloss_entropy_hist(entropy, mask, N, pass_, select_state, counts, stream=None) -> int:
    return lib.rlloss_entropy_hist(_p(entropy), _p(mask), ctypes.c_int64(N), c_int32(pass_), _p(select_state),
                                   _p(counts), _stream(stream))


def rlloss_entropy_select(pass_, counts, q, select_state, stream=None) -> int:
    return lib.rlloss_entropy_select(c_int32(pass_), _p(counts), c_float(q), _p(select_state), _stream(stream))


def rlloss_select_threshold(select_state) -> float:
    thr = ctypes.c_double(0.0)
    rc = lib.rlloss_select_threshold(_p(select_state), ctypes.byref(thr))
    if rc != OK:
        raise RllossError(rc, "rlloss_select_threshold")
    return float(thr.value)


def rlloss_loss_from_logp_dp(cfg, B_global, select_state, logp, entropy, old_logp, ref_logp, adv, mask, out_sums,
                             out_dlogp, out_entropy_mask, workspace, stream=None) -> int:
    return lib.rlloss_loss_from_logp_dp(ctypes.byref(cfg), c_int32(B_global), _p(select_state), _p(logp),
                                        _p(entropy), _p(old_logp), _p(ref_logp), _p(adv), _p(mask), _p(out_sums),
                                        _p(out_dlogp), _p(out_entropy_mask), _p(workspace),
                                        c_size_t(0 if workspace is None else workspace.numel()), _stream(stream))


def rlloss_metrics_from_sums(cfg, B_global, sums, threshold):
    """Host only: (loss, metrics list) of the whole batch from the batch sums
    added over ranks (a sequence of NSUMS numbers)."""
    s = (ctypes.c_double * NSUMS)(*[float(x) for x in sums])
    loss = c_float(0.0)
    m = (c_float * NMETRICS)()
    rc = lib.rlloss_metrics_from_sums(ctypes.byref(cfg), c_int32(B_global), s, ctypes.c_double(threshold),
                                      ctypes.byref(loss), m)
    if rc != OK:
        raise RllossError(rc, "rlloss_metrics_from_sums")
    return float(loss.value), [float(x) for x in m]


def rlloss_get_device_status(workspace) -> int:
    st = c_int32(0)
    rc = lib.rlloss_get_device_status(_p(workspace), ctypes.byref(st))
    if rc != OK:
        raise RllossError(rc, "rlloss_get_device_status")
    return int(st.value)


def rlloss_get_forward_tiles(workspace) -> int:
    tiles = c_int32(0)
    rc = lib.rlloss_get_forward_tiles(_p(workspace), ctypes.byref(tiles))
    if rc != OK:
        raise RllossError(rc, "rlloss_get_forward_tiles")
    return int(tiles.value)


def rlloss_get_backward_rows(workspace) -> int:
    rows = c_int32(0)
    rc = lib.rlloss_get_backward_rows(_p(workspace), ctypes.byref(rows))
    if rc != OK:
        raise RllossError(rc, "rlloss_get_backward_rows")
    return int(rows.value)


def rlloss_get_stored_rows(workspace) -> int:
    rows = c_int32(0)
    rc = lib.rlloss_get_stored_rows(_p(workspace), ctypes.byref(rows))
    if rc != OK:
        raise RllossError(rc, "rlloss_get_stored_rows")
    return int(rows.value)


def rlloss_get_stored_positions(workspace) -> int:
    rows = c_int32(0)
    rc = lib.rlloss_get_stored_positions(_p(workspace), ctypes.byref(rows))
    if rc != OK:
        raise RllossError(rc, "rlloss_get_stored_positions")
    return int(rows.value)


def rlloss_selftest_bounded_wait(workspace, limit_ns: int, stream=None) -> int:
    return lib.rlloss_selftest_bounded_wait(_p(workspace), c_uint64(limit_ns), _stream(stream))


NPHASES = 6
PHASE_NAMES = ["fwd_gemm", "merge_mask_loss", "bwd_dlogits", "bwd_dX_dW", "unused", "other"]


def rlloss_phase_timing(enable: bool) -> int:
    return lib.rlloss_phase_timing(int(bool(enable)))


def rlloss_phase_times():
    ms = (c_float * NPHASES)()
    n = (c_int32 * NPHASES)()
    rc = lib.rlloss_phase_times(ms, n, NPHASES)
    if rc != OK:
        raise RllossError(rc, "rlloss_phase_times")
    return [float(x) for x in ms], [int(x) for x in n]


def rlloss_kernel_launches() -> int:
    return int(lib.rlloss_kernel_launches())


# ---------------------------------------------------------------- convenience
def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def fwd_bwd(cfg: RllossCfg, X, W, b, targets, old_logp, ref_logp, adv, mask, workspace=None,
            outputs=None, stream=None, per_token=True):
    """Allocate outputs (torch) and run rlloss_fwd_bwd.  Returns a dict of tensors.
    per_token=False leaves out the per-token logp / entropy outputs (a
    training step needs only loss, metrics and gradients), which lets the
    library skip the forward of row tiles whose rows are all masked."""
    dev = X.device
    N, H, V = cfg.B * cfg.T, cfg.H, cfg.V
    if outputs is None:
        outputs = dict(
            loss=torch.empty(1, dtype=torch.float32, device=dev),
            metrics=torch.empty(NMETRICS, dtype=torch.float32, device=dev),
            dX=torch.empty(N, H, dtype=torch.float32, device=dev),
            dW=torch.empty(V, H, dtype=torch.float32, device=dev),
            db=torch.empty(V, dtype=torch.float32, device=dev) if cfg.has_bias else None,
            logp=torch.empty(N, dtype=torch.float32, device=dev) if per_token else None,
            entropy=torch.empty(N, dtype=torch.float32, device=dev) if per_token else None,
            emask=torch.empty(N, dtype=torch.uint8, device=dev),
        )
    if workspace is None:
        workspace = alloc_workspace(rlloss_workspace_bytes(cfg), dev)
    o = outputs
    rc = rlloss_fwd_bwd(cfg, X, W, b, targets, old_logp, ref_logp, adv, mask, o["loss"], o["metrics"],
                        o["dX"], o["dW"], o.get("db"), o.get("logp"), o.get("entropy"), o.get("emask"),
                        workspace, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_fwd_bwd")
    o["workspace"] = workspace
    return o


def forward(cfg: RllossCfg, X, W, b, targets, workspace=None, stream=None):
    """Scoring pass: per-token logp, entropy and lse (fp32 [N] each)."""
    dev = X.device
    N = cfg.B * cfg.T
    o = {k: torch.empty(N, dtype=torch.float32, device=dev) for k in ("logp", "entropy", "lse")}
    if workspace is None:
        workspace = alloc_workspace(rlloss_forward_workspace_bytes(cfg), dev)
    rc = rlloss_forward(cfg, X, W, b, targets, o["logp"], o["entropy"], o["lse"], workspace, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_forward")
    o["workspace"] = workspace
    return o


def forward_e4m3(cfg: RllossCfg, X8, x_scale, W8, w_scale, b, targets, workspace=None, stream=None):
    """Scoring pass with e4m3 operands (torch.float8_e4m3fn or uint8 tensors)
    and fp32 per-row scales: per-token logp, entropy and lse."""
    dev = X8.device
    N = cfg.B * cfg.T
    o = {k: torch.empty(N, dtype=torch.float32, device=dev) for k in ("logp", "entropy", "lse")}
    if workspace is None:
        workspace = alloc_workspace(rlloss_forward_workspace_bytes(cfg), dev)
    rc = rlloss_forward_e4m3(cfg, X8, x_scale, W8, w_scale, b, targets, o["logp"], o["entropy"], o["lse"],
                             workspace, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_forward_e4m3")
    o["workspace"] = workspace
    return o


def loss_from_logp(cfg: RllossCfg, logp, entropy, old_logp, ref_logp, adv, mask, workspace=None,
                   stream=None):
    dev = logp.device
    N = cfg.B * cfg.T
    o = dict(loss=torch.empty(1, dtype=torch.float32, device=dev),
             metrics=torch.empty(NMETRICS, dtype=torch.float32, device=dev),
             dlogp=torch.empty(N, dtype=torch.float32, device=dev),
             emask=torch.empty(N, dtype=torch.uint8, device=dev))
    if workspace is None:
        workspace = alloc_workspace(rlloss_loss_workspace_bytes(cfg), dev)
    rc = rlloss_loss_from_logp(cfg, logp, entropy, old_logp, ref_logp, adv, mask, o["loss"], o["metrics"],
                               o["dlogp"], o["emask"], workspace, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_loss_from_logp")
    o["workspace"] = workspace
    return o


# ---------------------------------------------------------------- vocabulary shards
def forward_shard(cfg: RllossCfg, X, W, b, targets, v_begin: int, workspace=None, stream=None):
    """Row states [N, STATE_FLOATS] of the vocabulary shard W (rows
    [v_begin, v_begin + cfg.V) of the whole vocabulary)."""
    dev = X.device
    state = torch.empty(cfg.B * cfg.T, STATE_FLOATS, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(rlloss_forward_workspace_bytes(cfg), dev)
    rc = rlloss_forward_shard(cfg, X, W, b, targets, v_begin, state, workspace, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_forward_shard")
    return state, workspace


def loss_from_shards(cfg: RllossCfg, states, targets, old_logp, ref_logp, adv, mask, workspace=None, stream=None):
    """Loss, metrics, lse, dL/dlogp, logp, entropy and entropy mask from the
    row states of all shards (states: [nshards, N, STATE_FLOATS]; cfg.V is
    the whole vocabulary)."""
    dev = states.device
    N = cfg.B * cfg.T
    f = lambda: torch.empty(N, dtype=torch.float32, device=dev)
    o = dict(loss=torch.empty(1, dtype=torch.float32, device=dev),
             metrics=torch.empty(NMETRICS, dtype=torch.float32, device=dev),
             lse=f(), dlogp=f(), logp=f(), entropy=f(), emask=torch.empty(N, dtype=torch.uint8, device=dev))
    if workspace is None:
        workspace = alloc_workspace(rlloss_shard_loss_workspace_bytes(cfg), dev)
    rc = rlloss_loss_from_shards(cfg, states.shape[0], states, targets, old_logp, ref_logp, adv, mask, o["loss"],
                                 o["metrics"], o["lse"], o["dlogp"], o["logp"], o["entropy"], o["emask"],
                                 workspace, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_loss_from_shards")
    o["workspace"] = workspace
    return o


def backward_shard(cfg: RllossCfg, X, W, b, targets, v_begin: int, lse, dlogp, outputs=None, workspace=None,
                   stream=None):
    """This shard's dW rows, db rows and part of dX (cfg.V = the shard's rows)."""
    dev = X.device
    N = cfg.B * cfg.T
    if outputs is None:
        outputs = dict(dX=torch.empty(N, cfg.H, dtype=torch.float32, device=dev),
                       dW=torch.empty(cfg.V, cfg.H, dtype=torch.float32, device=dev),
                       db=torch.empty(cfg.V, dtype=torch.float32, device=dev) if cfg.has_bias else None)
    if workspace is None:
        workspace = alloc_workspace(rlloss_backward_shard_workspace_bytes(cfg), dev)
    o = outputs
    rc = rlloss_backward_shard(cfg, X, W, b, targets, v_begin, lse, dlogp, o["dX"], o["dW"], o.get("db"),
                               workspace, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_backward_shard")
    o["workspace"] = workspace
    return o


# ---------------------------------------------------------------- batch split over ranks by sequences
def alloc_select_state(device="cuda") -> torch.Tensor:
    return torch.zeros(rlloss_select_state_bytes(), dtype=torch.uint8, device=device)


def entropy_hist(entropy, mask, pass_: int, select_state, counts=None, stream=None):
    """This rank's counts [SELECT_COUNTS] (uint32 as int32) for pass ``pass_``."""
    if counts is None:
        counts = torch.empty(SELECT_COUNTS, dtype=torch.int32, device=entropy.device)
    rc = rlloss_entropy_hist(entropy, mask, entropy.numel(), pass_, select_state, counts, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_entropy_hist")
    return counts


def entropy_select(pass_: int, counts, q: float, select_state, stream=None):
    rc = rlloss_entropy_select(pass_, counts, q, select_state, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_entropy_select")


def loss_from_logp_dp(cfg: RllossCfg, B_global: int, select_state, logp, entropy, old_logp, ref_logp, adv, mask,
                      workspace=None, stream=None):
    """One rank's loss stage: its batch sums [NSUMS] (fp64), dL/dlogp of the
    whole batch's loss for its tokens, and its entropy mask."""
    dev = logp.device
    N = cfg.B * cfg.T
    o = dict(sums=torch.empty(NSUMS, dtype=torch.float64, device=dev),
             dlogp=torch.empty(N, dtype=torch.float32, device=dev),
             emask=torch.empty(N, dtype=torch.uint8, device=dev))
    if workspace is None:
        workspace = alloc_workspace(rlloss_loss_workspace_bytes(cfg), dev)
    rc = rlloss_loss_from_logp_dp(cfg, B_global, select_state, logp, entropy, old_logp, ref_logp, adv, mask,
                                  o["sums"], o["dlogp"], o["emask"], workspace, stream)
    if rc != OK:
        raise RllossError(rc, "rlloss_loss_from_logp_dp")
    o["workspace"] = workspace
    return o
