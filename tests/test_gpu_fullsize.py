"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (default chunking and scheduling).

The oracle computes logp and entropy for every row (so the loss, metrics and
entropy threshold are compared exactly as defined), dX on 1024 sampled rows,
dW on 1024 sampled vocabulary rows (including every target of the sampled
rows), and db in full when there is a bias.  Each case takes the oracle a
few seconds to a few minutes on the host cores.
"""
import os

import numpy as np
import pytest
import torch

from lm_head_log_tma_gb300.workloads import WORKLOADS

from parity import Case, check_grads, check_loss_and_metrics, check_rows, reconcile_loss

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def R():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lm_head_log_tma_gb300 import rlloss
    return rlloss


@pytest.mark.parametrize("idx", [1, 2, 3, 4], ids=[WORKLOADS[i].name for i in (1, 2, 3, 4)])
def test_full_size_workload(R, idx):
    spec = WORKLOADS[idx]
    case = Case(spec, threads=os.cpu_count())
    out = case.run_gpu(R)
    assert out["status"] == 0, hex(out["status"])
    el, ee = check_rows(out, case)
    res = reconcile_loss(out, case)
    gl, ol = check_loss_and_metrics(out, case, res)
    rng = np.random.default_rng(1000 + idx)
    rows = np.sort(rng.choice(spec.N, 1024, replace=False))
    vs = np.unique(np.concatenate([rng.choice(spec.V, 512, replace=False),
                                   case.inp.targets.numpy()[rows[:512]], [0, spec.V - 1]]))
    stats = check_grads(out, case, res, dx_rows=rows, dw_rows=vs)
    print(f"{spec.name}: loss {gl:.9g} vs {ol:.9g} (rel {abs(gl - ol) / abs(ol):.2e}); "
          f"logp max err {el:.2e}, entropy max err {ee:.2e}; grads {stats}")
    # the training-step call the bench times (no per-token outputs: fully masked
    # row tiles skip the forward) meets the same bar on the same samples
    del out
    step = case.run_gpu(R, per_token=False)
    assert step["status"] == 0, hex(step["status"])
    res2 = reconcile_loss(step, case)
    check_loss_and_metrics(step, case, res2)
    stats2 = check_grads(step, case, res2, dx_rows=rows, dw_rows=vs)
    print(f"  training-step call: loss {step['loss'].item():.9g}; forward tiles "
          f"{R.rlloss_get_forward_tiles(step['workspace'])}, backward rows "
          f"{R.rlloss_get_backward_rows(step['workspace'])}; grads {stats2}")
