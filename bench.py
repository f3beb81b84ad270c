#!/usr/bin/env python
"""Throughput of the fused LM-head + GMPO forward+backward on GB300.

One step = one call of rlloss_fwd_bwd over one batch of the Qwen-0.5B
LM-head workload (B=1, T=4096, H=896, V=151936, bf16, GMPO eps 0.4/0.4,
beta 0): forward logits + streamed log-softmax / entropy, loss, and
dX, dW through tensor-core kernels.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the reference arm of this
build) on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused LM-head+GMPO fwd+bwd tokens/s at H896/V151936; % bf16 TC peak"
UNIT = "tokens/s"
WORKLOAD_INDEX = 1
REF_SAMPLE_TOKENS = 512


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunk-rows", type=int, default=0,
                    help="backward chunk (rows of G kept in HBM); 0 = the library's default")
    ap.add_argument("--workload", type=int, default=WORKLOAD_INDEX,
                    help="index into the workload list (default: the B=1 T=4096 Qwen-0.5B LM-head shape)")
    ap.add_argument("--all-configs", action="store_true",
                    help="one JSON line per workload (0-4) with the oracle timed on config 0 and on a "
                         "1-sequence slice of the others; not the single-line default")
    ap.add_argument("--scoring", choices=["bf16", "e4m3"], default=None,
                    help="time the forward-only scoring entry instead (per-token logp/entropy/lse, no "
                         "gradients); e4m3 quantizes X and W per row first (outside the timed region)")
    ap.add_argument("--all-rows", action="store_true",
                    help="run the backward over every row (RLLOSS_FLAG_ALL_ROWS), for comparison")
    ap.add_argument("--recompute", action="store_true",
                    help="recompute every backward row's logits (RLLOSS_FLAG_RECOMPUTE), for comparison")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay measurement")
    ap.add_argument("--no-naive-memory", action="store_true",
                    help="skip the full-logits torch path run for the memory comparison")
    # internal: time the oracle on workload INDEX in a child process whose BLAS
    # thread count was fixed before numpy loaded
    ap.add_argument("--cpu-oracle-child", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-threads", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), float(d["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons, each with
    nvidia-smi's own timestamp, so that the samples taken inside the timed
    region can be picked out exactly."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                       "-lms", str(self.PERIOD_MS), "-i", str(gpu_index)], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        self.marks = []

    def wait_first_sample(self, timeout=10.0):
        t = time.time()
        while self.p is not None and time.time() - t < timeout:
            self.f.flush()
            if os.path.getsize(self.f.name) > 0:
                return
            time.sleep(0.05)

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = [[c.strip() for c in r.split(",")] for r in open(self.f.name).read().strip().splitlines()
                if r.strip()]
        os.unlink(self.f.name)
        if not rows:
            return None

        def stamp(x):
            # "YYYY/MM/DD hh:mm:ss.mmm" in local time -> seconds since the epoch
            whole, _, frac = x.partition(".")
            try:
                return time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + (float("0." + frac) if frac else 0.0)
            except ValueError:
                return None
        a, b = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (None, None)
        sel = [r for r in rows if a is not None and (stamp(r[0]) or 0) >= a and (stamp(r[0]) or 0) <= b]
        aligned = bool(sel)
        if not sel:
            sel = rows[-3:]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in sel if num(r[2]) is not None]
        mx = [num(r[3]) for r in sel if num(r[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in sel:
            for k, name in enumerate(names):
                if len(r) > 6 + k and r[6 + k].lower() == "active":
                    reasons.add(name)
        pw = [num(r[4]) for r in sel if num(r[4]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "sm_mhz_min": min(sm) if sm else None, "reasons": sorted(reasons), "samples": len(sel),
                "power_w_max": max(pw) if pw else None, "power_w_median": statistics.median(pw) if pw else None,
                "aligned_to_timed_region": aligned}


def config_of(spec, world: int) -> dict:
    """The workload description both arms print (synthetic inputs of this shape)."""
    H, V = spec.H, spec.V
    w_bytes = V * H * (4 if spec.dtype == "fp32" else 2)
    return {"workload": spec.name, "B": spec.B, "T": spec.T, "H": H, "V": V,
            "loss": "gmpo" if spec.loss_type == 0 else "gspo_token", "dtype_in": spec.dtype,
            "eps_low": spec.eps_low, "eps_high": spec.eps_high, "beta": spec.beta,
            "temperature": spec.temperature, "top_entropy_quantile": spec.top_entropy_quantile,
            "bias": spec.has_bias,
            "l2": (f"inputs larger than L2 (W is {w_bytes / 1e6:.0f} MB, dW {V * H * 4 / 1e6:.0f} MB)"
                   if w_bytes > 129e6 else "inputs fit in L2 (not flushed between steps)"),
            "parallelism": "replicas" if world > 1 else "single"}


def max_over_ranks(x: float, device) -> float:
    """The largest of each rank's ``x`` (time-like values: the slowest rank
    sets the whole job's time).  Works with nccl (device tensors) and gloo
    (CPU tensors); a single process returns ``x``."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, steps: int, seconds: float) -> float:
    """Units per second over all ranks: every rank processes the same
    ``units_per_rank`` per step (weak scaling)."""
    return units_per_rank * world * steps / seconds


def make_workload(dev, index=WORKLOAD_INDEX):
    """Seeded inputs on the device; the sampler (and reference) log-probs are
    the policy's plus noise, where the policy logp comes from a plain chunked
    full-logits pass (cuBLAS matmul, fp32 log-softmax) used only to build
    this input."""
    import torch
    from lm_head_log_tma_gb300.workloads import WORKLOADS, make_inputs
    spec = WORKLOADS[index]
    inp = make_inputs(spec, device=dev)
    N = spec.N
    pol = torch.empty(N, dtype=torch.float32, device=dev)
    with torch.no_grad():
        for r0 in range(0, N, 1024):
            z = (inp.X[r0:r0 + 1024] @ inp.W.T).float()
            if inp.b is not None:
                z += inp.b.float()
            z /= spec.temperature
            pol[r0:r0 + 1024] = z.gather(1, inp.targets[r0:r0 + 1024, None])[:, 0] - torch.logsumexp(z, 1)
            del z
    old = inp.old_logp(pol)
    ref = inp.ref_logp(pol)
    torch.cuda.synchronize()
    return spec, inp, old, ref


def cfg_for(R, spec, chunk_rows=0, flags=0):
    return R.make_cfg(spec.B, spec.T, spec.H, spec.V, dtype=R.BF16 if spec.dtype == "bf16" else R.FP32,
                      loss_type=spec.loss_type, eps_low=spec.eps_low, eps_high=spec.eps_high, beta=spec.beta,
                      temperature=spec.temperature, top_entropy_quantile=spec.top_entropy_quantile,
                      has_bias=spec.has_bias, chunk_rows=chunk_rows, flags=flags)


NAIVE_BYTES_PER_LOGIT = 24.5   # measured peak of the path below at B=1, T=4096


def naive_peak_extra_bytes(spec, inp, old, dev):
    """Peak device memory above the inputs of a plain full-logits autograd
    path over the same batch (fp32 logits, log-softmax, target gather,
    entropy, the GMPO sequence term, backward to X and W) -- the comparison
    point for the fused path's workspace.  Returns (bytes or None, note):
    not run when its estimate exceeds 70% of the free device memory."""
    import torch
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info(dev)
    est = NAIVE_BYTES_PER_LOGIT * spec.N * spec.V
    if est > 0.7 * free:
        return None, f"not run: needs about {est / 2**30:.0f} GiB, {free / 2**30:.0f} GiB free"
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    try:
        X = inp.X.detach().clone().requires_grad_(True)
        W = inp.W.detach().clone().requires_grad_(True)
        z = (X @ W.T).float()
        if inp.b is not None:
            z = z + inp.b.float()
        lp = torch.log_softmax(z / spec.temperature, dim=-1)
        logp = lp.gather(1, inp.targets[:, None])[:, 0]
        ent = -(lp.exp() * lp).sum(-1)
        m = inp.mask.float().view(spec.B, spec.T)
        lr = (logp - old).view(spec.B, spec.T)
        adv = inp.adv.view(spec.B, 1)
        clr = torch.where(adv > 0, lr.clamp(max=spec.eps_high), lr.clamp(min=-spec.eps_low))
        r = torch.exp((clr * m).sum(1) / m.sum(1).clamp(min=1))
        loss = -(inp.adv * r).mean() + 0.0 * ent.sum()
        loss.backward()
        torch.cuda.synchronize(dev)
        peak = torch.cuda.max_memory_allocated(dev) - base
        del X, W, z, lp, logp, ent, lr, clr, r, loss
        note = "measured"
    except torch.OutOfMemoryError:
        peak, note = None, "out of memory"
    torch.cuda.empty_cache()
    return peak, note


def oracle_sample_rate(spec, inp, old, ref, tokens):
    """Oracle fwd+bwd over the last ``tokens`` rows of the batch (within the
    last sequence) taken as one sequence, or over the whole batch when
    ``tokens`` is N.  Returns (tokens/s, seconds, threads)."""
    import numpy as np
    import oracle as O
    n = spec.N
    if tokens == n:
        prob = O.Problem(spec.B, spec.T, spec.loss_type, spec.eps_low, spec.eps_high, spec.beta, spec.temperature,
                         spec.top_entropy_quantile)
        threads = os.cpu_count() or 1
        c = lambda x: None if x is None else x.cpu()
        t = time.perf_counter()
        O.fwd_bwd(prob, c(inp.X), c(inp.W), c(inp.b), c(inp.targets), c(old), c(ref), c(inp.adv), c(inp.mask),
                  threads=threads)
        dt = time.perf_counter() - t
        return tokens / dt, dt, threads
    r0 = n - tokens
    X = inp.X[r0:].cpu()
    W = inp.W.cpu()
    b = None if inp.b is None else inp.b.cpu()
    y = inp.targets[r0:].cpu()
    oldc = old[r0:].cpu()
    refc = None if ref is None else ref[r0:].cpu()
    mask = inp.mask[r0:].cpu()
    adv = inp.adv[-1:].cpu()
    prob = O.Problem(1, tokens, spec.loss_type, spec.eps_low, spec.eps_high, spec.beta, spec.temperature,
                     spec.top_entropy_quantile)
    threads = os.cpu_count() or 1
    t = time.perf_counter()
    O.fwd_bwd(prob, X, W, b, y, oldc, refc, adv, mask, threads=threads)
    dt = time.perf_counter() - t
    return tokens / dt, dt, threads


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_child(index, threads):
    """Body of --cpu-oracle-child: the oracle's fwd+bwd of the whole batch of
    workload ``index`` (CPU inputs from the same seeds; sampler log-probs from
    a CPU full-logits pass), repeated for at least 2 s.  Prints one JSON line."""
    import torch
    import oracle as O
    from lm_head_log_tma_gb300.workloads import WORKLOADS, make_inputs
    spec = WORKLOADS[index]
    inp = make_inputs(spec, device="cpu")
    z = (inp.X.double() @ inp.W.double().T)
    if inp.b is not None:
        z += inp.b.double()
    z /= spec.temperature
    pol = (z.gather(1, inp.targets[:, None])[:, 0] - torch.logsumexp(z, 1)).float()
    old, ref = inp.old_logp(pol), inp.ref_logp(pol)
    prob = O.Problem(spec.B, spec.T, spec.loss_type, spec.eps_low, spec.eps_high, spec.beta, spec.temperature,
                     spec.top_entropy_quantile)
    nt = threads or os.cpu_count() or 1
    run = lambda: O.fwd_bwd(prob, inp.X, inp.W, inp.b, inp.targets, old, ref, inp.adv, inp.mask, threads=nt)
    run()
    reps, t = 0, time.perf_counter()
    while reps < 3 or time.perf_counter() - t < 2.0:
        run()
        reps += 1
    dt = (time.perf_counter() - t) / reps
    print(json.dumps({"value": spec.N / dt, "unit": UNIT, "seconds_per_batch": dt, "threads": nt,
                      "reps": reps}), flush=True)
    return 0


def oracle_child_rate(index, threads):
    """Runs oracle_child in a fresh process: with threads == 1 every BLAS and
    OpenMP pool is held to one thread as well."""
    env = dict(os.environ)
    if threads == 1:
        env.update(OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1", BLIS_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-oracle-child", str(index),
                        "--oracle-threads", str(threads)], env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        raise RuntimeError("oracle child failed: " + r.stderr[-500:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if dev == "cuda":
        torch.cuda.set_device(local)
    from lm_head_log_tma_gb300.workloads import WORKLOADS, make_inputs
    spec = WORKLOADS[WORKLOAD_INDEX]
    inp = make_inputs(spec, device="cpu")
    # sampler log-probs: any value near the policy's keeps the clip mix realistic;
    # the oracle's own timing does not depend on it
    import oracle as O
    _, lp, _ = O.row_stats(inp.X[-REF_SAMPLE_TOKENS:], inp.W, inp.b, inp.targets[-REF_SAMPLE_TOKENS:],
                           spec.temperature)
    pol = torch.zeros(spec.N)
    pol[-REF_SAMPLE_TOKENS:] = torch.from_numpy(lp).float()
    old = inp.old_logp(pol)
    ref = inp.ref_logp(pol)
    for _ in range(args.warmup):
        oracle_sample_rate(spec, inp, old, ref, REF_SAMPLE_TOKENS)
    t = time.perf_counter()
    threads = os.cpu_count() or 1
    for _ in range(args.steps):
        _, _, threads = oracle_sample_rate(spec, inp, old, ref, REF_SAMPLE_TOKENS)
    dt = time.perf_counter() - t
    value = REF_SAMPLE_TOKENS * args.steps / dt
    sample = (f"last {REF_SAMPLE_TOKENS} tokens of the {spec.name} batch as one sequence, full H and V, "
              f"fp64 numpy oracle fwd+bwd per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(spec, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist
    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    indices = range(5) if args.all_configs else [args.workload]
    for k in indices:
        line = measure_scoring(args, k, dev, world) if args.scoring else measure(args, k, dev, world, rank, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()
    if world > 1:
        dist.destroy_process_group()
    return 0


def measure_scoring(args, index, dev, world):
    """Forward-only scoring throughput (rlloss_forward / rlloss_forward_e4m3)
    on workload ``index``: tokens/s and 2*N*H*V flop per step."""
    import torch
    from lm_head_log_tma_gb300 import rlloss as R
    from lm_head_log_tma_gb300.workloads import WORKLOADS, make_inputs
    spec = WORKLOADS[index]
    inp = make_inputs(spec, device=dev)
    N, H, V = spec.N, spec.H, spec.V
    peak, peak_sus, _, peak_src = load_peaks()
    if args.scoring == "e4m3":
        def q(x):
            x = x.float()
            sc = (x.abs().amax(dim=1) / 448.0).clamp(min=1e-30)
            return (x / sc[:, None]).to(torch.float8_e4m3fn), sc.contiguous()
        X8, xs = q(inp.X)
        W8, wsc = q(inp.W)
        b = None if inp.b is None else inp.b.float()
        cfg = R.make_cfg(spec.B, spec.T, H, V, dtype=R.FP8_E4M3, temperature=spec.temperature,
                         has_bias=spec.has_bias)
        call = lambda ws: R.forward_e4m3(cfg, X8, xs, W8, wsc, b, inp.targets, workspace=ws)
        dtype, bf16_equiv_peak = "e4m3", 2 * peak
    else:
        cfg = cfg_for(R, spec)
        call = lambda ws: R.forward(cfg, inp.X, inp.W, inp.b, inp.targets, workspace=ws)
        dtype, bf16_equiv_peak = spec.dtype, peak
    ws = R.alloc_workspace(R.rlloss_forward_workspace_bytes(cfg), dev)
    for _ in range(max(3, args.warmup)):
        call(ws)
    torch.cuda.synchronize()
    assert R.rlloss_get_device_status(ws) == 0
    clocks = ClockSampler(dev.index or 0)
    clocks.wait_first_sample()
    time.sleep(0.1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark()
    e0.record()
    for _ in range(args.steps):
        call(ws)
    e1.record()
    torch.cuda.synchronize()
    clocks.mark()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dev) / args.steps
    tflops = 2.0 * N * H * V / (ms / 1e3) / 1e12
    return {"metric": "LM-head forward-only scoring tokens/s (logp, entropy, lse) at H896/V151936",
            "value": whole_job_rate(N, world, args.steps, ms * args.steps / 1e3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": {"workload": spec.name, "B": spec.B, "T": spec.T, "H": H, "V": V, "mode": "scoring"},
            "tflops_2nhv": tflops,
            "peak_frac": tflops / bf16_equiv_peak,
            "peak_note": (f"{peak_src} bf16 burst x 2 (the nominal e4m3:bf16 ratio)" if dtype == "e4m3"
                          else f"{peak_src} bf16 burst"),
            "clocks": clk}


def measure(args, index, dev, world, rank, local):
    """One bench line for workload ``index``."""
    import torch
    import torch.distributed as dist
    from lm_head_log_tma_gb300 import rlloss as R

    spec, inp, old, ref = make_workload(dev, index)
    cfg = cfg_for(R, spec, args.chunk_rows, (R.FLAG_ALL_ROWS if args.all_rows else 0) |
                  (R.FLAG_RECOMPUTE if args.recompute else 0))
    N, H, V = spec.N, spec.H, spec.V
    ws_bytes = R.rlloss_workspace_bytes(cfg)
    naive_bytes, naive_note = (None, "skipped") if args.no_naive_memory else naive_peak_extra_bytes(
        spec, inp, old, dev)
    ws = R.alloc_workspace(ws_bytes, dev)
    outs = None

    def step():
        nonlocal outs
        outs = R.fwd_bwd(cfg, inp.X, inp.W, inp.b, inp.targets, old, ref, inp.adv, inp.mask, workspace=ws,
                         outputs=outs, per_token=False)

    def barrier():
        if world > 1:
            dist.barrier()

    step()   # outputs allocated here; later calls reuse them
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    mem0 = torch.cuda.memory_allocated(dev)
    for _ in range(max(3, args.warmup) - 1):
        step()
    torch.cuda.synchronize()
    call_alloc = torch.cuda.max_memory_allocated(dev) - mem0
    status = R.rlloss_get_device_status(ws)
    bwd_rows = R.rlloss_get_backward_rows(ws)   # recomputed rows with c_n != 0
    st_rows = R.rlloss_get_stored_rows(ws)      # rows whose dX, dW came from the stored probabilities
    st_pos = R.rlloss_get_stored_positions(ws)  # buffer rows those dX, dW ran over (taken 128-row blocks)
    # rows the forward computed: whole row tiles holding an unmasked row
    fwd_rows = min(N, R.rlloss_get_forward_tiles(ws) * (128 if (cfg.flags & R.FLAG_SINGLE_CTA_TILES) else 256))
    if status != 0:
        raise RuntimeError(f"device status {status:#x}")

    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.wait_first_sample()
    time.sleep(0.1)
    R.rlloss_phase_timing(True)
    n_launch0 = R.rlloss_kernel_launches()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark()
    barrier()
    launches = R.rlloss_kernel_launches() - n_launch0
    phase_ms, phase_n = R.rlloss_phase_times()
    R.rlloss_phase_timing(False)
    time.sleep(0.2)
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    ms_step = ms / args.steps
    value = whole_job_rate(N, world, args.steps, ms / 1e3)

    # ---- host time to enqueue one call (plan, tensor maps, launches), each
    # call from an empty queue (back to back, a call of many launches would
    # fill the launch queue and wait for the GPU instead)
    th = []
    for _ in range(20):
        torch.cuda.synchronize()
        t0h = time.perf_counter()
        step()
        th.append(time.perf_counter() - t0h)
    torch.cuda.synchronize()
    host_us = 1e6 * statistics.median(th)

    # ---- the same step captured once in a CUDA graph and replayed (every
    # operation of a call is stream-ordered and allocation-free)
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        gms = max_over_ranks(e0.elapsed_time(e1), dev) / args.steps
        graph = {"ms_per_step": gms, "value": whole_job_rate(N, world, args.steps, gms * args.steps / 1e3),
                 "unit": UNIT, "note": "one captured call replayed per step; kernels identical to the eager call"}
        del g

    # ---- end to end through the public API with host buffers: every step
    # copies its inputs from pinned host memory and reads its loss and
    # metrics back.  The copies of step k+1 run on a copy stream while step k
    # computes (two device buffer sets), as a training loop's input pipeline
    # would; each step's result is read back before the next step is issued.
    host = {k: v.cpu().pin_memory() for k, v in dict(X=inp.X, W=inp.W, targets=inp.targets, old=old,
                                                       adv=inp.adv, mask=inp.mask).items()}
    if inp.b is not None:
        host["b"] = inp.b.cpu().pin_memory()
    if ref is not None:
        host["ref"] = ref.cpu().pin_memory()
    dbufs = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    res_host = [torch.empty(1 + R.NMETRICS, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = res_host[0].numel() * 4
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]

    def issue_copy(k):
        slot = k % 2
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[slot])
            for name in host:
                dbufs[slot][name].copy_(host[name], non_blocking=True)
            copied[slot].record(copy_stream)

    done = [torch.cuda.Event(), torch.cuda.Event()]
    seen = []

    def e2e_run(n):
        # Each step's loss and metrics are read back to the host; the host
        # waits for step k-1's before returning to enqueue step k+1, so its own
        # per-call work overlaps step k on the GPU (a training loop that logs
        # the previous step's loss does the same).
        nonlocal outs
        issue_copy(0)
        for k in range(n):
            slot = k % 2
            if k + 1 < n:
                issue_copy(k + 1)
            stream.wait_event(copied[slot])
            d = dbufs[slot]
            outs = R.fwd_bwd(cfg, d["X"], d["W"], d.get("b"), d["targets"], d["old"], d.get("ref"), d["adv"],
                             d["mask"], workspace=ws, outputs=outs, per_token=False)
            consumed[slot].record(stream)
            res_host[slot][:1].copy_(outs["loss"], non_blocking=True)
            res_host[slot][1:].copy_(outs["metrics"], non_blocking=True)
            done[slot].record(stream)
            if k > 0:
                done[1 - slot].synchronize()
                seen.append(float(res_host[1 - slot][0]))
        done[(n - 1) % 2].synchronize()
        seen.append(float(res_host[(n - 1) % 2][0]))

    e2e_steps = max(3, args.steps)   # as many steps as the device-timed region: the same clock regime
    e2e_run(3)
    barrier()
    torch.cuda.synchronize()
    t = time.perf_counter()
    e2e_run(e2e_steps)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t, dev)
    e2e_value = whole_job_rate(N, world, e2e_steps, e2e_s)

    # ---- roofline of the dominant tensor-core kernel (phase timing, same timed region)
    peak, peak_sus, hbm, peak_src = load_peaks()
    per_step = [m / args.steps for m in phase_ms]
    # tensor-core phases and the flop they execute per step: the forward over
    # its rows, the recompute over the recomputed rows, dX/dW over those and
    # the stored-probability blocks' rows
    gemm_phases = {0: ("fwd_gemm", 2.0 * fwd_rows), 2: ("bwd_dlogits", 2.0 * bwd_rows),
                   3: ("bwd_dX_dW", 4.0 * (bwd_rows + st_pos))}
    dom = max(gemm_phases, key=lambda k: per_step[k])
    flops_phase = gemm_phases[dom][1] * H * V
    launches_per_step = max(1, phase_n[dom] // args.steps)
    achieved = flops_phase / (per_step[dom] / 1e3) / 1e12
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic_qwen05b_t4096.txt")
    if os.path.exists(tp):   # counters taken for this backward form only
        tr = json.load(open(tp))
        if tr.get("backward") == ("stored" if st_rows > 0 else "recompute"):
            traffic = tr.get(gemm_phases[dom][0])
    roofline = {"bound": "tensor", "kernel": gemm_phases[dom][0], "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} bf16 burst", "frac_of_sustained": achieved / peak_sus,
                "launches_per_step": launches_per_step}
    step_tflops = 6.0 * N * H * V / (ms_step / 1e3) / 1e12
    executed_tflops = (2.0 * fwd_rows + 4.0 * st_pos + 6.0 * bwd_rows) * H * V / (ms_step / 1e3) / 1e12

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(spec, world),
            "tc_peak_frac_6nhv": step_tflops / peak,
            "tc_tflops_6nhv": step_tflops,
            "forward_rows": fwd_rows,
            "backward_rows": bwd_rows,
            "stored_rows": st_rows,
            "stored_block_rows": st_pos,
            "executed_tflops": executed_tflops,
            "executed_peak_frac": executed_tflops / peak,
            "roofline": roofline,
            "phases_ms_per_step": {R.PHASE_NAMES[i]: per_step[i] for i in range(R.NPHASES)},
            "clocks": clk,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps,
                    "pipeline": "step k+1's H2D copies overlap step k on a copy stream; step k-1's loss and "
                                "metrics are read back while step k runs"},
            "gpu_launches": launches,
            "cuda_graph": graph,
            "host_enqueue_us_per_call": host_us,
            "memory": {"library_workspace_bytes": ws_bytes, "allocated_during_call_bytes": call_alloc,
                       "naive_full_logits_peak_extra_bytes": naive_bytes,
                       "naive_fits": naive_bytes is not None, "naive_note": naive_note,
                       "chunk_rows": args.chunk_rows or "default",
                       "backward": ("dense" if args.all_rows else "rows with c_n != 0") +
                                   ("; dX, dW of the stored rows from the forward's stored probabilities"
                                    if st_rows > 0 else "; every row recomputed")}}

    if rank == 0 and not args.no_cpu_baseline:
        # config 0 whole (1 thread and all threads), the others one whole sequence
        tokens = N if index == 0 else spec.T
        what = "the whole batch" if index == 0 else f"the last sequence ({spec.T} tokens)"
        if index == 0:
            one, every = oracle_child_rate(0, 1), oracle_child_rate(0, 0)
            rate, secs, threads = every["value"], every["seconds_per_batch"] * every["reps"], every["threads"]
        else:
            rate, secs, threads = oracle_sample_rate(spec, inp, old, ref, tokens)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "cpu_model": cpu_model(),
                                "sample": f"{what}, full H and V, fp64 numpy fwd+bwd ({secs:.1f} s)"}
        if index == 0:
            line["cpu_baseline"]["threads_1"] = one
            line["cpu_baseline"]["threads_all"] = every
    return line


def main():
    args = parse_args()
    if args.cpu_oracle_child is not None:
        return oracle_child(args.cpu_oracle_child, args.oracle_threads)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
