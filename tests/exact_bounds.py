"""Inputs that put a GSPO sequence ratio exactly on a clip bound.

The sequence ratio of the Tinker "GSPO" page is s = exp(mean over the masked
tokens of log p - log q).  To test the bounds themselves (the page's objective
formula and "Choosing clipping thresholds"), a test needs a mean log ratio x
whose fp64 exp is exactly the bound, or exactly one of its fp64 neighbours.

This module holds no arithmetic of the method: it searches fp64 values and
splits one into fp32 pieces.  Both the oracle pins and the GPU test use it.
"""
import numpy as np


def x_on_exp(target: float) -> float:
    """The fp64 x in the middle of the set {x : np.exp(x) == target}.

    The set spans about ulp(target)/target in x, so its middle lies far from
    both ends: the exact exponential there is within a tiny fraction of an
    ulp of ``target``, and any exp accurate to a fraction of an ulp rounds to
    ``target`` as well.  Raises if no fp64 x reaches ``target``."""
    x = np.log(target)
    for _ in range(1 << 16):
        if np.exp(x) >= target:
            break
        x = np.nextafter(x, np.inf)
    for _ in range(1 << 16):
        if np.exp(x) <= target:
            break
        x = np.nextafter(x, -np.inf)
    if np.exp(x) != target:
        raise ValueError(f"no fp64 x with exp(x) == {target!r}")
    lo = x
    while np.exp(np.nextafter(lo, -np.inf)) == target:
        lo = np.nextafter(lo, -np.inf)
    hi = x
    while np.exp(np.nextafter(hi, np.inf)) == target:
        hi = np.nextafter(hi, np.inf)
    mid = lo
    while mid < lo + (hi - lo) / 2:
        mid = np.nextafter(mid, np.inf)
    assert np.exp(mid) == target
    return float(mid)


def fp32_split(y: float):
    """Three fp32 values a, b, c with a + b + c == y exactly in fp64.

    a takes y's leading 24 bits, b the next 24, c the last 5.  Every partial
    sum is then a run of y's own bits, so any summation order is exact."""
    a = np.float32(y)
    b = np.float32(y - float(a))
    c = np.float32(y - float(a) - float(b))
    parts = [float(a), float(b), float(c)]
    for order in ((0, 1, 2), (0, 2, 1), (1, 0, 2), (1, 2, 0), (2, 0, 1), (2, 1, 0)):
        acc = 0.0
        for k in order:
            acc += parts[k]
        assert acc == y
    return a, b, c


def gspo_sequences_on_bounds(lo: float, hi: float):
    """Per-sequence log-prob rows whose masked mean log ratio has fp64 exp equal
    to each bound and to its two fp64 neighbours.

    Returns (targets, logp [k, 5] fp32, old [k, 5] fp32, mask [k, 5] uint8):
    token 0 is a prompt token (mask 0); tokens 1..4 carry log ratios a, b, c, 0
    (old = 0), so the masked sum is exactly 4x and the mean exactly x, the
    preimage of the target ratio."""
    targets = []
    for bnd in (lo, hi):
        targets += [float(np.nextafter(bnd, -np.inf)), float(bnd), float(np.nextafter(bnd, np.inf))]
    rows_lp, rows_old, rows_m = [], [], []
    for t in targets:
        x = x_on_exp(t)
        a, b, c = fp32_split(4.0 * x)
        rows_lp.append([-3.0, a, b, c, 0.0])
        rows_old.append([-1.0, 0.0, 0.0, 0.0, 0.0])
        rows_m.append([0, 1, 1, 1, 1])
    return (np.array(targets), np.array(rows_lp, np.float32), np.array(rows_old, np.float32),
            np.array(rows_m, np.uint8))
