"""Acceptance checks: GPU outputs against the fp64 oracle.

The bound for a GEMV output element is B = 1e-4 * sum_k |w x| + 1e-6 (the
library's stated tolerance). An fp32 output must lie within B of the exact
sum; a bf16 output must equal the round-to-nearest-even of some value within
B of it, i.e. lie in [rne(y - B), rne(y + B)] (rne is monotone).

SwiGLU (a reading; only the GEMV bound is stated): with gate/up exact values
a, b and GEMV bounds Ba, Bb, the computed silu(a') * b' differs from
silu(a) * b by at most
    L*Ba*(|b| + Bb) + |silu(a)|*Bb          (L = 1.1 >= sup |silu'|)
plus the fp32 evaluation of silu and the product, bounded by 2^-20 relative,
plus 1e-6.
"""
from __future__ import annotations

import numpy as np

import oracle as O

SILU_LIPSCHITZ = 1.1  # sup |d/dv v*sigmoid(v)| = 1.0998...


def gemv_bound(absacc):
    return 1e-4 * np.asarray(absacc, np.float64) + 1e-6


def swiglu_bound(a, b, Ba, Bb):
    sa = O.swiglu(a, np.ones_like(a))           # silu(a) from the oracle
    core = SILU_LIPSCHITZ * Ba * (np.abs(b) + Bb) + np.abs(sa) * Bb
    return core + 2.0 ** -20 * (np.abs(sa * b) + core) + 1e-6


def _fail(what, bad, y, yref, B):
    idx = np.argwhere(bad)[:5]
    lines = [f"{what}: {int(bad.sum())} of {bad.size} elements outside the bound"]
    for i in idx:
        t = tuple(i)
        lines.append(f"  at {t}: got {y[t]!r} ref {yref[t]!r} bound {B[t]!r}")
    raise AssertionError("\n".join(lines))


def check_f32(y, yref, B, what="fp32 output") -> float:
    y = np.asarray(y, np.float64)
    nan_ref = np.isnan(yref)
    bad = np.where(nan_ref, ~np.isnan(y), ~(np.abs(y - yref) <= B))
    if bad.any():
        _fail(what, bad, y, yref, B)
    ok = ~nan_ref & np.isfinite(yref)
    return float(np.max(np.abs(y - yref)[ok] / B[ok])) if ok.any() else 0.0


def check_bf16(y_bits, yref, B, what="bf16 output") -> float:
    y = O.bf16_array(np.asarray(y_bits, np.uint16))
    lo = O.round_bf16(yref - B)
    hi = O.round_bf16(yref + B)
    nan_ref = np.isnan(yref)
    bad = np.where(nan_ref, ~np.isnan(y), ~((y >= lo) & (y <= hi)))
    if bad.any():
        _fail(what, bad, y, yref, B)
    ok = ~nan_ref & np.isfinite(yref)
    return float(np.max(np.abs(y - yref)[ok] / B[ok])) if ok.any() else 0.0


def same_f32_bits(a, b) -> bool:
    """Bitwise equality of fp32 arrays, with every NaN equal and +0 == -0."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a.view(np.uint32) == b.view(np.uint32)) | ((a == 0) & (b == 0)) | both_nan
    return bool(eq.all())
