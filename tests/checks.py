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


def q_split_ratio(w: dict, x_bits, B, chain: int):
    """A-priori error bound of the groupwise-int split, relative to B.

    The Q kernels compute each group's contribution as scale*sum(q x) +
    min*sum(x) in fp32. With d the longest sequential chain of fp32 roundings
    an output element meets (`chain`), the error is at most d * 2^-24 * T,
    T = sum_g (|scale_g| sum_{k in g} |q_k x_k| + |min_g| sum_{k in g} |x_k|),
    which can exceed the stated bound B when scale*q and min cancel inside
    the groups. Returns the largest d * 2^-24 * T / B over the outputs.
    """
    x = O.bf16_array(np.asarray(x_bits, np.uint16))          # [M][K]
    lo = np.asarray(w["q_lo"], np.uint8)
    q = np.empty((lo.shape[0], lo.shape[1] * 2), np.float64)
    q[:, 0::2] = lo & 0xF
    q[:, 1::2] = lo >> 4
    if w.get("q_hi") is not None:
        hi = np.unpackbits(np.asarray(w["q_hi"], np.uint8), axis=1, bitorder="little")
        q += 16.0 * hi
    s = np.abs(O.f16_array(w["scale"]))                     # [N][K/32]
    mn = np.abs(O.f16_array(w["min"]))
    N, K = q.shape
    G = K // 32
    ax = np.abs(x).reshape(x.shape[0], G, 32)                # [M][G][32]
    qx = np.einsum("ngk,mgk->mng", q.reshape(N, G, 32), ax)  # sum_k |q x| per group
    sx = ax.sum(axis=2)                                      # [M][G]
    T = np.einsum("ng,mng->mn", s, qx) + np.einsum("ng,mg->mn", mn, sx)
    return float(np.max(chain * 2.0 ** -24 * T / B))


def q_chain(K: int) -> int:
    """Longest fp32 rounding chain of the groupwise-int kernels for K: up to
    32 products in a group, two accumulations per group along K, and the
    cross-lane, cross-warp and phase reductions."""
    return 32 + 2 * (K // 32) + 32
