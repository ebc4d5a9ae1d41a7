"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each pin raises AssertionError when the oracle disagrees with
  * values written out by hand or printed in a specification (tests/golden/),
  * a library routine (numpy / torch / scipy conversions, fp64 matmul, sort),
  * an exact algebraic property (identity, one-hot, linearity, symmetry).

The pins are plain functions so that the mutation tests can run the same set
against copies of the oracle with a planted mistake and require that every
planted mistake trips at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np

import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ helpers
def read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()
            rows.append((int(a, 16), float(b)))
    return rows


def read_kv(name):
    kv = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            kv[key] = vals
    return kv


def hexbytes(vals, dtype):
    return np.array([int(v, 16) for v in vals], dtype=dtype)


def same_value(a: float, b: float) -> bool:
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def nvfp4_from_dense_codes(codes_nk: np.ndarray, scales_nb: np.ndarray, g=1.0):
    """Pack per-weight 4-bit codes [N][K] (low nibble = even k) into the ABI."""
    c = codes_nk.astype(np.uint8)
    packed = (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)
    return {"codes": packed.astype(np.uint8), "scales": scales_nb.astype(np.uint8), "g": g}


def q45_from_dense_codes(q_nk, scale_bits, min_bits, bits):
    q = q_nk.astype(np.uint8)
    lo = (q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)
    hi = None
    if bits == 5:
        hb = (q >> 4) & 1
        N, K = q.shape
        hi = np.zeros((N, K // 8), np.uint8)
        for j in range(8):
            hi |= (hb[:, j::8] << j).astype(np.uint8)
    return {"q_lo": lo.astype(np.uint8), "q_hi": hi, "scale": np.asarray(scale_bits, np.uint16),
            "min": np.asarray(min_bits, np.uint16), "bits": bits}


def bf16_bits_of(values) -> np.ndarray:
    """bf16 bit patterns of values exactly representable in bf16 (via torch)."""
    import torch
    t = torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(np.asarray(values, np.float32)))
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ element decodes
def pin_e2m1_table():
    rows = read_table("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = O.e2m1(code)
        assert same_value(got, val), f"e2m1({code:#x}) = {got}, table says {val}"


def pin_e4m3_anchors():
    for code, val in read_table("e4m3_anchors.txt"):
        got = O.e4m3(code)
        assert same_value(got, val), f"e4m3({code:#x}) = {got}, table says {val}"


def pin_e4m3_library():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    ours = O.e4m3_array(codes)
    for c in range(256):
        assert same_value(ours[c], lib[c]), f"e4m3({c:#x}): oracle {ours[c]} torch {lib[c]}"


def pin_f16_library():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    lib = bits.view(np.float16).astype(np.float64)
    ours = O.f16_array(bits)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))


def pin_bf16_library():
    import torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().double().numpy()
    ours = O.bf16_array(bits)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))


def pin_round_bf16_library():
    """fp64 -> bf16 RNE agrees with torch's fp32 -> bf16 RNE on fp32 inputs
    (those are exact in fp64, so there is no double rounding on either side)."""
    import torch
    r = _rng(7)
    with np.errstate(over="ignore"):
        parts = [
            r.standard_normal(50000).astype(np.float32),
            (r.standard_normal(20000) * 2.0 ** r.integers(-140, 128, 20000)).astype(np.float32),
            np.float32(3.3895314e38) * r.uniform(0.99, 1.0, 2000).astype(np.float32),
        ]
    # exact ties: bf16 value + half a bf16 ulp (ties to even), odd and even
    base = r.integers(0x0080, 0x7F00, 5000).astype(np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    parts.append(ties)
    parts.append(-ties)
    v = np.concatenate(parts)
    v = v[np.isfinite(v)]
    lib = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    ours = O.round_bf16(v.astype(np.float64))
    assert np.array_equal(ours, lib), "round_bf16 differs from torch RNE"
    bits_lib = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_bits(v.astype(np.float64)), bits_lib)


def pin_round_bf16_ties_by_hand():
    # 1 + 2^-8 lies halfway between 1 (mantissa 0, even) and 1 + 2^-7: -> 1.
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6: -> 1 + 2^-6.
    cases = [(1 + 2.0 ** -8, 1.0), (1 + 3 * 2.0 ** -8, 1 + 2.0 ** -6),
             (-(1 + 2.0 ** -8), -1.0), (1 + 2.0 ** -8 + 2.0 ** -40, 1 + 2.0 ** -7),
             (3 * 2.0 ** -134, 2 * 2.0 ** -133), (2.0 ** -134, 0.0), (2.0 ** 128, math.inf)]
    for v, want in cases:
        got = O.round_bf16(np.array([v]))[0]
        assert got == want, f"round_bf16({v!r}) = {got!r}, want {want!r}"


# ------------------------------------------------------------------ GEMV, hand cases
def pin_hand_nvfp4():
    kv = read_kv("hand_nvfp4_4x16.txt")
    x = hexbytes(kv["x"], np.uint16)[None, :]
    codes = np.stack([hexbytes(kv[f"codes{i}"], np.uint8) for i in range(4)])
    w = {"codes": codes, "scales": hexbytes(kv["scales"], np.uint8)[:, None], "g": 1.0}
    y, _ = O.gemv_nvfp4(w, x)
    assert np.array_equal(y[0], np.array([float(v) for v in kv["y"]])), y
    r = hexbytes(kv["residual"], np.uint16)[None, :]
    y2, _ = O.gemv_nvfp4(w, x, residual=r)
    assert np.array_equal(y2[0], np.array([float(v) for v in kv["y_res"]])), y2
    w2 = dict(w, g=2.0)
    y3, _ = O.gemv_nvfp4(w2, x)
    assert np.array_equal(y3[0], 2.0 * np.array([float(v) for v in kv["y"]]))


def pin_hand_q45():
    kv = read_kv("hand_q45_4x32.txt")
    x = hexbytes(kv["x"], np.uint16)[None, :]
    w4 = {"q_lo": np.stack([hexbytes(kv[f"q4_lo{i}"], np.uint8) for i in range(2)]),
          "q_hi": None, "bits": 4,
          "scale": hexbytes(kv["q4_scale"], np.uint16)[:, None],
          "min": hexbytes(kv["q4_min"], np.uint16)[:, None]}
    y, _ = O.gemv_q45(w4, x)
    assert np.array_equal(y[0], np.array([float(v) for v in kv["q4_y"]])), y
    w5 = {"q_lo": np.stack([hexbytes(kv[f"q5_lo{i}"], np.uint8) for i in range(4)]),
          "q_hi": np.stack([hexbytes(kv[f"q5_hi{i}"], np.uint8) for i in range(4)]), "bits": 5,
          "scale": hexbytes(kv["q5_scale"], np.uint16)[:, None],
          "min": hexbytes(kv["q5_min"], np.uint16)[:, None]}
    y, _ = O.gemv_q45(w5, x)
    assert np.array_equal(y[0], np.array([float(v) for v in kv["q5_y"]])), y


# ------------------------------------------------------------------ identity / one-hot
def _x_distinct(M, K, seed):
    """bf16 values with distinct magnitudes so a wrong index cannot match."""
    r = _rng(seed)
    mant = r.integers(1, 128, size=(M, K))
    ex = r.integers(-3, 4, size=(M, K))
    sign = r.choice([-1.0, 1.0], size=(M, K))
    vals = sign * (1 + mant / 128.0) * 2.0 ** ex
    return bf16_bits_of(vals.astype(np.float32)), vals


def pin_identity_nvfp4():
    N = K = 512
    c = np.zeros((N, K), np.uint8)
    c[np.arange(N), np.arange(K)] = 0x2                # E2M1 1.0
    w = nvfp4_from_dense_codes(c, np.full((N, K // 16), 0x38, np.uint8))
    xb, xv = _x_distinct(2, K, 11)
    y, _ = O.gemv_nvfp4(w, xb)
    assert np.array_equal(y, xv), "identity NVFP4 GEMV does not reproduce x"


def pin_identity_q45():
    N = K = 256
    xb, xv = _x_distinct(2, K, 12)
    one, zero, sixteenth = 0x3C00, 0x0000, 0x2C00      # fp16 1.0, 0, 1/16
    q = np.zeros((N, K), np.uint8)
    q[np.arange(N), np.arange(K)] = 1
    w4 = q45_from_dense_codes(q, np.full((N, K // 32), one), np.full((N, K // 32), zero), 4)
    y, _ = O.gemv_q45(w4, xb)
    assert np.array_equal(y, xv), "identity Q4"
    q5 = np.zeros((N, K), np.uint8)
    q5[np.arange(N), np.arange(K)] = 16                # only the high bit plane
    w5 = q45_from_dense_codes(q5, np.full((N, K // 32), sixteenth), np.full((N, K // 32), zero), 5)
    y, _ = O.gemv_q45(w5, xb)
    assert np.array_equal(y, xv), "identity Q5 (high plane)"


def pin_one_hot_nvfp4():
    N, K = 3, 64
    xb, xv = _x_distinct(1, K, 13)
    scale_codes = np.array([0x30, 0x38, 0x3F, 0x44], np.uint8)   # 0.5, 1, 1.875, 3
    sval = [O.e4m3(s) for s in scale_codes]
    table = {c: v for c, v in read_table("e2m1_values.txt")}
    for kstar in range(K):
        for code in range(16):
            c = np.zeros((N, K), np.uint8)
            c[1, kstar] = code
            sc = np.tile(scale_codes, (N, 1))
            w = nvfp4_from_dense_codes(c, sc)
            y, _ = O.gemv_nvfp4(w, xb)
            want = table[code] * sval[kstar // 16] * xv[0, kstar]
            assert y[0, 1] == want, f"one-hot k*={kstar} code={code:#x}: {y[0, 1]} != {want}"
            assert y[0, 0] == 0 and y[0, 2] == 0


def pin_one_hot_q45():
    N, K = 2, 64
    xb, xv = _x_distinct(1, K, 14)
    sc_bits = np.array([[0x3C00, 0x4000], [0x3C00, 0x4000]], np.uint16)   # 1, 2 per group
    zero = np.zeros((N, K // 32), np.uint16)
    for bits in (4, 5):
        for kstar in range(K):
            for qv in (1, 7, 15, 16, 31) if bits == 5 else (1, 7, 15):
                q = np.zeros((N, K), np.uint8)
                q[0, kstar] = qv
                w = q45_from_dense_codes(q, sc_bits, zero, bits)
                y, _ = O.gemv_q45(w, xb)
                want = (1.0 if kstar < 32 else 2.0) * qv * xv[0, kstar]
                assert y[0, 0] == want, f"Q{bits} one-hot k*={kstar} q={qv}"
                assert y[0, 1] == 0
    # min alone: q = 0 everywhere, min = 0.5 in group 1 of row 0 only
    q = np.zeros((N, K), np.uint8)
    mn = zero.copy()
    mn[0, 1] = 0x3800
    w = q45_from_dense_codes(q, sc_bits, mn, 4)
    y, _ = O.gemv_q45(w, xb)
    assert y[0, 0] == 0.5 * xv[0, 32:].sum() and y[0, 1] == 0


# ------------------------------------------------------------------ library / invariants
def _rand_nvfp4(N, K, seed, g=1.0):
    r = _rng(seed)
    return {"codes": r.integers(0, 256, (N, K // 2), dtype=np.uint8),
            "scales": r.integers(0x10, 0x50, (N, K // 16), dtype=np.uint8), "g": g}


def _rand_q45(N, K, bits, seed):
    r = _rng(seed)
    return {"q_lo": r.integers(0, 256, (N, K // 2), dtype=np.uint8),
            "q_hi": r.integers(0, 256, (N, K // 8), dtype=np.uint8) if bits == 5 else None,
            "scale": np.asarray(r.uniform(0.002, 0.02, (N, K // 32)), np.float16).view(np.uint16),
            "min": np.asarray(r.normal(0, 0.05, (N, K // 32)), np.float16).view(np.uint16),
            "bits": bits}


def _rand_x(M, K, seed):
    import torch
    r = _rng(seed)
    return torch.from_numpy(r.standard_normal((M, K)).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def pin_library_matmul():
    """GEMV == fp64 matmul (numpy) of the decoded W and x, to summation order."""
    import torch
    x = _rand_x(3, 512, 21)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    for w, deq, gemv in (
        (_rand_nvfp4(64, 512, 22), O.dequant_nvfp4, O.gemv_nvfp4),
        (_rand_q45(64, 512, 4, 23), O.dequant_q45, O.gemv_q45),
        (_rand_q45(64, 512, 5, 24), O.dequant_q45, O.gemv_q45),
    ):
        W = deq(w)
        y, a = gemv(w, x)
        ref = xv @ W.T
        aref = np.abs(xv) @ np.abs(W).T
        assert np.all(np.abs(y - ref) <= 1e-12 * aref + 1e-300), "GEMV vs numpy matmul"
        assert np.allclose(a, aref, rtol=1e-12, atol=0)


def pin_linearity_and_symmetry():
    w = _rand_nvfp4(32, 256, 31)
    x = _rand_x(2, 256, 32)
    y, _ = O.gemv_nvfp4(w, x)
    # x -> 2x: add one to the bf16 exponent field of every nonzero normal value
    e = (x >> 7) & 0xFF
    assert np.all((e > 0) & (e < 0xFE))
    y2, _ = O.gemv_nvfp4(w, (x + 0x80).astype(np.uint16))
    assert np.array_equal(y2, 2 * y), "linearity in x"
    # flipping the E2M1 sign bit of every code negates y exactly
    wn = dict(w, codes=(w["codes"] ^ 0x88).astype(np.uint8))
    yn, _ = O.gemv_nvfp4(wn, x)
    assert np.array_equal(yn, -y), "sign symmetry"
    # g -> 2g doubles y
    yg, _ = O.gemv_nvfp4(dict(w, g=2.0), x)
    assert np.array_equal(yg, 2 * y), "global scale"


def pin_row_independence():
    for w, gemv in ((_rand_nvfp4(16, 256, 41), O.gemv_nvfp4), (_rand_q45(16, 256, 5, 42), O.gemv_q45)):
        x = _rand_x(4, 256, 43)
        y, _ = gemv(w, x)
        for m in range(4):
            ym, _ = gemv(w, x[m:m + 1])
            assert np.array_equal(ym[0], y[m]), "batch row differs from single-row call"


def pin_q_integer_gemv():
    r = _rng(51)
    N, K = 8, 128
    for bits in (4, 5):
        q = r.integers(0, 2 ** bits, (N, K)).astype(np.uint8)
        w = q45_from_dense_codes(q, np.full((N, K // 32), 0x3C00), np.zeros((N, K // 32)), bits)
        xi = r.integers(-8, 9, (2, K))
        y, _ = O.gemv_q45(w, bf16_bits_of(xi.astype(np.float32)))
        assert np.array_equal(y, (xi @ q.astype(np.int64).T).astype(np.float64)), f"Q{bits} integer"


# ------------------------------------------------------------------ epilogues / MoE
def pin_silu_library():
    from scipy.special import expit
    v = np.concatenate([np.linspace(-40, 40, 2001), [-745.0, -100.0, 0.0, 1e-300, 100.0]])
    for t in v:
        got = O.silu(t)
        want = t * expit(t)
        assert abs(got - want) <= 4e-16 * abs(want) + 1e-300, (t, got, want)
    g = np.linspace(-9, 9, 37)
    u = np.linspace(3, -3, 37)
    assert np.allclose(O.swiglu(g, u), g * expit(g) * u, rtol=1e-15, atol=0)


def pin_route_bruteforce():
    from scipy.special import softmax
    r = _rng(61)
    for M, E, k in ((8, 128, 8), (3, 16, 4), (2, 8, 8)):
        lg = r.standard_normal((M, E)).astype(np.float32)
        lg[0, 3] = lg[0, 5]                     # a tie: lower id must come first
        ids, w = O.route_topk(lg, k)
        p = softmax(lg.astype(np.float64), axis=1)
        for m in range(M):
            order = np.lexsort((np.arange(E), -p[m]))[:k]
            assert np.array_equal(ids[m], order), (m, ids[m], order)
            assert abs(w[m].sum() - 1.0) <= 1e-15
            assert np.allclose(w[m], p[m, order] / p[m, order].sum(), rtol=1e-14, atol=0)


def _moe_case(seed, E=4, H=64, I=32, M=2, topk=2):
    r = _rng(seed)
    gu = {"codes": r.integers(0, 256, (E, 2 * I, H // 2), dtype=np.uint8),
          "scales": r.integers(0x28, 0x40, (E, 2 * I, H // 16), dtype=np.uint8),
          "g": r.uniform(0.5, 2, E)}
    dn = {"codes": r.integers(0, 256, (E, H, I // 2), dtype=np.uint8),
          "scales": r.integers(0x28, 0x40, (E, H, I // 16), dtype=np.uint8),
          "g": r.uniform(0.5, 2, E)}
    x = _rand_x(M, H, seed + 1)
    return gu, dn, x


def pin_moe_reduces_to_dense():
    gu, dn, x = _moe_case(71)
    E, H, I = 4, 64, 32
    ids = np.array([[2, 0], [1, 3]], np.int32)
    w = np.array([[1.0, 0.0], [1.0, 0.0]])
    gate, up, ag, au, h = O.moe_gate_up(gu, x, ids)
    for m in range(2):
        e = ids[m, 0]
        we = {"codes": gu["codes"][e], "scales": gu["scales"][e], "g": gu["g"][e]}
        ye, _ = O.gemv_nvfp4(we, x[m:m + 1])
        assert np.array_equal(gate[m, 0], ye[0, :I]) and np.array_equal(up[m, 0], ye[0, I:])
        assert np.array_equal(O.bf16_bits(O.swiglu(ye[0, :I], ye[0, I:])), h[m, 0])
    hv = O.bf16_array(h)
    y = O.moe_down(dn, hv, ids, w)
    for m in range(2):
        e = ids[m, 0]
        wd = {"codes": dn["codes"][e], "scales": dn["scales"][e], "g": dn["g"][e]}
        yd, _ = O.gemv_nvfp4(wd, h[m, 0][None, :])
        assert np.array_equal(y[m], yd[0]), "MoE with one-hot routing weights != dense down"


def pin_moe_slot_permutation():
    gu, dn, x = _moe_case(81, E=6, M=2, topk=3)
    ids = np.array([[5, 1, 2], [0, 4, 2]], np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.25, 0.6, 0.15]])
    _, _, _, _, h = O.moe_gate_up(gu, x, ids)
    y = O.moe_down(dn, O.bf16_array(h), ids, w)
    a = O.moe_down(dn, np.abs(O.bf16_array(h)), ids, w, use_abs=True)
    perm = [2, 0, 1]
    _, _, _, _, hp = O.moe_gate_up(gu, x, ids[:, perm])
    assert np.array_equal(hp, h[:, perm])
    yp = O.moe_down(dn, O.bf16_array(hp), ids[:, perm], w[:, perm])
    assert np.all(np.abs(yp - y) <= 1e-12 * a), "slot order changed the MoE result"
    # linear in the routing weights
    y2 = O.moe_down(dn, O.bf16_array(h), ids, 2 * w)
    assert np.array_equal(y2, 2 * y)


# ------------------------------------------------------------------ RMSNorm
def pin_rmsnorm_hand():
    """Two hand-worked cases (tests/golden/hand_rmsnorm.txt): mean of squares,
    eps inside the root, gamma per element, bf16 rounding of the result."""
    kv = read_kv("hand_rmsnorm.txt")
    gamma = hexbytes(kv["gamma"], np.uint16)
    for case in ("a", "b"):
        x = hexbytes(kv["x" + case], np.uint16)[None, :]
        h, v, r = O.rmsnorm(x, gamma, float(kv["eps" + case][0]))
        assert r[0] == float(kv["r" + case][0]), (case, r[0])
        assert np.array_equal(h[0], hexbytes(kv["h" + case], np.uint16)), (case, [hex(a) for a in h[0]])


def pin_rmsnorm_invariants():
    """Exact properties: a constant row normalises to +-1 (eps = 0); scaling x
    by 2^j leaves h unchanged (eps = 0); doubling gamma doubles h exactly; a
    zero row gives zeros; rows are independent."""
    r = _rng(31)
    K = 96
    g1 = bf16_bits_of(np.ones(K))
    for c in (0.75, -3.0, 2.0 ** -20):
        x = bf16_bits_of(np.full((1, K), c))
        h, v, rr = O.rmsnorm(x, g1, 0.0)
        assert np.array_equal(O.bf16_array(h), np.full((1, K), math.copysign(1.0, c))), c
    # values with at most 8 significant bits (exact in bf16)
    x = bf16_bits_of(np.round(r.standard_normal((3, K)) * 64.0) / 64.0)
    gamma = bf16_bits_of(np.round(r.uniform(0.5, 1.5, K) * 128.0) / 128.0)
    h, v, rr = O.rmsnorm(x, gamma, 0.0)
    for j in (-7, 5):
        xs = bf16_bits_of(O.bf16_array(x) * 2.0 ** j)
        hs, vs, _ = O.rmsnorm(xs, gamma, 0.0)
        assert np.array_equal(hs, h) and np.array_equal(vs, v), j
    h2, v2, _ = O.rmsnorm(x, bf16_bits_of(O.bf16_array(gamma) * 2.0), 0.0)
    assert np.array_equal(O.bf16_array(h2), 2.0 * O.bf16_array(h))
    hz, vz, rz = O.rmsnorm(np.zeros((1, K), np.uint16), gamma, 1e-6)
    assert np.all(O.bf16_array(hz) == 0.0) and rz[0] == 1.0 / math.sqrt(1e-6)
    for m in range(3):
        hm, vm, _ = O.rmsnorm(x[m:m + 1], gamma, 0.25)
        ha, va, _ = O.rmsnorm(x, gamma, 0.25)
        assert np.array_equal(hm[0], ha[m]) and np.array_equal(vm[0], va[m])


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
