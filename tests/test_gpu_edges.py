"""The formats' edge values through every hot kernel, against the fp64 oracle (GPU).

Each case runs on the kernel the shape selects: one token on the CUDA-core
kernels (NVFP4 and Q4/Q5), 2..8 NVFP4 tokens on the tcgen05 kernel, 2..8
Q4/Q5 tokens on the groupwise-int tensor-core kernel, the MoE on the grouped
kernels, and K not a multiple of 256 on the exact fallback kernel.

* NVFP4 block scales: every finite E4M3 code -- 448 (0x7E), the subnormals
  0x01..0x07, zero and the negative codes -- with tensor scales g of 2^-20,
  3.0e-5, 1 and 1e4.
* Q4/Q5: fp16 scales and mins drawn from the whole finite range (zeros and
  subnormals included) and groups whose min cancels scale * mean(q).
* One-hot matrices: one nonzero weight per row, at every k mod 256 with every
  code value; the exact product is representable in fp32, so each hot decode
  must reproduce it bit for bit (fp32 out) or round it once (bf16 out).

The formats and the exact decode follow the NVIDIA NVFP4 blog ("How NVFP4
works": E2M1 values, E4M3 scale per 16, FP32 tensor scale) and the NInfer
article, section 2 (groupwise-int recipe w = scale * q + min).
"""
import numpy as np
import pytest

import oracle as O
import synth
from checks import (check_bf16, check_f32, gemv_bound, q_chain, q_split_ratio, same_f32_bits,
                    swiglu_bound)
from gpu_util import bits16, nvfp4_dev, q45_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("bit_quantized_weight_gb300")

FINITE_E4M3 = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)   # 254 codes


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    q.qg_debug_set_wait(0, False)
    yield
    assert q.qg_last_device_status() == q.QG_OK


def check_out(y, yref, a, what):
    B = gemv_bound(a)
    if y.dtype == torch.float32:
        return check_f32(y.cpu().numpy(), yref, B, what)
    return check_bf16(bits16(y), yref, B, what)


def edge_nvfp4(seed, N, K, g):
    """Random codes; block scales cycle through every finite E4M3 code so that
    each code sits in many rows and at every block position."""
    w = synth.nvfp4_weights(seed, f"edge{N}.{K}", N, K, g=g)
    nb = K // 16
    idx = (np.arange(N)[:, None] * 37 + np.arange(nb)[None, :]) % FINITE_E4M3.size
    w["scales"] = FINITE_E4M3[idx]
    return w


G_VALUES = [2.0 ** -20, 3.0e-5, 1.0, 1.0e4]


# ---------------------------------------------------------------- NVFP4 scales
@pytest.mark.parametrize("g", G_VALUES)
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_nvfp4_every_e4m3_scale(M, g):
    N, K = 600, 2048
    w = edge_nvfp4(40, N, K, g)
    x = synth.bf16_normal(41, f"edgex{M}", (M, K))
    yref, a = O.gemv_nvfp4(w, x)
    d = nvfp4_dev(w)
    xd = to_dev(x)
    for dt in (torch.float32, torch.bfloat16):
        y = torch.empty((M, N), dtype=dt, device="cuda")
        q.qgemv_nvfp4(d["codes"], d["scales"], w["g"], xd, y)
        torch.cuda.synchronize()
        check_out(y, yref, a, f"edge scales M={M} g={g} {dt}")


@pytest.mark.parametrize("g", [2.0 ** -20, 1.0e4])
@pytest.mark.parametrize("M", [1, 8])
def test_nvfp4_edge_scales_residual_and_swiglu(M, g):
    N, K = 512, 1536
    w = edge_nvfp4(42, N, K, g)
    x = synth.bf16_normal(43, f"edgerx{M}", (M, K))
    r = synth.bf16_normal(44, f"edger{M}", (M, N))
    d = nvfp4_dev(w)
    xd = to_dev(x)
    yref, a = O.gemv_nvfp4(w, x, residual=r)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    q.qgemv_nvfp4(d["codes"], d["scales"], w["g"], xd, y, residual=to_dev(r))
    torch.cuda.synchronize()
    check_out(y, yref, a, f"edge residual M={M} g={g}")
    yref, a = O.gemv_nvfp4(w, x)
    I = N // 2
    href = O.swiglu(yref[:, :I], yref[:, I:])
    B = swiglu_bound(yref[:, :I], yref[:, I:], gemv_bound(a[:, :I]), gemv_bound(a[:, I:]))
    h = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    q.qgemv_swiglu_nvfp4(d["codes"], d["scales"], w["g"], xd, h)
    torch.cuda.synchronize()
    check_bf16(bits16(h), href, B, f"edge swiglu M={M} g={g}")


def test_nvfp4_edge_scales_fallback_kernel():
    """K not a multiple of 256: the exact warp-per-row kernel."""
    M, N, K = 3, 300, 800
    w = edge_nvfp4(45, N, K, 1.0e4)
    x = synth.bf16_normal(46, "edgefx", (M, K))
    yref, a = O.gemv_nvfp4(w, x)
    d = nvfp4_dev(w)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    q.qgemv_nvfp4(d["codes"], d["scales"], w["g"], to_dev(x), y)
    torch.cuda.synchronize()
    check_out(y, yref, a, "edge scales fallback")


# ---------------------------------------------------------------- one-hot, NVFP4
def one_hot_nvfp4(K):
    """N = 8192 rows: row n holds its single nonzero code at k = n % 256 of
    chunk n // 4096 with code (n // 256) % 16 (codes 0 and 8 are +-0), so every
    (k mod 256, code) pair appears in both chunks. Each row's block scale is a
    finite E4M3 code (cycled), the other blocks' scales are random."""
    N = 8192
    w = synth.nvfp4_weights(47, f"onehot{K}", N, K)
    n = np.arange(N)
    k = n % 256 + 256 * (n // 4096)
    code = (n // 256) % 16
    codes = np.zeros((N, K // 2), np.uint8)
    codes[n, k // 2] = np.where(k % 2 == 0, code, code << 4).astype(np.uint8)
    w["codes"] = codes
    scales = w["scales"].copy()
    scales[n, k // 16] = FINITE_E4M3[(n * 7) % FINITE_E4M3.size]
    w["scales"] = scales
    return w


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_nvfp4_one_hot_bit_exact(M):
    K = 512
    w = one_hot_nvfp4(K)
    x = synth.bf16_normal(48, f"onehotx{M}", (M, K))
    yref, _ = O.gemv_nvfp4(w, x)           # one exact product per element
    assert np.array_equal(yref, yref.astype(np.float32).astype(np.float64)), "reference not exact in fp32"
    d = nvfp4_dev(w)
    xd = to_dev(x)
    y32 = torch.empty((M, w["codes"].shape[0]), dtype=torch.float32, device="cuda")
    y16 = torch.empty_like(y32, dtype=torch.bfloat16)
    q.qgemv_nvfp4(d["codes"], d["scales"], 1.0, xd, y32)
    q.qgemv_nvfp4(d["codes"], d["scales"], 1.0, xd, y16)
    torch.cuda.synchronize()
    assert same_f32_bits(y32.cpu().numpy(), yref.astype(np.float32)), "fp32 one-hot not bit-exact"
    want16 = O.bf16_bits(yref)
    got16 = bits16(y16)
    eq = (got16 == want16) | (((got16 & 0x7FFF) == 0) & ((want16 & 0x7FFF) == 0))
    assert eq.all(), f"bf16 one-hot: {int((~eq).sum())} elements differ"


# ---------------------------------------------------------------- one-hot, Q4/Q5
def one_hot_q45(bits, K):
    """Row n: single nonzero code q = 1 + (n // 256) % (2^bits - 1) at
    k = n % 256 of chunk (n // 256) % 2 (every k mod 256 with every nonzero
    code value); min = 0 everywhere; fp16 scales from the whole finite range.
    scale * q * x has at most 11 + 5 + 8 bits, so it is exact in fp32."""
    nq = (1 << bits) - 1
    N = 256 * nq * 2
    w = synth.q45_weights(49, f"qonehot{bits}", N, K, bits)
    n = np.arange(N)
    blk = n // 256
    k = n % 256 + 256 * (blk % 2)
    qv = 1 + (blk // 2) % nq
    q_lo = np.zeros((N, K // 2), np.uint8)
    lo = (qv & 0xF).astype(np.uint8)
    q_lo[n, k // 2] = np.where(k % 2 == 0, lo, lo << 4)
    w["q_lo"] = q_lo
    if bits == 5:
        q_hi = np.zeros((N, K // 8), np.uint8)
        q_hi[n, k // 8] = ((qv >> 4) << (k % 8)).astype(np.uint8)
        w["q_hi"] = q_hi
    r = np.random.default_rng(50)
    sc = (r.integers(0, 0x7C00, size=w["scale"].shape) | (r.integers(0, 2, size=w["scale"].shape) << 15))
    w["scale"] = sc.astype(np.uint16)
    w["min"] = np.zeros_like(w["min"])
    return w


@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_q45_one_hot_bit_exact(bits, M):
    K = 512
    w = one_hot_q45(bits, K)
    x = synth.bf16_normal(51, f"qonehotx{M}", (M, K))
    yref, _ = O.gemv_q45(w, x)
    assert np.array_equal(yref, yref.astype(np.float32).astype(np.float64)), "reference not exact in fp32"
    d = q45_dev(w)
    xd = to_dev(x)
    N = w["q_lo"].shape[0]
    y32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y16 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, xd, y32)
    q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, xd, y16)
    torch.cuda.synchronize()
    assert same_f32_bits(y32.cpu().numpy(), yref.astype(np.float32)), f"Q{bits} fp32 one-hot not bit-exact"
    want16 = O.bf16_bits(yref)
    got16 = bits16(y16)
    eq = (got16 == want16) | (((got16 & 0x7FFF) == 0) & ((want16 & 0x7FFF) == 0))
    assert eq.all(), f"Q{bits} bf16 one-hot: {int((~eq).sum())} elements differ"


# ---------------------------------------------------------------- Q4/Q5 scales and mins
def full_range_f16(r, shape):
    """fp16 bit patterns uniform over every finite value (zeros, subnormals,
    both signs, up to 65504)."""
    return (r.integers(0, 0x7C00, size=shape) | (r.integers(0, 2, size=shape) << 15)).astype(np.uint16)


def q_codes(w):
    lo = w["q_lo"]
    qq = np.empty((lo.shape[0], lo.shape[1] * 2), np.int64)
    qq[:, 0::2] = lo & 0xF
    qq[:, 1::2] = lo >> 4
    if w.get("q_hi") is not None:
        qq += 16 * np.unpackbits(w["q_hi"], axis=1, bitorder="little").astype(np.int64)
    return qq


def edge_q45(seed, bits, N, K, mode):
    """mode 'full': scale and min bit patterns over the whole finite fp16
    range; 'cancel': typical scales with min = -scale * mean(q) of the group
    (rounded to fp16) in every other group."""
    w = synth.q45_weights(seed, f"qedge{bits}.{mode}", N, K, bits)
    r = np.random.default_rng(seed)
    if mode == "full":
        w["scale"] = full_range_f16(r, w["scale"].shape)
        w["min"] = full_range_f16(r, w["min"].shape)
    else:
        qq = q_codes(w).reshape(N, K // 32, 32).mean(axis=2)
        s = O.f16_array(w["scale"])
        mn = (-s * qq).astype(np.float16).view(np.uint16)
        sel = (np.arange(K // 32)[None, :] + np.arange(N)[:, None]) % 2 == 0
        w["min"] = np.where(sel, mn, w["min"]).astype(np.uint16)
    return w


@pytest.mark.parametrize("mode", ["full", "cancel"])
@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_q45_edge_scales_and_mins(M, bits, mode, record_property):
    N, K = 520, 2048
    w = edge_q45(52 + bits, bits, N, K, mode)
    x = synth.bf16_normal(53, f"qedgex{M}", (M, K))
    yref, a = O.gemv_q45(w, x)
    B = gemv_bound(a)
    prior = q_split_ratio(w, x, B, q_chain(K))
    d = q45_dev(w)
    xd = to_dev(x)
    observed = None
    for dt in (torch.float32, torch.bfloat16):
        y = torch.empty((M, N), dtype=dt, device="cuda")
        q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, xd, y)
        torch.cuda.synchronize()
        r = check_out(y, yref, a, f"Q{bits} {mode} M={M} {dt}")   # raises outside the bound
        if dt == torch.float32:
            observed = r              # |y - y_ref| / B of the unrounded output
    record_property("q_split_prior_ratio", prior)
    record_property("observed_ratio", observed)
    print(f"Q{bits} {mode} M={M}: a-priori split bound / B = {prior:.3g}, observed fp32 error / B = {observed:.3g}")
    assert observed <= 1.0 and prior <= 1.0


@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("M", [1, 8])
def test_q45_edge_residual(M, bits):
    N, K = 384, 1024
    w = edge_q45(56 + bits, bits, N, K, "full")
    x = synth.bf16_normal(57, f"qedgerx{M}", (M, K))
    r = synth.bf16_normal(58, f"qedger{M}", (M, N))
    yref, a = O.gemv_q45(w, x, residual=r)
    d = q45_dev(w)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, to_dev(x), y, residual=to_dev(r))
    torch.cuda.synchronize()
    check_out(y, yref, a, f"Q{bits} edge residual M={M}")


@pytest.mark.parametrize("M", [1, 8])
def test_q45_config_data_split_ratio(M, record_property):
    """On the mixed recipe's own data (config shapes) the a-priori error bound
    of the scale * sum(q x) + min * sum(x) split stays below the stated
    bound, so the split needs no fallback there; reported per projection."""
    worst = 0.0
    for name, N, K, bits in synth.Q45_RECIPE:
        rows = slice(0, 512)
        w = synth.q45_weights(3, f"q45.{name}", N, K, bits)
        ws = {"q_lo": w["q_lo"][rows], "q_hi": None if w["q_hi"] is None else w["q_hi"][rows],
              "scale": w["scale"][rows], "min": w["min"][rows], "bits": bits}
        x = synth.bf16_normal(3, f"q45.{name}.x", (8, K))[:M]
        yref, a = O.gemv_q45(ws, x)
        r = q_split_ratio(ws, x, gemv_bound(a), q_chain(K))
        print(f"Q{bits} {name} M={M}: a-priori split bound / B = {r:.3g}")
        worst = max(worst, r)
    record_property("q_split_prior_ratio", worst)
    assert worst <= 1.0


# ---------------------------------------------------------------- MoE
def test_moe_edge_scales_and_expert_scales():
    """Expert weights with every finite E4M3 block scale and per-expert
    tensor scales of 2^-20, 3.0e-5, 1 and 1e4 through the grouped kernels."""
    from test_gpu_moe import check_moe, run_moe
    M, E, H, I, topk = 8, 12, 512, 768, 4
    gu = synth.nvfp4_weights(59, "moeedge.gu", E * 2 * I, H)
    dn = synth.nvfp4_weights(59, "moeedge.dn", E * H, I)
    for w in (gu, dn):
        n, nb = w["scales"].shape
        w["scales"] = FINITE_E4M3[(np.arange(n)[:, None] * 37 + np.arange(nb)[None, :]) % FINITE_E4M3.size]
    gvals = np.array(G_VALUES, np.float32).astype(np.float64)
    gu_h = {"codes": gu["codes"].reshape(E, 2 * I, H // 2), "scales": gu["scales"].reshape(E, 2 * I, H // 16),
            "g": gvals[np.arange(E) % 4]}
    dn_h = {"codes": dn["codes"].reshape(E, H, I // 2), "scales": dn["scales"].reshape(E, H, I // 16),
            "g": gvals[(np.arange(E) + 1) % 4]}
    x = synth.bf16_normal(60, "moeedge.x", (M, H))
    r = np.random.default_rng(61)
    ids = np.stack([r.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    w = r.uniform(0.05, 1.0, (M, topk)).astype(np.float32).astype(np.float64)
    y, h = run_moe(gu_h, dn_h, x, ids, w)
    check_moe(gu_h, dn_h, x, ids, w, y, h)
