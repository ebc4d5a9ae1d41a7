"""Fused RMSNorm prologue and the mixed-width groupwise-int SwiGLU (GPU).

NInfer article, section 2: the engine fuses the normalisation with the
matmul ("one read, one write") and its groupwise-int recipe puts gate in Q5
and up in Q4. Reference: the oracle's RMSNorm (fp64 r, h = bf16(x r gamma))
followed by the oracle GEMV on h.

The kernels compute r in fp32 (sums of squares in one fixed order), so an
element of h may come out as the neighbouring bf16 value when x * r * gamma
lies within a relative distance DELTA of a rounding boundary; DELTA = 2^-16
is about four times the fp32 error of r (at most ~90 roundings of 2^-24 for
K <= 17408) and of the two products. The bound adds sum_k |w_k| * dh_k with
dh_k the larger distance from the oracle's h_k to the ends of its allowed
interval [rne(v (1 - DELTA)), rne(v (1 + DELTA))] -- zero away from a
boundary -- so a wrong r, gamma or h fails it.
"""
import numpy as np
import pytest

import oracle as O
import synth
from checks import check_bf16, check_f32, gemv_bound, swiglu_bound
from gpu_util import bits16, nvfp4_dev, q45_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("bit_quantized_weight_gb300")

DELTA = 2.0 ** -16
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    q.qg_debug_set_wait(0, False)
    yield
    assert q.qg_last_device_status() == q.QG_OK


def gamma_bits(K, seed):
    r = np.random.default_rng(seed)
    g = np.round(r.uniform(0.5, 1.5, K) * 128.0) / 128.0          # exact in bf16
    return O.bf16_bits(g)


def norm_ref(x, gamma, eps=EPS):
    """Oracle h (bf16 bits), and per element the allowed deviation of h."""
    h, v, _ = O.rmsnorm(x, gamma, eps)
    lo = O.round_bf16(v * (1.0 - DELTA))
    hi = O.round_bf16(v * (1.0 + DELTA))
    hv = O.bf16_array(h)
    dh = np.maximum(np.abs(np.maximum(lo, hi) - hv), np.abs(hv - np.minimum(lo, hi)))
    return h, dh


def widened(dense_w, a, dh):
    """GEMV bound on the oracle's h plus sum_k |w_k| dh_k (dense_w: fp64 [N][K])."""
    return gemv_bound(a) + dh @ np.abs(dense_w).T


def check_out(y, yref, B, what):
    if y.dtype == torch.float32:
        return check_f32(y.cpu().numpy(), yref, B, what)
    return check_bf16(bits16(y), yref, B, what)


def nvfp4_op(d, x, y, epi="none", residual=None, norm=None):
    op = {"codes": d["codes"], "scales": d["scales"], "g": d["g"], "x": x, "y": y, "epilogue": epi}
    if residual is not None:
        op["residual"] = residual
    if norm is not None:
        op["norm"], op["norm_eps"] = norm, EPS
    return op


def q_op(d, x, y, residual=None, norm=None, up=None):
    op = {"q_lo": d["q_lo"], "q_hi": d["q_hi"], "scale": d["scale"], "min": d["min"], "x": x, "y": y}
    if residual is not None:
        op["residual"] = residual
    if norm is not None:
        op["norm"], op["norm_eps"] = norm, EPS
    if up is not None:
        op["up"] = up
        op["epilogue"] = "swiglu"
    return op


# ---------------------------------------------------------------- RMSNorm + NVFP4
@pytest.mark.parametrize("M,N,K", [(1, 1000, 5120), (2, 777, 2048), (4, 512, 1536), (8, 640, 5120),
                                   (1, 300, 800), (3, 200, 96)])
@pytest.mark.parametrize("epi", ["none", "residual", "swiglu"])
def test_rmsnorm_nvfp4(M, N, K, epi):
    if epi == "swiglu" and N % 2:
        N += 1
    w = synth.nvfp4_weights(80, f"rn{N}.{K}", N, K, g=0.75)
    x = synth.bf16_normal(81, f"rnx{M}.{K}", (M, K))
    gamma = gamma_bits(K, 82)
    h, dh = norm_ref(x, gamma)
    W = O.dequant_nvfp4(w)
    d = nvfp4_dev(w)
    xd, gd = to_dev(x), to_dev(gamma)
    if epi == "swiglu":
        I = N // 2
        y = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
        q.qgemv_chain([nvfp4_op(d, xd, y, "swiglu", norm=gd)])
        torch.cuda.synchronize()
        yref, a = O.gemv_nvfp4(w, h)
        Bg, Bu = widened(W[:I], a[:, :I], dh), widened(W[I:], a[:, I:], dh)
        check_bf16(bits16(y), O.swiglu(yref[:, :I], yref[:, I:]),
                   swiglu_bound(yref[:, :I], yref[:, I:], Bg, Bu), f"rmsnorm swiglu M={M} K={K}")
        return
    r = synth.bf16_normal(83, f"rnr{M}", (M, N)) if epi == "residual" else None
    yref, a = O.gemv_nvfp4(w, h, residual=r)
    B = widened(W, a, dh)
    for dt in (torch.float32, torch.bfloat16):
        y = torch.empty((M, N), dtype=dt, device="cuda")
        q.qgemv_chain([nvfp4_op(d, xd, y, epi, residual=None if r is None else to_dev(r), norm=gd)])
        torch.cuda.synchronize()
        check_out(y, yref, B, f"rmsnorm nvfp4 {epi} M={M} N={N} K={K} {dt}")


def test_rmsnorm_changes_the_result():
    """The prologue is applied: without it the output differs beyond the bound."""
    M, N, K = 1, 256, 1024
    w = synth.nvfp4_weights(84, "rnc", N, K)
    x = synth.bf16_normal(85, "rncx", (M, K))
    x = O.bf16_bits(O.bf16_array(x) * 8.0)              # mean square 64: r = 1/8
    gamma = gamma_bits(K, 86)
    d = nvfp4_dev(w)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    q.qgemv_chain([nvfp4_op(d, to_dev(x), y, norm=to_dev(gamma))])
    torch.cuda.synchronize()
    plain, a = O.gemv_nvfp4(w, x)
    assert np.max(np.abs(y.cpu().numpy() - plain)) > 100 * np.max(gemv_bound(a))


# ---------------------------------------------------------------- RMSNorm + Q4/Q5
@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 5120), (2, 300, 1024), (4, 500, 17408), (8, 640, 2048), (1, 200, 800)])
def test_rmsnorm_q45(bits, M, N, K):
    w = synth.q45_weights(87, f"rnq{bits}.{N}", N, K, bits)
    x = synth.bf16_normal(88, f"rnqx{M}.{K}", (M, K))
    gamma = gamma_bits(K, 89)
    h, dh = norm_ref(x, gamma)
    W = O.dequant_q45(w)
    r = synth.bf16_normal(90, f"rnqr{M}", (M, N))
    yref, a = O.gemv_q45(w, h, residual=r)
    B = widened(W, a, dh)
    d = q45_dev(w)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    q.qgemv_chain([q_op(d, to_dev(x), y, residual=to_dev(r), norm=to_dev(gamma))])
    torch.cuda.synchronize()
    check_out(y, yref, B, f"rmsnorm Q{bits} M={M} N={N} K={K}")


# ---------------------------------------------------------------- mixed-width SwiGLU
def swiglu_q45_case(M, I, K, gbits, ubits, seed, norm):
    gw = synth.q45_weights(seed, f"sgq.gate{gbits}.{I}.{K}", I, K, gbits)
    uw = synth.q45_weights(seed, f"sgq.up{ubits}.{I}.{K}", I, K, ubits)
    x = synth.bf16_normal(seed + 1, f"sgqx{M}.{K}", (M, K))
    gamma = gamma_bits(K, seed + 2) if norm else None
    if norm:
        h, dh = norm_ref(x, gamma)
    else:
        h, dh = x, np.zeros((M, K))
    g_ref, ag = O.gemv_q45(gw, h)
    u_ref, au = O.gemv_q45(uw, h)
    Bg = widened(O.dequant_q45(gw), ag, dh)
    Bu = widened(O.dequant_q45(uw), au, dh)
    return gw, uw, x, gamma, O.swiglu(g_ref, u_ref), swiglu_bound(g_ref, u_ref, Bg, Bu)


@pytest.mark.parametrize("gbits,ubits", [(5, 4), (4, 4), (5, 5), (4, 5)])
@pytest.mark.parametrize("M", [1, 2, 3, 8])
@pytest.mark.parametrize("norm", [False, True])
def test_swiglu_q45(gbits, ubits, M, norm):
    I, K = 1000, 2048
    gw, uw, x, gamma, href, B = swiglu_q45_case(M, I, K, gbits, ubits, 91, norm)
    gd, ud = q45_dev(gw), q45_dev(uw)
    y = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    q.qgemv_swiglu_q45(gd, ud, to_dev(x), y, norm=None if gamma is None else to_dev(gamma), norm_eps=EPS)
    torch.cuda.synchronize()
    check_bf16(bits16(y), href, B, f"swiglu Q{gbits}/Q{ubits} M={M} norm={norm}")


@pytest.mark.parametrize("M", [1, 2, 8])
def test_swiglu_q45_config_shapes(M):
    """The recipe's FFN at full size: gate Q5 + up Q4, I = 17408, K = 5120,
    with the RMSNorm prologue."""
    d = synth.DENSE27B
    gw, uw, x, gamma, href, B = swiglu_q45_case(M, d.inter, d.hidden, 5, 4, 92, True)
    y = torch.empty((M, d.inter), dtype=torch.bfloat16, device="cuda")
    q.qgemv_swiglu_q45(q45_dev(gw), q45_dev(uw), to_dev(x), y, norm=to_dev(gamma), norm_eps=EPS)
    torch.cuda.synchronize()
    check_bf16(bits16(y), href, B, f"FFN Q5/Q4 M={M}")


def test_swiglu_q45_ragged_and_small():
    for (M, I, K) in [(1, 17, 256), (1, 333, 768), (3, 50, 96), (1, 40, 800)]:
        gw, uw, x, gamma, href, B = swiglu_q45_case(M, I, K, 5, 4, 93, False)
        y = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
        q.qgemv_swiglu_q45(q45_dev(gw), q45_dev(uw), to_dev(x), y)
        torch.cuda.synchronize()
        check_bf16(bits16(y), href, B, f"swiglu Q5/Q4 M={M} I={I} K={K}")


# ---------------------------------------------------------------- chain with the new ops
@pytest.mark.parametrize("M", [1, 4])
def test_chain_with_rmsnorm_matches_single_calls(M):
    """RMSNorm ops inside the persistent kernel (one token: CUDA-core stage;
    four: warp-MMA stage) give exactly what the same records give one by one."""
    K = 5120
    gamma = to_dev(gamma_bits(K, 94))
    ops, host = [], []
    for name, N, epi in [("qkv", 7168, "none"), ("gu", 2 * 4096, "swiglu")]:
        w = synth.nvfp4_weights(95, f"chn.{name}", N, K)
        x = to_dev(synth.bf16_normal(96, f"chn.{name}.x", (4, K))[:M])
        n_out = N // 2 if epi == "swiglu" else N
        d = nvfp4_dev(w)
        ops.append(nvfp4_op(d, x, torch.empty((M, n_out), dtype=torch.bfloat16, device="cuda"), epi, norm=gamma))
        host.append((d, x, n_out, epi))
    q.qgemv_chain(ops)
    torch.cuda.synchronize()
    for op, (d, x, n_out, epi) in zip(ops, host):
        y1 = torch.empty((M, n_out), dtype=torch.bfloat16, device="cuda")
        q.qgemv_chain([nvfp4_op(d, x, y1, epi, norm=gamma)])
        torch.cuda.synchronize()
        assert torch.equal(op["y"].view(torch.int16), y1.view(torch.int16))


@pytest.mark.parametrize("M", [1, 4, 8])
def test_q45_layer_with_fused_ffn_in_one_call(M):
    """The mixed recipe's layer as one qgemv_chain call: QK (Q4) and V (Q5)
    with the RMSNorm prologue, O (Q4), the Q5/Q4 SwiGLU FFN with its own
    RMSNorm, down (Q4) with the residual; every output against the oracle.
    (Four and eight tokens: the warp-MMA stage.)"""
    d27 = synth.DENSE27B
    H, I = d27.hidden, d27.inter
    gam1, gam2 = gamma_bits(H, 97), gamma_bits(H, 98)
    specs = {name: (N, K, bits) for name, N, K, bits in synth.Q45_RECIPE}
    W = {name: synth.q45_weights(3, f"q45.{name}", N, K, bits) for name, (N, K, bits) in specs.items()}
    xa = synth.bf16_normal(99, "lay.xa", (8, H))[:M]
    attn = synth.bf16_normal(99, "lay.attn", (8, d27.o_k))[:M]
    xf = synth.bf16_normal(99, "lay.xf", (8, H))[:M]
    hmid = synth.bf16_normal(99, "lay.hmid", (8, I))[:M]
    res = synth.bf16_normal(99, "lay.res", (8, H))[:M]
    D = {k: q45_dev(v) for k, v in W.items()}
    ys = {"qk": (M, specs["qk"][0]), "v": (M, specs["v"][0]), "o": (M, H), "ffn": (M, I), "down": (M, H)}
    Y = {k: torch.empty(s, dtype=torch.bfloat16, device="cuda") for k, s in ys.items()}
    g1, g2 = to_dev(gam1), to_dev(gam2)
    ops = [q_op(D["qk"], to_dev(xa), Y["qk"], norm=g1),
           q_op(D["v"], to_dev(xa), Y["v"], norm=g1),
           q_op(D["o"], to_dev(attn), Y["o"]),
           q_op(D["gate"], to_dev(xf), Y["ffn"], norm=g2, up=D["up"]),
           q_op(D["down"], to_dev(hmid), Y["down"], residual=to_dev(res))]
    q.qgemv_chain(ops)
    torch.cuda.synchronize()
    assert q.qg_last_device_status() == q.QG_OK
    h1, dh1 = norm_ref(xa, gam1)
    for name in ("qk", "v"):
        yref, a = O.gemv_q45(W[name], h1)
        check_bf16(bits16(Y[name]), yref, widened(O.dequant_q45(W[name]), a, dh1), f"layer {name}")
    yref, a = O.gemv_q45(W["o"], attn)
    check_bf16(bits16(Y["o"]), yref, gemv_bound(a), "layer o")
    h2, dh2 = norm_ref(xf, gam2)
    g_ref, ag = O.gemv_q45(W["gate"], h2)
    u_ref, au = O.gemv_q45(W["up"], h2)
    B = swiglu_bound(g_ref, u_ref, widened(O.dequant_q45(W["gate"]), ag, dh2),
                     widened(O.dequant_q45(W["up"]), au, dh2))
    check_bf16(bits16(Y["ffn"]), O.swiglu(g_ref, u_ref), B, "layer ffn")
    yref, a = O.gemv_q45(W["down"], hmid, residual=res)
    check_bf16(bits16(Y["down"]), yref, gemv_bound(a), "layer down")
