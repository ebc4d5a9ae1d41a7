"""Dense GEMV kernels against the fp64 oracle, through the C ABI (GPU).

Bit-exact dequantisation; GEMV outputs within the stated bound for NVFP4 and
Q4/Q5, M = 1..8, fp32 and bf16 outputs, residual and SwiGLU epilogues, ragged
shapes (rows not a multiple of the 16-row tile, one-row CTAs, K not a
multiple of the 256-wide chunk), activations that need the exact multi-term
path, determinism, untouched guard bands and the bounded-wait error path.
"""
import numpy as np
import pytest

import oracle as O
import synth
from checks import check_bf16, check_f32, gemv_bound, same_f32_bits, swiglu_bound
from gpu_util import bits16, guarded, nvfp4_dev, q45_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("bit_quantized_weight_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    q.qg_debug_set_wait(0, False)
    yield
    assert q.qg_last_device_status() == q.QG_OK


def run_nvfp4(w, x_bits, out=torch.bfloat16, residual=None):
    d = nvfp4_dev(w)
    x = to_dev(x_bits)
    M, N = x_bits.shape[0], w["codes"].shape[0]
    y = torch.empty((M, N), dtype=out, device="cuda")
    r = to_dev(residual) if residual is not None else None
    q.qgemv_nvfp4(d["codes"], d["scales"], d["g"], x, y, residual=r)
    torch.cuda.synchronize()
    return y


def check_out(y, yref, a, what):
    B = gemv_bound(a)
    if y.dtype == torch.float32:
        return check_f32(y.cpu().numpy(), yref, B, what)
    return check_bf16(bits16(y), yref, B, what)


# ---------------------------------------------------------------- dequant
@pytest.mark.parametrize("g", [1.0, 0.7, 3.0e-5])
def test_dequant_nvfp4_bit_exact(g):
    N, K = 256, 512
    w = synth.nvfp4_weights(101, "deq", N, K, g=g)
    # every E4M3 code, NaN codes included, appears as a block scale
    w["scales"] = ((np.arange(N)[:, None] + np.arange(K // 16)[None, :]) % 256).astype(np.uint8)
    # every code byte appears in every row
    w["codes"][:, :128] = (np.arange(128)[None, :] * 2 + np.arange(N)[:, None]) % 256
    d = nvfp4_dev(w)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    q.qdequant_nvfp4(d["codes"], d["scales"], w["g"], out)
    ref = O.dequant_nvfp4(w).astype(np.float32)          # RNE fp64 -> fp32
    assert same_f32_bits(out.cpu().numpy(), ref)


@pytest.mark.parametrize("bits", [4, 5])
def test_dequant_q45_bit_exact(bits):
    N, K = 128, 512
    w = synth.q45_weights(102, f"deq{bits}", N, K, bits)
    r = np.random.default_rng(5)
    # also arbitrary fp16 scale/min bit patterns (finite)
    sc = r.integers(0, 0x7C00, size=w["scale"].shape).astype(np.uint16) | (
        r.integers(0, 2, size=w["scale"].shape).astype(np.uint16) << 15)
    w["scale"][: N // 2] = sc[: N // 2]
    d = q45_dev(w)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    q.qdequant_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, out)
    ref = O.dequant_q45(w).astype(np.float32)
    assert same_f32_bits(out.cpu().numpy(), ref)


# ---------------------------------------------------------------- NVFP4 GEMV
def test_tiny_config_bf16_and_fp32():
    c = synth.TINY
    w = synth.nvfp4_weights(0, "tiny.w", c.N, c.K)
    x = synth.bf16_normal(0, "tiny.x", (c.M, c.K))
    yref, a = O.gemv_nvfp4(w, x)
    check_out(run_nvfp4(w, x, torch.bfloat16), yref, a, "tiny bf16")
    check_out(run_nvfp4(w, x, torch.float32), yref, a, "tiny fp32")


SHAPES = [
    # (M, N, K): ragged row counts, single-tile and multi-tile CTAs, several chunks
    (1, 1, 256), (1, 15, 512), (1, 17, 768), (2, 300, 1024), (3, 1000, 1280), (4, 4099, 512),
    (5, 2048, 2304), (6, 333, 4608), (7, 160, 256), (8, 1024, 1536), (8, 7001, 512),
    (1, 5000, 2048), (8, 64, 9216), (1, 40000, 256),
    # two tokens: many units, few rows, long K
    (2, 40000, 256), (2, 5000, 2048), (2, 17, 768), (2, 513, 17408),
    # K % 256 != 0 takes the exact CUDA-core kernel
    (1, 40, 32), (3, 77, 96), (8, 33, 800),
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_nvfp4_shapes(M, N, K, out):
    w = synth.nvfp4_weights(7, f"s{M}.{N}.{K}", N, K, g=0.75)
    x = synth.bf16_normal(8, f"x{M}.{K}", (M, K))
    yref, a = O.gemv_nvfp4(w, x)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    check_out(run_nvfp4(w, x, dt), yref, a, f"nvfp4 M={M} N={N} K={K} {out}")


@pytest.mark.parametrize("M,N,K", [(1, 513, 1024), (8, 200, 768), (2, 96, 32 * 7), (2, 513, 1024)])
def test_nvfp4_residual(M, N, K):
    w = synth.nvfp4_weights(9, "res", N, K)
    x = synth.bf16_normal(10, "resx", (M, K))
    r = synth.bf16_normal(11, "resr", (M, N))
    yref, a = O.gemv_nvfp4(w, x, residual=r)
    check_out(run_nvfp4(w, x, torch.bfloat16, residual=r), yref, a, "residual bf16")
    check_out(run_nvfp4(w, x, torch.float32, residual=r), yref, a, "residual fp32")


def test_nvfp4_residual_in_place():
    M, N, K = 2, 300, 512
    w = synth.nvfp4_weights(12, "rip", N, K)
    x = synth.bf16_normal(13, "ripx", (M, K))
    r = synth.bf16_normal(14, "ripr", (M, N))
    yref, a = O.gemv_nvfp4(w, x, residual=r)
    d = nvfp4_dev(w)
    y = to_dev(r).clone()
    q.qgemv_nvfp4(d["codes"], d["scales"], 1.0, to_dev(x), y, residual=y)
    torch.cuda.synchronize()
    check_out(y, yref, a, "in-place residual")


@pytest.mark.parametrize("M,I,K", [(1, 256, 512), (1, 300, 1024), (4, 1000, 768), (8, 64, 2048), (3, 50, 96),
                                   (1, 20000, 256), (2, 300, 1024), (2, 20000, 256)])
def test_swiglu(M, I, K):
    w = synth.nvfp4_weights(15, f"sw{I}", 2 * I, K, g=1.25)
    x = synth.bf16_normal(16, "swx", (M, K))
    yref, a = O.gemv_nvfp4(w, x)
    ga, ua = yref[:, :I], yref[:, I:]
    Bg, Bu = gemv_bound(a[:, :I]), gemv_bound(a[:, I:])
    href = O.swiglu(ga, ua)
    d = nvfp4_dev(w)
    y = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    q.qgemv_swiglu_nvfp4(d["codes"], d["scales"], 1.25, to_dev(x), y)
    torch.cuda.synchronize()
    check_bf16(bits16(y), href, swiglu_bound(ga, ua, Bg, Bu), "swiglu")


# ---------------------------------------------------------------- Q4 / Q5
@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (3, 1000, 1024), (8, 4099, 768), (2, 17, 256), (5, 70, 96),
                                   (1, 4099, 768), (1, 17, 256), (1, 1000, 4608), (1, 40000, 256)])
def test_q45(bits, M, N, K):
    w = synth.q45_weights(17, f"q{bits}.{N}.{K}", N, K, bits)
    x = synth.bf16_normal(18, f"qx{K}", (M, K))
    yref, a = O.gemv_q45(w, x)
    d = q45_dev(w)
    xd = to_dev(x)
    for dt in (torch.bfloat16, torch.float32):
        y = torch.empty((M, N), dtype=dt, device="cuda")
        q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, xd, y)
        torch.cuda.synchronize()
        check_out(y, yref, a, f"Q{bits} M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_q45_residual(M):
    N, K = 640, 1024
    w = synth.q45_weights(19, "qres", N, K, 5)
    x = synth.bf16_normal(20, "qresx", (M, K))
    r = synth.bf16_normal(21, "qresr", (M, N))
    yref, a = O.gemv_q45(w, x, residual=r)
    d = q45_dev(w)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], 5, to_dev(x), y, residual=to_dev(r))
    torch.cuda.synchronize()
    check_out(y, yref, a, "Q5 residual")


@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("M", [2, 3, 8])
def test_q45_long_k(bits, M):
    """K = 17408 (68 stages): the stage ring wraps many times, and the
    activation copies of the first ring's stages are issued after the
    weight copies."""
    N, K = 200, 17408
    w = synth.q45_weights(26, f"qlong{bits}", N, K, bits)
    x = synth.bf16_normal(27, "qlongx", (M, K))
    yref, a = O.gemv_q45(w, x)
    d = q45_dev(w)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, to_dev(x), y)
    torch.cuda.synchronize()
    check_out(y, yref, a, f"Q{bits} long K M={M}")


@pytest.mark.parametrize("big,small", [(8, 7), (6, 3)])
def test_q45_deterministic_and_row_independent(big, small):
    """Q4/Q5 with several tokens: repeated calls are bit-identical and a
    token's result does not depend on the other tokens of the call, within
    one kernel (7..8 tokens: the groupwise mma.sync kernel; 3..6: the
    warp-MMA kernel). One and two tokens take the CUDA-core kernel, whose
    two-token results equal one-token calls (checked separately)."""
    N, K = 700, 2048
    w = synth.q45_weights(33, "qdet", N, K, 5)
    x = synth.bf16_normal(34, "qdetx", (big, K))
    d = q45_dev(w)

    def run(xb):
        y = torch.empty((xb.shape[0], N), dtype=torch.float32, device="cuda")
        q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], 5, to_dev(xb), y)
        torch.cuda.synchronize()
        return y.cpu().numpy()
    y1, y2 = run(x), run(x)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32)), "two runs differ"
    for m in (0, big - 2):
        ym = run(np.stack([x[(m + i) % big] for i in range(small)]))
        assert np.array_equal(ym[0].view(np.uint32), y1[m].view(np.uint32)), \
            f"row {m}: M={small} call != M={big} call"
    yref, a = O.gemv_q45(w, x)
    check_out(torch.from_numpy(y1), yref, a, f"Q5 M={big}")


# ---------------------------------------------------------------- activations
def wide_range_x(M, K, seed):
    """bf16 activations whose magnitudes span 2^-60 .. 2^20 inside every
    256-wide chunk (plus zeros and bf16 subnormals), so that a single f16 term
    cannot hold them exactly."""
    r = np.random.default_rng(seed)
    e = r.integers(-60, 21, size=(M, K))
    v = r.choice([-1.0, 1.0], size=(M, K)) * (1 + r.integers(0, 128, size=(M, K)) / 128.0) * np.exp2(e)
    v[:, ::37] = 0.0
    v[:, 5::101] = np.exp2(-130.0)                 # bf16 subnormal
    import torch as T
    return T.from_numpy(v.astype(np.float32)).to(T.bfloat16).view(T.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_nvfp4_wide_dynamic_range_activations(M):
    N, K = 300, 1024
    w = synth.nvfp4_weights(22, "wide", N, K)
    x = wide_range_x(M, K, 23)
    yref, a = O.gemv_nvfp4(w, x)
    check_out(run_nvfp4(w, x, torch.float32), yref, a, "wide-range fp32")
    check_out(run_nvfp4(w, x, torch.bfloat16), yref, a, "wide-range bf16")


@pytest.mark.parametrize("M", [4, 8])
def test_nvfp4_activation_windows_with_wide_range_chunks(M):
    """K = 17408 at four and eight tokens: the warp-MMA kernel holds the
    activations a window of chunks at a time; chunks in later windows whose
    values f16 cannot carry exactly (for one token only) switch those stages
    to bf16 operands."""
    N, K = 600, 17408
    w = synth.nvfp4_weights(24, "win", N, K)
    x = synth.bf16_normal(25, "winx", (M, K))
    wide = wide_range_x(1, K, 26)
    for kc in (3, 40, 41, 66):                       # one token, chunks spread over the windows
        x[M - 1, kc * 256:(kc + 1) * 256] = wide[0, kc * 256:(kc + 1) * 256]
    yref, a = O.gemv_nvfp4(w, x)
    check_out(run_nvfp4(w, x, torch.float32), yref, a, f"windows M={M}")
    r = synth.bf16_normal(27, "winr", (M, N))
    yref, a = O.gemv_nvfp4(w, x, residual=r)
    check_out(run_nvfp4(w, x, torch.bfloat16, residual=r), yref, a, f"windows + residual M={M}")


@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_q45_wide_dynamic_range_activations(bits, M):
    N, K = 200, 512
    w = synth.q45_weights(24, "qwide", N, K, bits)
    x = wide_range_x(M, K, 25)
    yref, a = O.gemv_q45(w, x)
    d = q45_dev(w)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, to_dev(x), y)
    torch.cuda.synchronize()
    check_out(y, yref, a, f"Q{bits} wide-range")


def test_zero_and_tiny_activations():
    N, K = 128, 512
    w = synth.nvfp4_weights(26, "zero", N, K)
    x = np.zeros((2, K), np.uint16)
    x[1] = synth.bf16_normal(27, "tinyx", (1, K))[0]
    x[1] = (x[1] & 0x807F) | (0x01 << 7)              # exponent field 1: |x| ~ 2^-126
    yref, a = O.gemv_nvfp4(w, x)
    check_out(run_nvfp4(w, x, torch.float32), yref, a, "zero/tiny fp32")
    for m in range(2):                                  # one token at a time
        yref1, a1 = O.gemv_nvfp4(w, x[m:m + 1])
        check_out(run_nvfp4(w, x[m:m + 1], torch.float32), yref1, a1, f"zero/tiny fp32 row {m}")


def test_non_finite_activations_propagate():
    N, K = 64, 256
    w = synth.nvfp4_weights(28, "nan", N, K)
    x = synth.bf16_normal(29, "nanx", (2, K))
    x[0, 3] = 0x7F80                                   # +inf
    x[1, 200] = 0x7FC0                                 # NaN
    y = run_nvfp4(w, x, torch.float32).cpu().numpy()
    assert not np.isfinite(y[0]).any() or np.isinf(y[0]).any()
    assert np.isnan(y[1]).all()
    y1 = run_nvfp4(w, x[1:2], torch.float32).cpu().numpy()   # one token
    assert np.isnan(y1).all()


# ---------------------------------------------------------------- config 1 at full size
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_dense_layer_full_size(M):
    d27 = synth.DENSE27B
    for name, N, K, epi in synth.dense_layer_shapes():
        w = synth.nvfp4_weights(1, f"dense.{name}", N, K)
        x = synth.bf16_normal(1, f"dense.{name}.x.M{M}", (M, K))
        if epi == "swiglu":
            yref, a = O.gemv_nvfp4(w, x)
            I = N // 2
            href = O.swiglu(yref[:, :I], yref[:, I:])
            B = swiglu_bound(yref[:, :I], yref[:, I:], gemv_bound(a[:, :I]), gemv_bound(a[:, I:]))
            dd = nvfp4_dev(w)
            y = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
            q.qgemv_swiglu_nvfp4(dd["codes"], dd["scales"], 1.0, to_dev(x), y)
            torch.cuda.synchronize()
            check_bf16(bits16(y), href, B, f"{name} M={M}")
        else:
            r = synth.bf16_normal(1, f"dense.{name}.r.M{M}", (M, N)) if epi == "residual" else None
            yref, a = O.gemv_nvfp4(w, x, residual=r)
            check_out(run_nvfp4(w, x, torch.bfloat16, residual=r), yref, a, f"{name} M={M}")
    assert d27.hidden == 5120


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_mixed_q45_layer_full_size(M):
    for name, N, K, bits in synth.Q45_RECIPE:
        w = synth.q45_weights(3, f"q45.{name}", N, K, bits)
        x = synth.bf16_normal(3, f"q45.{name}.x", (8, K))[:M]
        yref, a = O.gemv_q45(w, x)
        d = q45_dev(w)
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, to_dev(x), y)
        torch.cuda.synchronize()
        check_out(y, yref, a, f"Q{bits} {name}")


@pytest.mark.parametrize("bits", [4, 5])
@pytest.mark.parametrize("residual", [False, True])
def test_q45_two_tokens_match_one_token_calls(bits, residual):
    """The two-token groupwise-int kernel decodes each code once for both
    tokens but keeps their prescales, sums and epilogues apart: with
    activations that prescale exactly, each token equals its own one-token
    call bit for bit."""
    N, K = 3001, 2560
    w = synth.q45_weights(40 + bits, f"q2tok{bits}", N, K, bits)
    x = synth.bf16_normal(41, "q2tokx", (2, K))
    r = synth.bf16_normal(42, "q2tokr", (2, N)) if residual else None
    d = q45_dev(w)
    xd = to_dev(x)
    rd = to_dev(r) if residual else None
    y2 = torch.empty((2, N), dtype=torch.float32, device="cuda")
    q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, xd, y2, residual=rd)
    for t in range(2):
        y1 = torch.empty((1, N), dtype=torch.float32, device="cuda")
        q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], bits, xd[t:t + 1].clone(), y1,
                    residual=None if rd is None else rd[t:t + 1].clone())
        torch.cuda.synchronize()
        assert torch.equal(y1[0], y2[t]), f"token {t}: two-token call != one-token call"
    yref, a = O.gemv_q45(w, x, residual=r)
    check_out(y2, yref, a, f"Q{bits} two tokens")


# ---------------------------------------------------------------- properties
def test_deterministic_and_row_independent():
    """Repeated calls are bit-identical; a token's result does not depend on
    the other tokens of a 3..8-token call (same arithmetic for every such M);
    the one- and two-token CUDA-core kernel applies block scales per 16-k
    block instead, so it is checked against the oracle's bound, and its
    two-token results against one-token calls bit for bit."""
    M, N, K = 8, 2000, 2048
    w = synth.nvfp4_weights(30, "det", N, K)
    x = synth.bf16_normal(31, "detx", (M, K))
    y1 = run_nvfp4(w, x, torch.float32).cpu().numpy()
    y2 = run_nvfp4(w, x, torch.float32).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32)), "two runs differ"
    for m in (0, 5):
        three = np.stack([x[m], x[(m + 3) % M], x[(m + 1) % M]])
        ym = run_nvfp4(w, three, torch.float32).cpu().numpy()
        assert np.array_equal(ym[0].view(np.uint32), y1[m].view(np.uint32)), f"row {m}: M=3 call != M=8 call"
        y_one = run_nvfp4(w, x[m:m + 1], torch.float32)
        y_one2 = run_nvfp4(w, x[m:m + 1], torch.float32)
        assert torch.equal(y_one, y_one2), "one-token runs differ"
        yref, a = O.gemv_nvfp4(w, x[m:m + 1])
        check_out(y_one, yref, a, f"row {m} one-token call")
        y_two = run_nvfp4(w, np.stack([x[m], x[(m + 3) % M]]), torch.float32)
        assert torch.equal(y_two[0], y_one[0]), f"row {m}: two-token call != one-token call"
        y_b = run_nvfp4(w, x[(m + 3) % M:(m + 3) % M + 1], torch.float32)
        assert torch.equal(y_two[1], y_b[0]), f"row {(m + 3) % M}: two-token call != one-token call"


def test_outputs_stay_inside_their_buffer():
    M, N, K = 3, 1001, 768
    w = synth.nvfp4_weights(32, "guard", N, K)
    x = synth.bf16_normal(33, "guardx", (M, K))
    d = nvfp4_dev(w)
    for dt in (torch.bfloat16, torch.float32):
        y, check = guarded((M, N), dt)
        q.qgemv_nvfp4(d["codes"], d["scales"], 1.0, to_dev(x), y)
        torch.cuda.synchronize()
        check()
    y, check = guarded((M, N // 2), torch.bfloat16)
    q.qgemv_swiglu_nvfp4(d["codes"][: 2 * (N // 2)].contiguous(), d["scales"][: 2 * (N // 2)].contiguous(),
                         1.0, to_dev(x), y)
    torch.cuda.synchronize()
    check()


def test_rejects_misaligned_device_pointers():
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    L = q.lib()
    p = buf.data_ptr()
    assert L.qgemv_nvfp4(p, p, 1.0, p + 8, p, 0, None, 1, 16, 256, None) == q.QG_ERR_MISALIGNED
    assert L.qgemv_nvfp4(p + 4, p, 1.0, p, p, 0, None, 1, 16, 256, None) == q.QG_ERR_MISALIGNED
    assert L.qgemv_nvfp4(p, p, 1.0, p, p, 0, None, 0, 16, 256, None) == q.QG_ERR_INVALID_ARG


def _nvfp4_call(M, N, K, seed):
    w = synth.nvfp4_weights(seed, f"starve{M}", N, K)
    x = synth.bf16_normal(seed + 1, f"starvex{M}", (M, K))
    d = nvfp4_dev(w)
    xd = to_dev(x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")

    def call():
        q.qgemv_nvfp4(d["codes"], d["scales"], 1.0, xd, y)
    ref = O.gemv_nvfp4(w, x)
    return call, y, ref


def _q5_call(M, N, K, seed):
    w = synth.q45_weights(seed, f"starveq{M}", N, K, 5)
    x = synth.bf16_normal(seed + 1, f"starveqx{M}", (M, K))
    d = q45_dev(w)
    xd = to_dev(x)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")

    def call():
        q.qgemv_q45(d["q_lo"], d["q_hi"], d["scale"], d["min"], 5, xd, y)
    ref = O.gemv_q45(w, x)
    return call, y, ref


# One case per pipelined kernel: the one-token CUDA-core NVFP4 and Q5
# kernels, their two-token variants, the warp-MMA kernel (NVFP4 at 8 tokens,
# Q5 at 4) and the mma.sync groupwise-int kernel (Q5, 8 tokens).
STARVE_CASES = [("nvfp4", 1), ("nvfp4", 2), ("nvfp4", 8), ("q5", 1), ("q5", 2), ("q5", 4), ("q5", 8)]


@pytest.mark.parametrize("fmt,M", STARVE_CASES)
def test_bounded_wait_reports_timeout_and_recovers(fmt, M):
    N, K = 512, 1024
    call, y, (yref, a) = (_nvfp4_call if fmt == "nvfp4" else _q5_call)(M, N, K, 34 + M)
    assert q.qg_last_device_status() == q.QG_OK
    q.qg_debug_set_wait(20_000_000, True)             # 20 ms, the weight stream issues nothing
    try:
        call()
        assert q.qg_last_device_status() == q.QG_ERR_DEVICE_TIMEOUT
    finally:
        q.qg_debug_set_wait(0, False)
    call()                                            # a clean call right after
    torch.cuda.synchronize()
    assert q.qg_last_device_status() == q.QG_OK
    check_out(y, yref, a, f"{fmt} M={M} after timeout")
