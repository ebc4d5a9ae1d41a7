"""MoE router and expert-gathered NVFP4 FFN against the fp64 oracle (GPU).

Router: top-k ids equal the oracle's (softmax order, ties to the lower id);
the renormalised weights agree to fp32 rounding.

MoE (a reading; only the GEMV bound is stated): the intermediate
h = bf16(silu(G x) * (U x)) is read back from the workspace and checked per
(token, slot) with the SwiGLU bound. The output y is checked against the
oracle's own h (never the GPU's): each h element the GPU may legitimately
produce lies in [rne(v - B), rne(v + B)], and the down projection turns those
intervals into the bound
    sum_i |w_i| * ( sum_q |d_jq| * dh_q + 1e-4 * sum_q |d_jq h_q| ) + 1e-6
with dh_q the larger distance from the oracle's h_q to its interval ends.
"""
import numpy as np
import pytest

import oracle as O
import synth
from checks import check_bf16, gemv_bound, swiglu_bound
from gpu_util import bits16, to_dev

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


# ---------------------------------------------------------------- router
@pytest.mark.parametrize("M,E,k", [(8, 128, 8), (3, 16, 4), (1, 8, 8), (8, 1000, 2)])
def test_router_matches_oracle(M, E, k):
    lg = synth.router_logits(4, f"route{E}", M, E)
    lg[0, 1] = lg[0, 3]                                  # a tie: lower id first
    ids_ref, w_ref = O.route_topk(lg, k)
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    w = torch.empty((M, k), dtype=torch.float32, device="cuda")
    q.moe_route_topk(torch.from_numpy(lg).cuda(), k, ids, w)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    wg = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(wg - w_ref) <= 4e-7 * w_ref + 1e-12), np.max(np.abs(wg - w_ref) / w_ref)


# ---------------------------------------------------------------- MoE
def make_moe(seed, E, H, I, M, g_range=(1.0, 1.0)):
    gu = synth.nvfp4_weights(seed, "moe.gu", E * 2 * I, H)
    dn = synth.nvfp4_weights(seed, "moe.dn", E * H, I)
    r = np.random.default_rng(seed)
    gu_g = np.asarray(r.uniform(*g_range, E), np.float32).astype(np.float64)
    dn_g = np.asarray(r.uniform(*g_range, E), np.float32).astype(np.float64)
    gu_h = {"codes": gu["codes"].reshape(E, 2 * I, H // 2), "scales": gu["scales"].reshape(E, 2 * I, H // 16),
            "g": gu_g}
    dn_h = {"codes": dn["codes"].reshape(E, H, I // 2), "scales": dn["scales"].reshape(E, H, I // 16), "g": dn_g}
    x = synth.bf16_normal(seed, "moe.x", (M, H))
    return gu_h, dn_h, x


def run_moe(gu, dn, x, ids, w):
    E, two_i, hh = gu["codes"].shape
    H, I = hh * 2, two_i // 2
    M, topk = ids.shape
    ws_bytes = q.moe_qgemv_nvfp4_workspace_size(M, topk, H, I, E)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    y = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    q.moe_qgemv_nvfp4(to_dev(gu["codes"]), to_dev(gu["scales"]), torch.from_numpy(gu["g"].astype(np.float32)).cuda(),
                      to_dev(dn["codes"]), to_dev(dn["scales"]), torch.from_numpy(dn["g"].astype(np.float32)).cuda(),
                      to_dev(x), torch.from_numpy(ids.astype(np.int32)).cuda(),
                      torch.from_numpy(w.astype(np.float32)).cuda(), y, ws)
    torch.cuda.synchronize()
    h = ws[: M * topk * I * 2].view(torch.bfloat16).view(M, topk, I)
    return bits16(y), bits16(h)


def check_moe(gu, dn, x, ids, w32, y_bits, h_bits, valid=None):
    """w32: the fp32 routing weights both sides used (as float64 values)."""
    M, topk = ids.shape
    if valid is None:
        valid = np.ones(ids.shape, bool)
    ids_o = np.where(valid, ids, 0).astype(np.int32)
    gate, up, ag, au, h_ref = O.moe_gate_up(gu, x, ids_o)
    Bh = swiglu_bound(gate, up, gemv_bound(ag), gemv_bound(au))
    v = O.swiglu(gate, up)
    for m in range(M):
        seen = set()
        for i in range(topk):
            # h is stored for the first slot of each (token, expert); a repeated
            # expert reuses that row
            if valid[m, i] and ids[m, i] not in seen:
                seen.add(ids[m, i])
                check_bf16(h_bits[m, i], v[m, i], Bh[m, i], f"h token {m} slot {i}")
    hv = O.bf16_array(h_ref)
    lo = O.round_bf16(v - Bh)
    hi = O.round_bf16(v + Bh)
    dh = np.maximum(np.abs(hi - hv), np.abs(hv - lo))
    wv = np.where(valid, w32, 0.0)
    y_ref = O.moe_down(dn, hv, ids_o, wv)
    a_dh = O.moe_down(dn, dh, ids_o, np.abs(wv), use_abs=True)
    a_h = O.moe_down(dn, np.abs(hv), ids_o, np.abs(wv), use_abs=True)
    B = a_dh + 1e-4 * a_h + 2.0 ** -20 * a_h + 1e-6
    return check_bf16(y_bits, y_ref, B, "MoE y")


def test_moe_decode_layer_35b_a3b_shapes():
    c = synth.MOE35B
    gu, dn, x = make_moe(4, c.experts, c.hidden, c.inter, c.M)
    lg = synth.router_logits(4, "moe.logits", c.M, c.experts)
    ids, w64 = O.route_topk(lg, c.topk)
    w32 = w64.astype(np.float32).astype(np.float64)
    y, h = run_moe(gu, dn, x, ids, w32)
    check_moe(gu, dn, x, ids, w32, y, h)


def test_moe_full_path_with_device_router():
    c = synth.MOE35B
    gu, dn, x = make_moe(5, c.experts, c.hidden, c.inter, c.M)
    lg = synth.router_logits(5, "moe.logits", c.M, c.experts)
    ids_d = torch.empty((c.M, c.topk), dtype=torch.int32, device="cuda")
    w_d = torch.empty((c.M, c.topk), dtype=torch.float32, device="cuda")
    q.moe_route_topk(torch.from_numpy(lg).cuda(), c.topk, ids_d, w_d)
    torch.cuda.synchronize()
    ids_ref, w_ref = O.route_topk(lg, c.topk)
    assert np.array_equal(ids_d.cpu().numpy(), ids_ref)
    w32 = w_d.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(w32 - w_ref) <= 4e-7 * w_ref)
    y, h = run_moe(gu, dn, x, ids_ref, w32)
    check_moe(gu, dn, x, ids_ref, w32, y, h)


@pytest.mark.parametrize("M,E,H,I,topk", [(3, 6, 256, 256, 2), (8, 10, 512, 768, 4), (1, 4, 256, 512, 4)])
def test_moe_small_shapes_with_scales(M, E, H, I, topk):
    gu, dn, x = make_moe(6, E, H, I, M, g_range=(0.5, 2.0))
    r = np.random.default_rng(7)
    ids = np.stack([r.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    w = r.uniform(0.05, 1.0, (M, topk)).astype(np.float32).astype(np.float64)
    y, h = run_moe(gu, dn, x, ids, w)
    check_moe(gu, dn, x, ids, w, y, h)


def test_moe_tokens_sharing_experts():
    """Every expert routed by several tokens (the CUDA-core kernels pair them
    two per pass and repeat the expert's rows for a third and fourth), and
    two tokens with identical routing."""
    M, E, H, I, topk = 8, 5, 512, 512, 4
    gu, dn, x = make_moe(14, E, H, I, M, g_range=(0.5, 2.0))
    r = np.random.default_rng(15)
    ids = np.stack([r.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    ids[5] = ids[2]
    w = r.uniform(0.05, 1.0, (M, topk)).astype(np.float32).astype(np.float64)
    y, h = run_moe(gu, dn, x, ids, w)
    check_moe(gu, dn, x, ids, w, y, h)


def test_moe_tcgen05_fallback_when_the_plan_does_not_fit():
    """I = 3072: the down projection's activation rows overflow the CUDA-core
    kernel's shared memory, so it runs on the tcgen05 grouped kernel while
    gate/up stays on the CUDA cores."""
    M, E, H, I, topk = 8, 16, 2048, 3072, 8
    gu, dn, x = make_moe(16, E, H, I, M)
    r = np.random.default_rng(17)
    ids = np.stack([r.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    w = r.uniform(0.05, 1.0, (M, topk)).astype(np.float32).astype(np.float64)
    y, h = run_moe(gu, dn, x, ids, w)
    check_moe(gu, dn, x, ids, w, y, h)


def test_moe_duplicate_and_invalid_expert_ids():
    M, E, H, I, topk = 4, 6, 256, 256, 3
    gu, dn, x = make_moe(8, E, H, I, M)
    ids = np.array([[1, 1, 4], [2, 5, 0], [3, 99, 3], [0, 1, 2]], np.int32)   # dup, out of range
    valid = (ids >= 0) & (ids < E)
    w = np.full((M, topk), 0.25, np.float64)
    y, h = run_moe(gu, dn, x, ids, w)
    assert q.qg_last_device_status() == q.QG_ERR_INVALID_ARG
    check_moe(gu, dn, x, ids, w, y, h, valid=valid)
    assert q.qg_last_device_status() == q.QG_OK


def test_moe_bounded_wait_reports_timeout_and_recovers():
    """The grouped expert kernels' waits run out when the weight stream
    issues nothing; the call reports QG_ERR_DEVICE_TIMEOUT and a clean call
    right after matches the oracle."""
    M, E, H, I, topk = 4, 6, 256, 512, 2
    gu, dn, x = make_moe(12, E, H, I, M)
    r = np.random.default_rng(13)
    ids = np.stack([r.choice(E, topk, replace=False) for _ in range(M)]).astype(np.int32)
    w = r.uniform(0.05, 1.0, (M, topk)).astype(np.float32).astype(np.float64)
    assert q.qg_last_device_status() == q.QG_OK
    q.qg_debug_set_wait(20_000_000, True)
    try:
        run_moe(gu, dn, x, ids, w)
        assert q.qg_last_device_status() == q.QG_ERR_DEVICE_TIMEOUT
    finally:
        q.qg_debug_set_wait(0, False)
    y, h = run_moe(gu, dn, x, ids, w)
    assert q.qg_last_device_status() == q.QG_OK
    check_moe(gu, dn, x, ids, w, y, h)
