"""qgemv_chain: a decode layer's projections in one call (GPU).

The ops run in one persistent kernel (one or two tokens: the CUDA-core
stage; three to eight: the warp-MMA stage, with the activations converted
per CTA, or once into a workspace when the chain has one -- the default of
GemvChain; `ws` below selects); each op must give exactly what
its single-projection call gives where that call takes the same stage (same
plan and arithmetic: bit for bit where the standalone kernel also picks 32-k
segments), and match the oracle within the stated bound. Ops flagged
after_previous read earlier outputs of the same call through the grid-wide
barrier; each such stage is checked against the oracle fed the GPU's own
earlier output.
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


def sync_words():
    return torch.zeros(4, dtype=torch.int32, device="cuda")   # 16 bytes; the call uses two words


def dense_layer_ops(M, seed=1):
    """The 27B-class layer's four NVFP4 projections with independent inputs."""
    ops, host = [], []
    for name, N, K, epi in synth.dense_layer_shapes():
        w = synth.nvfp4_weights(seed, f"dense.{name}", N, K)
        x = synth.bf16_normal(seed, f"chain.{name}.x.M{M}", (M, K))
        r = synth.bf16_normal(seed, f"chain.{name}.r.M{M}", (M, N)) if epi == "residual" else None
        d = nvfp4_dev(w)
        n_out = N // 2 if epi == "swiglu" else N
        op = {"codes": d["codes"], "scales": d["scales"], "g": d["g"], "x": to_dev(x),
              "y": torch.empty((M, n_out), dtype=torch.bfloat16, device="cuda"),
              "epilogue": epi}
        if r is not None:
            op["residual"] = to_dev(r)
        ops.append(op)
        host.append((name, N, K, epi, w, x, r))
    return ops, host


def run_separately(ops):
    outs = []
    for op in ops:
        y = torch.empty_like(op["y"])
        if op.get("epilogue") == "swiglu":
            q.qgemv_swiglu_nvfp4(op["codes"], op["scales"], op["g"], op["x"], y)
        elif "codes" in op:
            q.qgemv_nvfp4(op["codes"], op["scales"], op["g"], op["x"], y, residual=op.get("residual"))
        else:
            q.qgemv_q45(op["q_lo"], op.get("q_hi"), op["scale"], op["min"], 5 if op.get("q_hi") is not None else 4,
                        op["x"], y, residual=op.get("residual"))
        outs.append(y)
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("M,ws", [(1, True), (2, True), (4, True), (8, True), (4, False), (8, False)])
def test_chain_dense_layer_matches_separate_calls(M, ws):
    ops, host = dense_layer_ops(M)
    q.qgemv_chain(ops, workspace=ws)
    torch.cuda.synchronize()
    assert q.qg_last_device_status() == q.QG_OK
    sep = run_separately(ops)
    for op, ys, (name, N, K, epi, w, x, r) in zip(ops, sep, host):
        assert torch.equal(op["y"].view(torch.int16), ys.view(torch.int16)), f"{name}: chain != separate call"
        if M in (1, 2, 8):
            if epi == "swiglu":
                yref, a = O.gemv_nvfp4(w, x)
                I = N // 2
                B = swiglu_bound(yref[:, :I], yref[:, I:], gemv_bound(a[:, :I]), gemv_bound(a[:, I:]))
                check_bf16(bits16(op["y"]), O.swiglu(yref[:, :I], yref[:, I:]), B, f"chain {name}")
            else:
                yref, a = O.gemv_nvfp4(w, x, residual=r)
                check_out(op["y"], yref, a, f"chain {name}")


@pytest.mark.parametrize("M,ws", [(1, True), (2, True), (4, True), (8, True), (4, False)])
def test_chain_dependent_ops_through_the_grid_barrier(M, ws):
    """o: y1 = W_o x (+ r); gate/up reads y1; down reads h with y1 as its
    residual; a last projection reads the down output -- each op after the
    first waits for the earlier ones inside the one launch."""
    H, I = 1024, 2048
    wo = synth.nvfp4_weights(70, "dep.o", H, 1536)
    wgu = synth.nvfp4_weights(70, "dep.gu", 2 * I, H)
    wdn = synth.nvfp4_weights(70, "dep.dn", H, I)
    wl = synth.nvfp4_weights(70, "dep.last", 512, H)
    x = synth.bf16_normal(71, "dep.x", (8, 1536))[:M]
    r = synth.bf16_normal(71, "dep.r", (8, H))[:M]
    D = {k: nvfp4_dev(w) for k, w in (("o", wo), ("gu", wgu), ("dn", wdn), ("last", wl))}
    y1 = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    h = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    y3 = torch.empty((M, 512), dtype=torch.float32, device="cuda")
    ops = [
        {**D["o"], "x": to_dev(x), "y": y1, "residual": to_dev(r)},
        {**D["gu"], "x": y1, "y": h, "epilogue": "swiglu", "after_previous": True},
        {**D["dn"], "x": h, "y": y2, "residual": y1, "after_previous": True},
        {**D["last"], "x": y2, "y": y3, "after_previous": True},
    ]
    sync = sync_words()
    for rep in range(2):                    # the sync words are reusable
        q.qgemv_chain(ops, sync=sync, workspace=ws)
        torch.cuda.synchronize()
        assert q.qg_last_device_status() == q.QG_OK
        assert int(sync[0].item()) == 0, "arrival count not reset"
        # a waiting op: one barrier; with the workspace at 3..8 tokens a second
        # one after its activations are converted
        per_op = 2 if (ws and M >= 3) else 1
        assert int(sync[1].item()) == 3 * per_op * (rep + 1), "barrier generations"
    y1b, hb, y2b = bits16(y1), bits16(h), bits16(y2)
    yref, a = O.gemv_nvfp4(wo, x, residual=r)
    check_bf16(y1b, yref, gemv_bound(a), "dep o")
    g_ref, ag = O.gemv_nvfp4(wgu, y1b)
    B = swiglu_bound(g_ref[:, :I], g_ref[:, I:], gemv_bound(ag[:, :I]), gemv_bound(ag[:, I:]))
    check_bf16(hb, O.swiglu(g_ref[:, :I], g_ref[:, I:]), B, "dep gate/up")
    yref, a = O.gemv_nvfp4(wdn, hb, residual=y1b)
    check_bf16(y2b, yref, gemv_bound(a), "dep down")
    yref, a = O.gemv_nvfp4(wl, y2b)
    check_f32(y3.cpu().numpy(), yref, gemv_bound(a), "dep last")


@pytest.mark.parametrize("M,ws", [(1, True), (2, True), (4, True), (8, True), (4, False), (8, False)])
def test_chain_q45_layer_full_size(M, ws):
    ops, host = [], []
    for name, N, K, bits in synth.Q45_RECIPE:
        w = synth.q45_weights(3, f"q45.{name}", N, K, bits)
        x = synth.bf16_normal(72, f"chainq.{name}.x", (8, K))[:M]
        r = synth.bf16_normal(72, f"chainq.{name}.r", (8, N))[:M] if name == "down" else None
        d = q45_dev(w)
        op = {"q_lo": d["q_lo"], "q_hi": d["q_hi"], "scale": d["scale"], "min": d["min"], "x": to_dev(x),
              "y": torch.empty((M, N), dtype=torch.bfloat16, device="cuda")}
        if r is not None:
            op["residual"] = to_dev(r)
        ops.append(op)
        host.append((name, w, x, r))
    q.qgemv_chain(ops, workspace=ws)
    torch.cuda.synchronize()
    assert q.qg_last_device_status() == q.QG_OK
    sep = run_separately(ops)
    for op, ys, (name, w, x, r) in zip(ops, sep, host):
        if M <= 6:   # seven or eight tokens: the separate call takes the groupwise mma.sync kernel
            assert torch.equal(op["y"].view(torch.int16), ys.view(torch.int16)), f"{name}: chain != separate call"
        yref, a = O.gemv_q45(w, x, residual=r)
        check_out(op["y"], yref, a, f"chain Q {name}")


@pytest.mark.parametrize("M,ws", [(1, True), (2, True), (5, True), (5, False), (3, True)])
def test_chain_mixed_formats_and_fp32_outputs(M, ws):
    """NVFP4 and Q4/Q5 ops in one launch, fp32 and bf16 outputs, ragged rows."""
    specs = [("nvfp4", 1000, 768, torch.float32), ("q5", 333, 1024, torch.bfloat16),
             ("q4", 2049, 512, torch.float32), ("nvfp4", 77, 2304, torch.bfloat16)]
    ops, host = [], []
    for i, (fmt, N, K, dt) in enumerate(specs):
        x = synth.bf16_normal(73, f"mix.x{i}", (8, K))[:M]
        if fmt == "nvfp4":
            w = synth.nvfp4_weights(73, f"mix.w{i}", N, K, g=0.5)
            d = nvfp4_dev(w)
            op = {"codes": d["codes"], "scales": d["scales"], "g": d["g"]}
        else:
            w = synth.q45_weights(73, f"mix.w{i}", N, K, 5 if fmt == "q5" else 4)
            d = q45_dev(w)
            op = {"q_lo": d["q_lo"], "q_hi": d["q_hi"], "scale": d["scale"], "min": d["min"]}
        op.update({"x": to_dev(x), "y": torch.empty((M, N), dtype=dt, device="cuda")})
        ops.append(op)
        host.append((fmt, w, x))
    q.qgemv_chain(ops, workspace=ws)
    torch.cuda.synchronize()
    assert q.qg_last_device_status() == q.QG_OK
    for op, (fmt, w, x) in zip(ops, host):
        yref, a = (O.gemv_nvfp4 if fmt == "nvfp4" else O.gemv_q45)(w, x)
        check_out(op["y"], yref, a, f"chain mixed {fmt}")


@pytest.mark.parametrize("M,ws", [(1, True), (4, True), (4, False)])
def test_chain_bounded_wait_reports_timeout_and_recovers(M, ws):
    ops, host = dense_layer_ops(M, seed=2)
    ops = ops[:2]
    chain = q.GemvChain(ops, workspace=ws)
    assert q.qg_last_device_status() == q.QG_OK
    q.qg_debug_set_wait(20_000_000, True)
    try:
        chain.run()
        assert q.qg_last_device_status() == q.QG_ERR_DEVICE_TIMEOUT
    finally:
        q.qg_debug_set_wait(0, False)
    chain.run()
    torch.cuda.synchronize()
    assert q.qg_last_device_status() == q.QG_OK
    sep = run_separately(ops)
    for op, ys in zip(ops, sep):
        assert torch.equal(op["y"].view(torch.int16), ys.view(torch.int16))


@pytest.mark.parametrize("M", [4, 8])
def test_chain_workspace_groupwise_op_after_an_earlier_output(M):
    """The workspace plan converts an after_previous op inside the launch:
    a Q5 op (residual) and a Q4 op reading the NVFP4 op's output, against
    the oracle fed the GPU's own earlier output, and against the plan
    without the workspace bit for bit."""
    H = 1024
    w0 = synth.nvfp4_weights(74, "wsdep.0", H, 768)
    w1 = synth.q45_weights(74, "wsdep.1", 640, H, 5)
    w2 = synth.q45_weights(74, "wsdep.2", 300, H, 4)
    x = synth.bf16_normal(75, "wsdep.x", (8, 768))[:M]
    r = synth.bf16_normal(75, "wsdep.r", (8, 640))[:M]
    d0, d1, d2 = nvfp4_dev(w0), q45_dev(w1), q45_dev(w2)
    outs = {}
    for ws in (True, False):
        y0 = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
        y1 = torch.empty((M, 640), dtype=torch.bfloat16, device="cuda")
        y2 = torch.empty((M, 300), dtype=torch.float32, device="cuda")
        ops = [{**d0, "x": to_dev(x), "y": y0},
               {"q_lo": d1["q_lo"], "q_hi": d1["q_hi"], "scale": d1["scale"], "min": d1["min"], "x": y0, "y": y1,
                "residual": to_dev(r), "after_previous": True},
               {"q_lo": d2["q_lo"], "scale": d2["scale"], "min": d2["min"], "x": y0, "y": y2,
                "after_previous": True}]
        q.qgemv_chain(ops, sync=sync_words(), workspace=ws)
        torch.cuda.synchronize()
        assert q.qg_last_device_status() == q.QG_OK
        outs[ws] = (y0, y1, y2)
    for a, b in zip(outs[True], outs[False]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
    y0, y1, y2 = outs[True]
    y0b = bits16(y0)
    yref, a = O.gemv_nvfp4(w0, x)
    check_bf16(y0b, yref, gemv_bound(a), "ws dep nvfp4")
    yref, a = O.gemv_q45(w1, y0b, residual=r)
    check_bf16(bits16(y1), yref, gemv_bound(a), "ws dep q5")
    yref, a = O.gemv_q45(w2, y0b)
    check_f32(y2.cpu().numpy(), yref, gemv_bound(a), "ws dep q4")


def test_chain_workspace_argument_errors():
    ops, _ = dense_layer_ops(4, seed=3)
    chain = q.GemvChain(ops)
    L = q.lib()
    st = q.qg_last_device_status
    ws = torch.empty(chain.ws_bytes + 256, dtype=torch.uint8, device="cuda")
    s = L.qgemv_chain_ws(chain.ops, chain.n, chain.M, None, ws.data_ptr(), chain.ws_bytes - 16, None)
    assert s == q.QG_ERR_WORKSPACE
    s = L.qgemv_chain_ws(chain.ops, chain.n, chain.M, None, ws.data_ptr() + 16, chain.ws_bytes, None)
    assert s == q.QG_ERR_MISALIGNED
    torch.cuda.synchronize()
    assert st() == q.QG_OK
