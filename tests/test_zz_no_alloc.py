"""The MoE entry point that allocates nothing (GPU).

moe_qgemv_nvfp4_noalloc serves callers that cannot allocate device memory
(a plugin whose host framework owns all device memory, a decode loop that may
not call cudaMalloc): it uses the library's fixed device scratch instead of a
caller workspace. Two calls in a row, with different routing, must each give
the same output as moe_qgemv_nvfp4 with a workspace, within the oracle bound
the other MoE tests use. This file is collected last so that a run stopping
at the first failure has already run every other test.
"""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_util import bits16, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
q = pytest.importorskip("bit_quantized_weight_gb300")


def _inputs(seed, c):
    E, H, I, M = c.experts, c.hidden, c.inter, c.M
    gu = synth.nvfp4_weights(seed, "moe.gu", E * 2 * I, H)
    dn = synth.nvfp4_weights(seed, "moe.dn", E * H, I)
    gu_h = {"codes": gu["codes"].reshape(E, 2 * I, H // 2), "scales": gu["scales"].reshape(E, 2 * I, H // 16),
            "g": np.ones(E)}
    dn_h = {"codes": dn["codes"].reshape(E, H, I // 2), "scales": dn["scales"].reshape(E, H, I // 16),
            "g": np.ones(E)}
    return gu_h, dn_h


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from test_gpu_moe import check_moe
    torch.cuda.set_device(0)
    q.qg_debug_set_wait(0, False)
    c = synth.MOE35B
    gu, dn = _inputs(9, c)
    d = {k: to_dev(v) for k, v in (("gc", gu["codes"]), ("gs", gu["scales"]), ("dc", dn["codes"]),
                                   ("ds", dn["scales"]))}
    gg = torch.ones(c.experts, dtype=torch.float32, device="cuda")
    dg = torch.ones(c.experts, dtype=torch.float32, device="cuda")
    ws = torch.empty(q.moe_qgemv_nvfp4_workspace_size(c.M, c.topk, c.hidden, c.inter, c.experts),
                     dtype=torch.uint8, device="cuda")
    # every device tensor of both calls exists before the calls, so that the
    # free device memory measured around them can only move if the entry
    # point itself allocated
    calls = []
    for call in range(2):                        # two calls in a row, different routing
        x = synth.bf16_normal(10 + call, "noalloc.x", (c.M, c.hidden))
        lg = synth.router_logits(10 + call, "noalloc.logits", c.M, c.experts)
        ids, w64 = O.route_topk(lg, c.topk)
        w32 = w64.astype(np.float32).astype(np.float64)
        calls.append({"x": x, "ids": ids, "w32": w32, "xd": to_dev(x), "idd": torch.from_numpy(ids).cuda(),
                      "wd": torch.from_numpy(w32.astype(np.float32)).cuda(),
                      "y_ws": torch.empty((c.M, c.hidden), dtype=torch.bfloat16, device="cuda"),
                      "y_na": torch.empty((c.M, c.hidden), dtype=torch.bfloat16, device="cuda"),
                      "h_ws": torch.empty(c.M * c.topk * c.inter, dtype=torch.bfloat16, device="cuda")})
    # one call first: on a device where the library's code is not loaded yet,
    # it makes the driver load it (and the scratch array with it)
    k0 = calls[0]
    q.moe_qgemv_nvfp4_noalloc(d["gc"], d["gs"], gg, d["dc"], d["ds"], dg, k0["xd"], k0["idd"], k0["wd"],
                              k0["y_na"])
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for k in calls:
        q.moe_qgemv_nvfp4(d["gc"], d["gs"], gg, d["dc"], d["ds"], dg, k["xd"], k["idd"], k["wd"], k["y_ws"], ws)
        k["h_ws"].copy_(ws[: c.M * c.topk * c.inter * 2].view(torch.bfloat16))
        q.moe_qgemv_nvfp4_noalloc(d["gc"], d["gs"], gg, d["dc"], d["ds"], dg, k["xd"], k["idd"], k["wd"],
                                  k["y_na"])
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert q.qg_last_device_status() == q.QG_OK
    assert free_after == free_before, f"free device memory moved by {free_before - free_after} bytes"
    for call, k in enumerate(calls):
        a, b = bits16(k["y_ws"]), bits16(k["y_na"])
        assert np.array_equal(a, b), f"call {call}: no-alloc output differs from the workspace entry point"
        h_ws = bits16(k["h_ws"].view(c.M, c.topk, c.inter))
        check_moe(gu, dn, k["x"], k["ids"], k["w32"], b, h_ws)
