"""The C-ABI library: it builds, loads, exports every declared symbol, and
rejects bad arguments with the documented status before launching anything
(no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")


@pytest.fixture(scope="module")
def L():
    from bit_quantized_weight_gb300 import build as B
    if B.needs_build():
        B.build()
    import bit_quantized_weight_gb300 as q
    return q.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*QG_API\s+(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("qgemv_nvfp4", "qgemv_q45", "qgemv_swiglu_nvfp4", "moe_qgemv_nvfp4", "qgemv_chain", "qgemv_swiglu_q45",
              "qgemv_chain_ws", "qgemv_chain_workspace_size",
              "moe_qgemv_nvfp4_workspace_size", "moe_route_topk", "qdequant_nvfp4", "qdequant_q45",
              "qg_last_device_status", "qg_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in include/qgemv.h but not exported"


def test_library_hides_cuda_runtime_symbols(L):
    for name in ("cudaMalloc", "cudaLaunchKernel", "cudaStreamSynchronize"):
        with pytest.raises(AttributeError):
            getattr(L, name)


def test_status_strings(L):
    import bit_quantized_weight_gb300 as q
    assert q.qg_status_string(0) == "QG_OK"
    assert q.qg_status_string(q.QG_ERR_DEVICE_TIMEOUT) == "QG_ERR_DEVICE_TIMEOUT"
    assert q.qg_status_string(99) == "QG_ERR_UNKNOWN"


A = 0x100000  # fake, 16-byte-aligned addresses: validation never dereferences


def _no_visible_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


# These calls pass fake device addresses and must be rejected before any
# launch; they only run where no GPU is visible, so a regression that let one
# through could never touch a device. (The GPU suite repeats the rejections
# with real, deliberately misaligned allocations.)
fake_ptr = pytest.mark.skipif(not _no_visible_gpu(), reason="fake-pointer validation runs without a GPU")


@pytest.mark.parametrize("M,N,K,want", [
    (0, 16, 256, 1), (9, 16, 256, 1), (1, 0, 256, 1), (1, 16, 0, 1), (1, 16, 48, 1), (1, 16, 16, 1),
])
@fake_ptr
def test_dense_rejects_bad_sizes(L, M, N, K, want):
    assert L.qgemv_nvfp4(A, A, 1.0, A, A, 0, None, M, N, K, None) == want
    assert L.qgemv_swiglu_nvfp4(A, A, 1.0, A, A, M, 2 * N, K, None) == want
    assert L.qgemv_q45(A, None, A, A, 4, A, A, 0, None, M, N, K, None) == want


@fake_ptr
def test_dense_rejects_null_and_misaligned(L):
    assert L.qgemv_nvfp4(None, A, 1.0, A, A, 0, None, 1, 16, 256, None) == 1
    assert L.qgemv_nvfp4(A, A, 1.0, A + 8, A, 0, None, 1, 16, 256, None) == 3
    assert L.qgemv_nvfp4(A, A, 1.0, A, A + 2, 0, None, 1, 16, 256, None) == 3
    assert L.qgemv_nvfp4(A, A, 1.0, A, A, 0, A + 4, 1, 16, 256, None) == 3
    assert L.qgemv_nvfp4(A, A, 1.0, A, A, 7, None, 1, 16, 256, None) == 1      # bad y dtype
    assert L.qgemv_swiglu_nvfp4(A, A, 1.0, A, A, 1, 15, 256, None) == 1        # odd N


@fake_ptr
def test_q45_rejects_bad_bits_and_planes(L):
    assert L.qgemv_q45(A, None, A, A, 3, A, A, 0, None, 1, 16, 256, None) == 1
    assert L.qgemv_q45(A, None, A, A, 5, A, A, 0, None, 1, 16, 256, None) == 1  # Q5 needs q_hi
    assert L.qgemv_q45(A, A, A, A, 4, A, A, 0, None, 1, 16, 256, None) == 1     # Q4 takes none
    assert L.qgemv_q45(A, A, A, None, 5, A, A, 0, None, 1, 16, 256, None) == 1
    assert L.qgemv_q45(A, A + 1, A, A, 5, A, A, 0, None, 1, 16, 256, None) == 3


@fake_ptr
def test_router_and_moe_validation(L):
    assert L.moe_route_topk(A, 8, 128, 9, A, A, None) == 1
    assert L.moe_route_topk(A, 8, 4, 8, A, A, None) == 1
    assert L.moe_route_topk(A, 0, 128, 8, A, A, None) == 1
    assert L.moe_route_topk(A + 4, 8, 128, 8, A, A, None) == 3
    sz = ctypes.c_size_t(0)
    assert L.moe_qgemv_nvfp4_workspace_size(8, 8, 2048, 768, 128, ctypes.byref(sz)) == 0
    assert sz.value > 8 * 8 * 768 * 2
    assert L.moe_qgemv_nvfp4_workspace_size(8, 8, 2000, 768, 128, ctypes.byref(sz)) == 1
    args = [A] * 10
    # workspace too small / missing
    assert L.moe_qgemv_nvfp4(*args, A, 16, 8, 2048, 768, 128, 8, None) == 4
    assert L.moe_qgemv_nvfp4(*args, None, 1 << 30, 8, 2048, 768, 128, 8, None) == 4
    assert L.moe_qgemv_nvfp4(*args, A + 16, 1 << 30, 8, 2048, 768, 128, 8, None) == 3
    assert L.moe_qgemv_nvfp4(*args, A, 1 << 30, 8, 2048, 768, 128, 9, None) == 1


@fake_ptr
def test_noalloc_moe_validation(L):
    args = [A] * 10
    # the same argument checks as the workspace entry point, in the same order
    assert L.moe_qgemv_nvfp4_noalloc(None, *args[1:], 8, 2048, 768, 128, 8, None) == 1
    assert L.moe_qgemv_nvfp4_noalloc(*args, 8, 2048, 768, 128, 9, None) == 1
    assert L.moe_qgemv_nvfp4_noalloc(A + 8, *args[1:], 8, 2048, 768, 128, 8, None) == 3
    # misaligned and too large: the pointer check comes first
    assert L.moe_qgemv_nvfp4_noalloc(A + 8, *args[1:], 8, 16384, 8192, 64, 8, None) == 3
    # H = 16384, I = 8192 at M = 8, top-8 needs far more than the 4 MiB scratch
    assert L.moe_qgemv_nvfp4_noalloc(*args, 8, 16384, 8192, 64, 8, None) == 4


def _op(**kw):
    import bit_quantized_weight_gb300 as q
    rec = q.QgGemvOp()
    base = dict(format=0, epilogue=0, y_dtype=0, after_previous=0, N=64, K=256, codes=A, q_hi=None, scales=A,
                mins=None, global_scale=1.0, x=A, residual=None, y=A)
    base.update(kw)
    for k, v in base.items():
        setattr(rec, k, v)
    return rec


def _chain(L, recs, M=1, sync=None):
    import bit_quantized_weight_gb300 as q
    arr = (q.QgGemvOp * len(recs))(*recs)
    return L.qgemv_chain(arr, len(recs), M, sync, None)


@fake_ptr
def test_chain_validation(L):
    assert _chain(L, [_op(format=3)]) == 1
    assert _chain(L, [_op(epilogue=5)]) == 1
    assert _chain(L, [_op(y_dtype=2)]) == 1
    assert _chain(L, [_op(epilogue=1)]) == 1                      # residual epilogue without residual
    assert _chain(L, [_op(residual=A)]) == 1                      # residual without its epilogue
    assert _chain(L, [_op(format=1, epilogue=2, mins=A)]) == 1   # SwiGLU is NVFP4 only
    assert _chain(L, [_op(epilogue=2, N=63)]) == 1
    assert _chain(L, [_op(epilogue=2, y_dtype=1)]) == 1
    assert _chain(L, [_op(format=1)]) == 1                        # Q needs mins
    assert _chain(L, [_op(format=2, mins=A)]) == 1                # Q5 needs q_hi
    assert _chain(L, [_op(format=1, mins=A, q_hi=A)]) == 1        # Q4 takes none
    assert _chain(L, [_op(mins=A)]) == 1                          # NVFP4 takes no mins
    assert _chain(L, [_op(K=48)]) == 1
    assert _chain(L, [_op(x=A + 8)]) == 3
    assert _chain(L, [_op(format=1, mins=A + 4)]) == 3
    assert _chain(L, [_op()], M=0) == 1
    assert _chain(L, [_op()], M=9) == 1
    assert L.qgemv_chain(None, 1, 1, None, None) == 1
    assert _chain(L, [_op()] * 9) == 1
    # a later op reading earlier outputs needs the sync words
    assert _chain(L, [_op(), _op(after_previous=1)]) == 1
    assert _chain(L, [_op(), _op(after_previous=1)], sync=A + 4) == 3
    # RMSNorm weight alignment; separate up matrices only for groupwise-int SwiGLU
    assert _chain(L, [_op(norm_weight=A + 2)]) == 3
    q5 = dict(format=2, mins=A, q_hi=A)
    assert _chain(L, [_op(up_codes=A, up_format=1, up_scales=A, up_mins=A)]) == 1        # no SwiGLU
    assert _chain(L, [_op(epilogue=2, up_codes=A, up_format=1, up_scales=A, up_mins=A)]) == 1  # NVFP4
    assert _chain(L, [_op(epilogue=2, **q5)]) == 1                                        # Q needs up
    assert _chain(L, [_op(epilogue=2, up_codes=A, up_format=0, up_scales=A, up_mins=A, **q5)]) == 1
    assert _chain(L, [_op(epilogue=2, up_codes=A, up_format=2, up_scales=A, up_mins=A, **q5)]) == 1  # Q5 up: plane
    assert _chain(L, [_op(epilogue=2, up_codes=A, up_format=1, up_scales=A, up_mins=None, **q5)]) == 1
    assert _chain(L, [_op(epilogue=2, up_codes=A + 4, up_format=1, up_scales=A, up_mins=A, **q5)]) == 3
    assert _chain(L, [_op(up_scales=A)]) == 1                                             # stray up field


def test_chain_workspace_size(L):
    import bit_quantized_weight_gb300 as q
    recs = [_op(N=64, K=1024), _op(format=2, mins=A, q_hi=A, N=32, K=512), _op(K=256 * 68)]
    arr = (q.QgGemvOp * 3)(*recs)
    sz = ctypes.c_size_t(0)
    for M in (1, 3, 8):
        assert L.qgemv_chain_workspace_size(arr, 3, M, ctypes.byref(sz)) == 0
        up = lambda v: (v + 255) // 256 * 256
        want = up(4 * (M * 576 + 48)) + up(2 * (M * 576 + 304)) + up(68 * (M * 576 + 48))
        assert sz.value == want
    assert L.qgemv_chain_workspace_size(arr, 3, 9, ctypes.byref(sz)) == 1
    assert L.qgemv_chain_workspace_size(arr, 0, 4, ctypes.byref(sz)) == 1
    assert L.qgemv_chain_workspace_size(None, 1, 4, ctypes.byref(sz)) == 1
    assert L.qgemv_chain_workspace_size(arr, 3, 4, None) == 1


@fake_ptr
def test_chain_ws_validation(L):
    import bit_quantized_weight_gb300 as q
    arr = (q.QgGemvOp * 2)(_op(K=1024), _op(K=512))
    sz = ctypes.c_size_t(0)
    assert L.qgemv_chain_workspace_size(arr, 2, 4, ctypes.byref(sz)) == 0
    # op checks first, then the workspace's size and alignment
    bad = (q.QgGemvOp * 1)(_op(x=A + 8))
    assert L.qgemv_chain_ws(bad, 1, 4, None, A, 1 << 20, None) == 3
    assert L.qgemv_chain_ws(arr, 2, 4, None, A, sz.value - 16, None) == 4
    assert L.qgemv_chain_ws(arr, 2, 4, None, A + 16, sz.value, None) == 3
    assert L.qgemv_chain_ws(arr, 2, 9, None, A, sz.value, None) == 1


@fake_ptr
def test_swiglu_q45_validation(L):
    args = dict(gate=(A, A, A, A, 5), up=(A, None, A, A, 4))
    def call(gate=args["gate"], up=args["up"], x=A, nw=None, y=A, M=1, I=64, K=256):
        return L.qgemv_swiglu_q45(*gate, *up, x, nw, 1e-6, y, M, I, K, None)
    assert call(gate=(A, A, A, A, 3)) == 1
    assert call(up=(A, None, A, A, 6)) == 1
    assert call(gate=(A, None, A, A, 5)) == 1          # Q5 gate needs its plane
    assert call(up=(A, A, A, A, 4)) == 1               # Q4 up takes none
    assert call(M=0) == 1
    assert call(M=9) == 1
    assert call(K=48) == 1
    assert call(x=A + 8) == 3
    assert call(nw=A + 2) == 3
    assert call(up=(A, None, A, A + 4, 4)) == 3


def test_chain_record_layout_matches_the_header(tmp_path):
    """The binding's qg_gemv_op has the C struct's size and field offsets."""
    import shutil
    import subprocess
    import bit_quantized_weight_gb300 as q
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    fields = [f for f, _ in q.QgGemvOp._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "qgemv.h"\nint main(void){\n'
                   '  printf("%zu", sizeof(qg_gemv_op));\n'
                   + "".join(f'  printf(" %zu", offsetof(qg_gemv_op, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    cuda_inc = "/usr/local/cuda/include"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [ctypes.sizeof(q.QgGemvOp)] + [getattr(q.QgGemvOp, f).offset for f in fields]
    assert got == want


@fake_ptr
def test_dequant_validation(L):
    assert L.qdequant_nvfp4(A, A, 1.0, A, 0, 256, None) == 1
    assert L.qdequant_nvfp4(A, A, 1.0, A + 4, 16, 256, None) == 3
    assert L.qdequant_q45(A, None, A, A, 5, A, 16, 256, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import bit_quantized_weight_gb300.qgemv as qm
    monkeypatch.setattr(qm, "_lib", None)
    monkeypatch.setattr(qm, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not found"):
        qm.lib()
