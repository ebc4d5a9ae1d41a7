"""ctypes binding of libqgemv (argument marshalling only).

The functions keep the C names. Tensor arguments are torch tensors on the
current CUDA device in the layouts of include/qgemv.h; the call is enqueued on
torch.cuda.current_stream(). A missing library raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

QG_OK = 0
QG_ERR_INVALID_ARG = 1
QG_ERR_UNSUPPORTED = 2
QG_ERR_MISALIGNED = 3
QG_ERR_WORKSPACE = 4
QG_ERR_CUDA = 5
QG_ERR_DEVICE_TIMEOUT = 6
QG_OUT_BF16 = 0
QG_OUT_F32 = 1
QG_FMT_NVFP4 = 0
QG_FMT_Q4 = 1
QG_FMT_Q5 = 2
QG_EPI_NONE = 0
QG_EPI_RESIDUAL = 1
QG_EPI_SWIGLU = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libqgemv.so")
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float


class QgGemvOp(ctypes.Structure):
    """qg_gemv_op of include/qgemv.h."""
    _fields_ = [("format", ctypes.c_int), ("epilogue", ctypes.c_int), ("y_dtype", ctypes.c_int),
                ("after_previous", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("codes", ctypes.c_void_p), ("q_hi", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("mins", ctypes.c_void_p), ("global_scale", ctypes.c_float), ("x", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("y", ctypes.c_void_p), ("norm_weight", ctypes.c_void_p),
                ("norm_eps", ctypes.c_float), ("up_format", ctypes.c_int), ("up_codes", ctypes.c_void_p),
                ("up_q_hi", ctypes.c_void_p), ("up_scales", ctypes.c_void_p), ("up_mins", ctypes.c_void_p)]


class QGemvError(RuntimeError):
    def __init__(self, name, status):
        super().__init__(f"{name} failed: {qg_status_string(status)} ({status})")
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load libqgemv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libqgemv.so not found at {_LIB_PATH}; build it with "
                "`python bit_quantized_weight_gb300/build.py` (needs nvcc)")
        L = ctypes.CDLL(_LIB_PATH)
        L.qgemv_nvfp4.argtypes = [_P, _P, _F, _P, _P, _I, _P, _I, _I, _I, _P]
        L.qgemv_q45.argtypes = [_P, _P, _P, _P, _I, _P, _P, _I, _P, _I, _I, _I, _P]
        L.qgemv_swiglu_nvfp4.argtypes = [_P, _P, _F, _P, _P, _I, _I, _I, _P]
        L.moe_route_topk.argtypes = [_P, _I, _I, _I, _P, _P, _P]
        L.moe_qgemv_nvfp4_workspace_size.argtypes = [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_qgemv_nvfp4.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                      _I, _I, _I, _I, _I, _P]
        L.moe_qgemv_nvfp4_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]
        L.qgemv_chain.argtypes = [ctypes.POINTER(QgGemvOp), _I, _I, _P, _P]
        L.qgemv_chain_ws.argtypes = [ctypes.POINTER(QgGemvOp), _I, _I, _P, _P, ctypes.c_size_t, _P]
        L.qgemv_chain_workspace_size.argtypes = [ctypes.POINTER(QgGemvOp), _I, _I, ctypes.POINTER(ctypes.c_size_t)]
        L.qgemv_swiglu_q45.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _P, _P, _F, _P, _I, _I, _I, _P]
        L.qdequant_nvfp4.argtypes = [_P, _P, _F, _P, _I, _I, _P]
        L.qdequant_q45.argtypes = [_P, _P, _P, _P, _I, _P, _I, _I, _P]
        L.qg_last_device_status.argtypes = [_P]
        L.qg_read_probe.argtypes = [_P, ctypes.c_size_t, _P, _P]
        L.qg_status_string.argtypes = [_I]
        L.qg_status_string.restype = ctypes.c_char_p
        L.qg_debug_set_wait.argtypes = [ctypes.c_uint64, _I]
        for name in ("qgemv_nvfp4", "qgemv_q45", "qgemv_swiglu_nvfp4", "moe_route_topk",
                     "moe_qgemv_nvfp4_workspace_size", "moe_qgemv_nvfp4", "moe_qgemv_nvfp4_noalloc",
                     "qgemv_chain", "qgemv_chain_ws", "qgemv_chain_workspace_size", "qgemv_swiglu_q45",
                     "qdequant_nvfp4",
                     "qdequant_q45", "qg_last_device_status", "qg_debug_set_wait"):
            getattr(L, name).restype = _I
        _lib = L
    return _lib


def qg_status_string(status: int) -> str:
    return lib().qg_status_string(int(status)).decode()


def _check(name, status):
    if status != QG_OK:
        raise QGemvError(name, status)


def _ptr(t):
    # ctypes converts a Python int for a c_void_p argument
    return None if t is None else t.data_ptr()


_raw_stream = None


def _stream(stream=None, like=None):
    """The stream handle: `stream`'s, else the current stream of the device
    of tensor `like` (else of the current device)."""
    global _raw_stream
    if stream is not None:
        return stream.cuda_stream
    import torch
    if _raw_stream is None:
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None) or False
    if _raw_stream:
        dev = like.get_device() if like is not None else torch.cuda.current_device()
        return _raw_stream(dev)
    return torch.cuda.current_stream().cuda_stream


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def qgemv_nvfp4(codes, scales, g, x, y, residual=None, stream=None):
    """y[M][N] (bf16 or fp32 tensor) = NVFP4 W[N][K] @ x[M][K] (+ residual)."""
    import torch
    _cuda(codes, scales, x, y, residual)
    M, K = x.shape
    N = codes.shape[0]
    out = QG_OUT_F32 if y.dtype == torch.float32 else QG_OUT_BF16
    _check("qgemv_nvfp4", lib().qgemv_nvfp4(_ptr(codes), _ptr(scales), float(g), _ptr(x), _ptr(y), out,
                                            _ptr(residual), M, N, K, _stream(stream, y)))
    return y


def qgemv_q45(q_lo, q_hi, scale, mn, bits, x, y, residual=None, stream=None):
    import torch
    _cuda(q_lo, q_hi, scale, mn, x, y, residual)
    M, K = x.shape
    N = q_lo.shape[0]
    out = QG_OUT_F32 if y.dtype == torch.float32 else QG_OUT_BF16
    _check("qgemv_q45", lib().qgemv_q45(_ptr(q_lo), _ptr(q_hi), _ptr(scale), _ptr(mn), int(bits), _ptr(x),
                                        _ptr(y), out, _ptr(residual), M, N, K, _stream(stream, y)))
    return y


def qgemv_swiglu_nvfp4(codes, scales, g, x, y, stream=None):
    _cuda(codes, scales, x, y)
    M, K = x.shape
    N = codes.shape[0]
    _check("qgemv_swiglu_nvfp4", lib().qgemv_swiglu_nvfp4(_ptr(codes), _ptr(scales), float(g), _ptr(x),
                                                          _ptr(y), M, N, K, _stream(stream, y)))
    return y


def moe_route_topk(logits, topk, ids, w, stream=None):
    _cuda(logits, ids, w)
    M, E = logits.shape
    _check("moe_route_topk", lib().moe_route_topk(_ptr(logits), M, E, int(topk), _ptr(ids), _ptr(w),
                                                  _stream(stream, logits)))
    return ids, w


def moe_qgemv_nvfp4_workspace_size(M, topk, H, I, E) -> int:
    b = ctypes.c_size_t(0)
    _check("moe_qgemv_nvfp4_workspace_size",
           lib().moe_qgemv_nvfp4_workspace_size(M, topk, H, I, E, ctypes.byref(b)))
    return b.value


def moe_qgemv_nvfp4(gu_codes, gu_scales, gu_g, dn_codes, dn_scales, dn_g, x, ids, w, y, workspace,
                    stream=None):
    _cuda(gu_codes, gu_scales, gu_g, dn_codes, dn_scales, dn_g, x, ids, w, y, workspace)
    E, two_i, hh = gu_codes.shape
    M, H = x.shape
    topk = ids.shape[1]
    _check("moe_qgemv_nvfp4", lib().moe_qgemv_nvfp4(
        _ptr(gu_codes), _ptr(gu_scales), _ptr(gu_g), _ptr(dn_codes), _ptr(dn_scales), _ptr(dn_g), _ptr(x),
        _ptr(ids), _ptr(w), _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        M, H, two_i // 2, E, topk, _stream(stream, y)))
    return y


def moe_qgemv_nvfp4_noalloc(gu_codes, gu_scales, gu_g, dn_codes, dn_scales, dn_g, x, ids, w, y, stream=None):
    """moe_qgemv_nvfp4 for callers that cannot allocate: the library's own
    fixed 4 MiB device scratch replaces the workspace (see include/qgemv.h)."""
    _cuda(gu_codes, gu_scales, gu_g, dn_codes, dn_scales, dn_g, x, ids, w, y)
    E, two_i, hh = gu_codes.shape
    M, H = x.shape
    topk = ids.shape[1]
    _check("moe_qgemv_nvfp4_noalloc", lib().moe_qgemv_nvfp4_noalloc(
        _ptr(gu_codes), _ptr(gu_scales), _ptr(gu_g), _ptr(dn_codes), _ptr(dn_scales), _ptr(dn_g), _ptr(x),
        _ptr(ids), _ptr(w), _ptr(y), M, H, two_i // 2, E, topk, _stream(stream, y)))
    return y


_FORMATS = {"nvfp4": QG_FMT_NVFP4, "q4": QG_FMT_Q4, "q5": QG_FMT_Q5}
_EPILOGUES = {"none": QG_EPI_NONE, "residual": QG_EPI_RESIDUAL, "swiglu": QG_EPI_SWIGLU}


class GemvChain:
    """A prepared qgemv_chain call: the op records are built once, so that
    run() is one C call. Each op is a dict with the weight tensors of its
    format (NVFP4: codes, scales, g; Q4/Q5: q_lo, q_hi (Q5), scale, min),
    "x", "y", optionally "residual", "epilogue" ("none", "residual",
    "swiglu") and "after_previous" (bool). The tensors must stay alive and
    unchanged in place for as long as the chain is run. By default the chain
    owns a workspace (qgemv_chain_ws: activations converted once per call);
    workspace=False runs qgemv_chain without one. Runs of one chain must not
    overlap on the GPU (they share the workspace)."""

    def __init__(self, ops, sync=None, workspace=True):
        """ops: dicts as above; optional "norm" (bf16 gamma [K] tensor) and
        "norm_eps" select the RMSNorm prologue, and for groupwise-int SwiGLU
        "up" is a dict with the up matrix's q_lo, q_hi, scale, min."""
        import torch
        n = len(ops)
        self.ops = (QgGemvOp * n)()
        self.keep = []
        M = None
        for i, op in enumerate(ops):
            x, y = op["x"], op["y"]
            r = op.get("residual")
            if "codes" in op:
                fmt, codes, q_hi, scales, mins, g = QG_FMT_NVFP4, op["codes"], None, op["scales"], None, op["g"]
            else:
                fmt = QG_FMT_Q5 if op.get("q_hi") is not None else QG_FMT_Q4
                codes, q_hi, scales, mins, g = op["q_lo"], op.get("q_hi"), op["scale"], op["min"], 1.0
            _cuda(codes, q_hi, scales, mins, x, y, r)
            epi = op.get("epilogue", "residual" if r is not None else "none")
            rec = self.ops[i]
            rec.format = fmt
            rec.epilogue = _EPILOGUES[epi]
            rec.y_dtype = QG_OUT_F32 if y.dtype == torch.float32 else QG_OUT_BF16
            rec.after_previous = int(bool(op.get("after_previous", False)))
            rec.N = codes.shape[0]
            rec.K = x.shape[1]
            rec.codes, rec.q_hi, rec.scales, rec.mins = _ptr(codes), _ptr(q_hi), _ptr(scales), _ptr(mins)
            rec.global_scale = float(g)
            rec.x, rec.residual, rec.y = _ptr(x), _ptr(r), _ptr(y)
            nw = op.get("norm")
            _cuda(nw)
            rec.norm_weight = _ptr(nw)
            rec.norm_eps = float(op.get("norm_eps", 1e-6))
            up = op.get("up")
            if up is not None:
                _cuda(up["q_lo"], up.get("q_hi"), up["scale"], up["min"])
                rec.up_format = QG_FMT_Q5 if up.get("q_hi") is not None else QG_FMT_Q4
                rec.up_codes, rec.up_q_hi = _ptr(up["q_lo"]), _ptr(up.get("q_hi"))
                rec.up_scales, rec.up_mins = _ptr(up["scale"]), _ptr(up["min"])
            self.keep.append(op)
            if M is None:
                M = x.shape[0]
            elif x.shape[0] != M:
                raise ValueError("every op of a chain takes the same number of tokens")
        self.n, self.M = n, M
        self.sync = sync
        self.like = ops[0]["y"]
        self.ws, self.ws_bytes = None, 0
        if workspace:
            nb = ctypes.c_size_t(0)
            _check("qgemv_chain_workspace_size", lib().qgemv_chain_workspace_size(self.ops, n, M, ctypes.byref(nb)))
            self.ws_bytes = max(int(nb.value), 256)
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.like.device)

    def run(self, stream=None):
        _check("qgemv_chain", lib().qgemv_chain_ws(self.ops, self.n, self.M, _ptr(self.sync), _ptr(self.ws),
                                                   self.ws_bytes, _stream(stream, self.like)))


def qgemv_chain(ops, sync=None, stream=None, workspace=True):
    """Run a list of projections as one qgemv_chain call (see GemvChain)."""
    GemvChain(ops, sync, workspace).run(stream)


def qgemv_swiglu_q45(gate, up, x, y, norm=None, norm_eps=1e-6, stream=None):
    """y[M][I] = bf16(silu(G h) * (U h)) over separate groupwise-int gate and
    up matrices (dicts with q_lo, q_hi (Q5 only), scale, min); h = x, or the
    RMSNorm of x with gamma `norm` (bf16 [K])."""
    _cuda(gate["q_lo"], gate.get("q_hi"), gate["scale"], gate["min"], up["q_lo"], up.get("q_hi"), up["scale"],
          up["min"], x, y, norm)
    M, K = x.shape
    I = gate["q_lo"].shape[0]
    gb = 5 if gate.get("q_hi") is not None else 4
    ub = 5 if up.get("q_hi") is not None else 4
    _check("qgemv_swiglu_q45", lib().qgemv_swiglu_q45(
        _ptr(gate["q_lo"]), _ptr(gate.get("q_hi")), _ptr(gate["scale"]), _ptr(gate["min"]), gb,
        _ptr(up["q_lo"]), _ptr(up.get("q_hi")), _ptr(up["scale"]), _ptr(up["min"]), ub, _ptr(x), _ptr(norm),
        float(norm_eps), _ptr(y), M, I, K, _stream(stream, y)))
    return y


def qdequant_nvfp4(codes, scales, g, w, stream=None):
    _cuda(codes, scales, w)
    N, K = w.shape
    _check("qdequant_nvfp4", lib().qdequant_nvfp4(_ptr(codes), _ptr(scales), float(g), _ptr(w), N, K,
                                                  _stream(stream, w)))
    return w


def qdequant_q45(q_lo, q_hi, scale, mn, bits, w, stream=None):
    _cuda(q_lo, q_hi, scale, mn, w)
    N, K = w.shape
    _check("qdequant_q45", lib().qdequant_q45(_ptr(q_lo), _ptr(q_hi), _ptr(scale), _ptr(mn), int(bits),
                                              _ptr(w), N, K, _stream(stream, w)))
    return w


def read_probe(buf, sink, stream=None):
    """XOR every 32-bit word of the CUDA tensor `buf` into the one-word
    int32 CUDA tensor `sink` with 128-bit streaming loads (see qg_read_probe)."""
    _cuda(buf, sink)
    _check("qg_read_probe", lib().qg_read_probe(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink),
                                                _stream(stream, buf)))
    return sink


def qg_last_device_status(stream=None) -> int:
    return lib().qg_last_device_status(_stream(stream))


def qg_debug_set_wait(limit_ns: int = 0, starve: bool = False) -> None:
    _check("qg_debug_set_wait", lib().qg_debug_set_wait(int(limit_ns), int(bool(starve))))
