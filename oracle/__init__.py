"""fp64 CPU oracle for the quantised decode GEMV -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package. The product (the CUDA library and its Python binding) never
imports, links or runs it. The arithmetic lives in oracle.c (plain C, fp64);
this module only marshals numpy arrays and splits independent output rows
over host threads (ctypes releases the GIL during each call, and each output
element is still one sequential fp64 sum in k order).
"""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_D = ctypes.c_double


def _configure(lib):
    for name in ("orc_e2m1", "orc_e4m3", "orc_f16", "orc_bf16"):
        getattr(lib, name).restype = _D
        getattr(lib, name).argtypes = [ctypes.c_uint]
    lib.orc_round_bf16.restype = _D
    lib.orc_round_bf16.argtypes = [_D]
    lib.orc_bf16_bits.restype = ctypes.c_uint
    lib.orc_bf16_bits.argtypes = [_D]
    lib.orc_silu.restype = _D
    lib.orc_silu.argtypes = [_D]
    lib.orc_dequant_nvfp4.argtypes = [_P, _P, _D, _I64, _I64, _P]
    lib.orc_dequant_q45.argtypes = [_P, _P, _P, _P, ctypes.c_int, _I64, _I64, _P]
    lib.orc_gemv_nvfp4.argtypes = [_P, _P, _D, _P, _P, _I64, _I64, _I64, _I64, _I64, _P, _P]
    lib.orc_gemv_q45.argtypes = [_P, _P, _P, _P, ctypes.c_int, _P, _P, _I64, _I64, _I64,
                                 _I64, _I64, _P, _P]
    lib.orc_swiglu.argtypes = [_P, _P, _I64, _P]
    lib.orc_rmsnorm.argtypes = [_P, _P, _D, _I64, _I64, _P, _P, _P]
    lib.orc_round_bf16_array.argtypes = [_P, _I64, _P]
    lib.orc_bf16_bits_array.argtypes = [_P, _I64, _P]
    lib.orc_bf16_array.argtypes = [_P, _I64, _P]
    lib.orc_f16_array.argtypes = [_P, _I64, _P]
    lib.orc_e4m3_array.argtypes = [_P, _I64, _P]
    lib.orc_route_topk.argtypes = [_P, _I64, _I64, ctypes.c_int, _P, _P]
    lib.orc_moe_gate_up.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, ctypes.c_int, _I64,
                                    _I64, _P, _P, _P, _P, _P]
    lib.orc_moe_down.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, ctypes.c_int,
                                 ctypes.c_int, _I64, _I64, _P]
    return lib


def _load():
    global _lib
    if _lib is None:
        if _build.needs_build():
            _build.build()
        _lib = _configure(ctypes.CDLL(_build.LIB))
    return _lib


def lib():
    return _load()


def use_library(path: str | None):
    """Point the wrapper at another build of oracle.c (the mutation tests
    compile copies with a planted mistake). None restores the default build.
    Returns the handle that was active before."""
    global _lib
    prev = _lib
    _lib = None if path is None else _configure(ctypes.CDLL(path))
    return prev


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _split(n, parts):
    parts = max(1, min(parts, n)) if n > 0 else 1
    step = -(-n // parts) if n > 0 else 0
    return [(i, min(n, i + step)) for i in range(0, n, step)] if n > 0 else []


def _run_ranges(fn, n, threads):
    ranges = _split(n, threads)
    if len(ranges) <= 1:
        for a, b in ranges:
            fn(a, b)
        return
    with ThreadPoolExecutor(max_workers=len(ranges)) as ex:
        list(ex.map(lambda ab: fn(*ab), ranges))


# ---------------------------------------------------------------- scalars
def e2m1(code: int) -> float:
    return _load().orc_e2m1(int(code))


def e4m3(code: int) -> float:
    return _load().orc_e4m3(int(code))


def f16(bits: int) -> float:
    return _load().orc_f16(int(bits))


def bf16(bits: int) -> float:
    return _load().orc_bf16(int(bits))


def silu(v: float) -> float:
    return _load().orc_silu(float(v))


# ---------------------------------------------------------------- arrays
def bf16_array(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().orc_bf16_array(_ptr(b), b.size, _ptr(out))
    return out


def f16_array(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().orc_f16_array(_ptr(b), b.size, _ptr(out))
    return out


def e4m3_array(codes) -> np.ndarray:
    b = _c(codes, np.uint8)
    out = np.empty(b.shape, np.float64)
    _load().orc_e4m3_array(_ptr(b), b.size, _ptr(out))
    return out


def round_bf16(v) -> np.ndarray:
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.float64)
    _load().orc_round_bf16_array(_ptr(a), a.size, _ptr(out))
    return out


def bf16_bits(v) -> np.ndarray:
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().orc_bf16_bits_array(_ptr(a), a.size, _ptr(out))
    return out


def swiglu(gate, up) -> np.ndarray:
    g = _c(gate, np.float64)
    u = _c(up, np.float64)
    assert g.shape == u.shape
    out = np.empty(g.shape, np.float64)
    _load().orc_swiglu(_ptr(g), _ptr(u), g.size, _ptr(out))
    return out


def rmsnorm(x, gamma, eps: float):
    """RMSNorm of bf16 rows x[M][K] with bf16 weight gamma[K]: returns
    (h bf16 bits [M][K], unrounded v [M][K], r [M])."""
    xx = _c(x, np.uint16)
    gg = _c(gamma, np.uint16)
    M, K = xx.shape
    assert gg.shape == (K,)
    r = np.empty(M, np.float64)
    v = np.empty((M, K), np.float64)
    h = np.empty((M, K), np.uint16)
    _load().orc_rmsnorm(_ptr(xx), _ptr(gg), float(eps), M, K, _ptr(r), _ptr(v), _ptr(h))
    return h, v, r


# ---------------------------------------------------------------- weights
def dequant_nvfp4(w: dict) -> np.ndarray:
    codes, scales = _c(w["codes"], np.uint8), _c(w["scales"], np.uint8)
    N, K = codes.shape[0], codes.shape[1] * 2
    out = np.empty((N, K), np.float64)
    _load().orc_dequant_nvfp4(_ptr(codes), _ptr(scales), float(w["g"]), N, K, _ptr(out))
    return out


def dequant_q45(w: dict) -> np.ndarray:
    q_lo = _c(w["q_lo"], np.uint8)
    q_hi = _c(w.get("q_hi"), np.uint8)
    N, K = q_lo.shape[0], q_lo.shape[1] * 2
    out = np.empty((N, K), np.float64)
    _load().orc_dequant_q45(_ptr(q_lo), _ptr(q_hi), _ptr(_c(w["scale"], np.uint16)),
                            _ptr(_c(w["min"], np.uint16)), int(w["bits"]), N, K, _ptr(out))
    return out


def gemv_nvfp4(w: dict, x, residual=None, threads: int | None = None):
    """y[m][n] = sum_k w[n][k] x[m][k] (+ r[m][n]) in fp64, and sum_k |w x|."""
    codes, scales = _c(w["codes"], np.uint8), _c(w["scales"], np.uint8)
    xx = _c(x, np.uint16)
    r = _c(residual, np.uint16)
    N, K = codes.shape[0], codes.shape[1] * 2
    M = xx.shape[0]
    assert xx.shape == (M, K)
    y = np.empty((M, N), np.float64)
    a = np.empty((M, N), np.float64)
    L = _load()

    def run(n0, n1):
        L.orc_gemv_nvfp4(_ptr(codes), _ptr(scales), float(w["g"]), _ptr(xx), _ptr(r),
                         M, N, K, n0, n1, _ptr(y), _ptr(a))

    _run_ranges(run, N, threads or default_threads())
    return y, a


def gemv_q45(w: dict, x, residual=None, threads: int | None = None):
    q_lo = _c(w["q_lo"], np.uint8)
    q_hi = _c(w.get("q_hi"), np.uint8)
    sc, mn = _c(w["scale"], np.uint16), _c(w["min"], np.uint16)
    xx = _c(x, np.uint16)
    r = _c(residual, np.uint16)
    N, K = q_lo.shape[0], q_lo.shape[1] * 2
    M = xx.shape[0]
    assert xx.shape == (M, K)
    y = np.empty((M, N), np.float64)
    a = np.empty((M, N), np.float64)
    L = _load()

    def run(n0, n1):
        L.orc_gemv_q45(_ptr(q_lo), _ptr(q_hi), _ptr(sc), _ptr(mn), int(w["bits"]), _ptr(xx),
                       _ptr(r), M, N, K, n0, n1, _ptr(y), _ptr(a))

    _run_ranges(run, N, threads or default_threads())
    return y, a


# ---------------------------------------------------------------- MoE
def route_topk(logits, topk: int):
    lg = _c(logits, np.float32)
    M, E = lg.shape
    ids = np.empty((M, topk), np.int32)
    w = np.empty((M, topk), np.float64)
    _load().orc_route_topk(_ptr(lg), M, E, int(topk), _ptr(ids), _ptr(w))
    return ids, w


def moe_gate_up(gu: dict, x, ids, threads: int | None = None):
    """Per (token, slot): gate, up, sum|.| of each, and h = bf16(silu(gate) up)."""
    codes, scales = _c(gu["codes"], np.uint8), _c(gu["scales"], np.uint8)
    g = _c(gu["g"], np.float64)
    E, rows, hh = codes.shape
    H, I = hh * 2, rows // 2
    xx, ii = _c(x, np.uint16), _c(ids, np.int32)
    M, topk = ii.shape
    P = M * topk
    gate = np.empty((M, topk, I), np.float64)
    up = np.empty_like(gate)
    ag = np.empty_like(gate)
    au = np.empty_like(gate)
    h = np.empty((M, topk, I), np.uint16)
    L = _load()

    def run(p0, p1):
        L.orc_moe_gate_up(_ptr(codes), _ptr(scales), _ptr(g), _ptr(xx), _ptr(ii), H, I, topk,
                          p0, p1, _ptr(gate), _ptr(up), _ptr(ag), _ptr(au), _ptr(h))

    _run_ranges(run, P, threads or default_threads())
    return gate, up, ag, au, h


def moe_down(dn: dict, v, ids, w, use_abs: bool = False, threads: int | None = None):
    """y[m][j] = sum_i w[m][i] * (D_{ids[m][i]} v[m][i])[j], slots in order."""
    codes, scales = _c(dn["codes"], np.uint8), _c(dn["scales"], np.uint8)
    g = _c(dn["g"], np.float64)
    E, H, ii2 = codes.shape
    I = ii2 * 2
    vv = _c(v, np.float64)
    ii = _c(ids, np.int32)
    ww = _c(w, np.float64)
    M, topk = ii.shape
    assert vv.shape == (M, topk, I)
    y = np.empty((M, H), np.float64)
    L = _load()

    def run(j0, j1):
        L.orc_moe_down(_ptr(codes), _ptr(scales), _ptr(g), _ptr(vv), _ptr(ii), _ptr(ww), M, H, I,
                       topk, int(bool(use_abs)), j0, j1, _ptr(y))

    _run_ranges(run, H, threads or default_threads())
    return y
