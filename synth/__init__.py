"""Seeded synthetic inputs for the quantised decode GEMV workloads.

This module is shared by the tests, the benchmark and the smoke check. It only
draws random numbers and stores them in the packed layouts the library reads;
it holds none of the method's arithmetic (no decode, no dot product, no
epilogue). Rounding a drawn real number to a storage type (bf16, fp16,
FP8-E4M3) is delegated to library conversions (torch / numpy), which round to
nearest even.

Value recipe (the pages name the formats -- NInfer article, section 2
"自研 CUDA 算子 混合量化权重"; Decapybara README, "Blackwell CUDA 内核套件"
(mx_gemv.cu, moe.cu) -- but print no data, so these distributions are the
library's stated synthetic workload):

* activations x and residual r: bf16(N(0, 1));
* NVFP4 codes: every nibble uniform over the 16 E2M1 codes (two per byte,
  low nibble = even k), one E4M3 scale per 16 weights equal to
  e4m3(2^U(-4, 2)), global FP32 scale 1.0;
* Q4/Q5 codes: q uniform over [0, 2^bits), fp16 scale = f16(U(0.002, 0.02)),
  fp16 min = f16(N(0, 0.05)) per group of 32 along K; Q5 stores the low
  4 bits as nibbles and the 5th bit as a separate LSB-first bit plane;
* router logits: fp32 N(0, 1).

Every tensor has its own stream, keyed by (seed, name), so a tensor can be
regenerated alone.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import numpy as np

__all__ = [
    "rng_for", "bf16_normal", "nvfp4_weights", "q45_weights", "router_logits",
    "TINY", "DENSE27B", "MOE35B", "SWEEP_M", "Q45_RECIPE", "dense_layer_shapes",
]


# --------------------------------------------------------------------------
# workload shapes (data only)
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Tiny:
    M: int = 1
    N: int = 256
    K: int = 512


@dataclass(frozen=True)
class Dense27B:
    hidden: int = 5120
    qkv_n: int = 7168      # fused Q|K|V output rows
    q_rows: int = 6144     # Q part of the fused projection (matches O's K)
    k_rows: int = 512
    v_rows: int = 512
    o_k: int = 6144
    inter: int = 17408     # FFN intermediate size I (gate+up has 2I rows)


@dataclass(frozen=True)
class Moe35B:
    M: int = 8
    hidden: int = 2048
    experts: int = 128
    inter: int = 768
    topk: int = 8


TINY = Tiny()
DENSE27B = Dense27B()
MOE35B = Moe35B()
SWEEP_M = (1, 2, 4, 8)


def dense_layer_shapes(d: Dense27B = DENSE27B):
    """(name, N, K, epilogue) of the four projections of one dense layer."""
    return [
        ("qkv", d.qkv_n, d.hidden, "none"),
        ("o", d.hidden, d.o_k, "none"),
        ("gate_up", 2 * d.inter, d.hidden, "swiglu"),
        ("down", d.hidden, d.inter, "residual"),
    ]


# Mixed groupwise-int recipe on the dense shapes: (name, N, K, bits).
# Q and K rows of the fused projection are Q4, V rows Q5, gate Q5, up Q4,
# O and down Q4.
Q45_RECIPE = (
    ("qk", DENSE27B.q_rows + DENSE27B.k_rows, DENSE27B.hidden, 4),
    ("v", DENSE27B.v_rows, DENSE27B.hidden, 5),
    ("o", DENSE27B.hidden, DENSE27B.o_k, 4),
    ("gate", DENSE27B.inter, DENSE27B.hidden, 5),
    ("up", DENSE27B.inter, DENSE27B.hidden, 4),
    ("down", DENSE27B.hidden, DENSE27B.inter, 4),
)


# --------------------------------------------------------------------------
# random streams
# --------------------------------------------------------------------------
def rng_for(seed: int, name: str) -> np.random.Generator:
    """Independent PCG64 stream for tensor `name` under `seed`."""
    key = zlib.crc32(name.encode("utf-8"))
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), key])))


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def _to_f16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64).astype(np.float16).view(np.uint16).copy()


def bf16_normal(seed: int, name: str, shape) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0, 1) draws."""
    return _to_bf16_bits(rng_for(seed, name).standard_normal(shape, dtype=np.float32))


def nvfp4_weights(seed: int, name: str, N: int, K: int, g: float = 1.0) -> dict:
    """Packed NVFP4 weights: codes u8[N][K/2], e4m3 scales u8[N][K/16], g."""
    assert K % 16 == 0
    codes = rng_for(seed, name + ".codes").integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    u = rng_for(seed, name + ".scales").uniform(-4.0, 2.0, size=(N, K // 16))
    scales = _to_e4m3_bits(np.exp2(u))
    # the per-tensor scale is an FP32 value: store exactly what the kernel gets
    return {"codes": codes, "scales": scales, "g": float(np.float32(g)), "N": N, "K": K}


def q45_weights(seed: int, name: str, N: int, K: int, bits: int) -> dict:
    """Packed groupwise-int weights.

    q_lo u8[N][K/2] (low nibble = even k), q_hi u8[N][K/8] (bit k%8 of byte
    k/8, Q5 only, else None), scale/min fp16 bit patterns u16[N][K/32].
    """
    assert K % 32 == 0 and bits in (4, 5)
    q_lo = rng_for(seed, name + ".q_lo").integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    q_hi = None
    if bits == 5:
        q_hi = rng_for(seed, name + ".q_hi").integers(0, 256, size=(N, K // 8), dtype=np.uint8)
    scale = _to_f16_bits(rng_for(seed, name + ".scale").uniform(0.002, 0.02, size=(N, K // 32)))
    mn = _to_f16_bits(rng_for(seed, name + ".min").normal(0.0, 0.05, size=(N, K // 32)))
    return {"q_lo": q_lo, "q_hi": q_hi, "scale": scale, "min": mn, "bits": bits, "N": N, "K": K}


def router_logits(seed: int, name: str, M: int, E: int) -> np.ndarray:
    return rng_for(seed, name).standard_normal((M, E), dtype=np.float32)
