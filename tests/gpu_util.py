"""Helpers for the GPU tests: move seeded host inputs to the device and back."""
from __future__ import annotations

import numpy as np


def dev():
    import torch
    return torch.device("cuda", 0)


def to_dev(a, dtype=None):
    """numpy array -> contiguous CUDA tensor with the same bytes."""
    import torch
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.int16)
        t = t.view(torch.bfloat16) if dtype is None else t.view(dtype)
    elif a.dtype == np.uint8:
        t = torch.from_numpy(a)
    else:
        t = torch.from_numpy(a)
    return t.to(dev())


def bits16(t) -> np.ndarray:
    """bf16/fp16 CUDA tensor -> uint16 bit patterns on the host."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def nvfp4_dev(w: dict) -> dict:
    return {"codes": to_dev(w["codes"]), "scales": to_dev(w["scales"]), "g": float(w["g"])}


def q45_dev(w: dict) -> dict:
    import torch
    return {"q_lo": to_dev(w["q_lo"]), "q_hi": to_dev(w.get("q_hi")),
            "scale": to_dev(w["scale"], torch.float16), "min": to_dev(w["min"], torch.float16),
            "bits": int(w["bits"])}


def guarded(shape, dtype, fill_byte=0x5A, pad=4096):
    """A tensor of `shape` inside a larger buffer whose padding holds a
    sentinel byte pattern; returns (view, check_fn) where check_fn() asserts
    the padding is untouched."""
    import torch
    n = int(np.prod(shape))
    elt = torch.empty(0, dtype=dtype).element_size()
    pad_elems = (pad + elt - 1) // elt
    raw = torch.full(((n + 2 * pad_elems) * elt,), fill_byte, dtype=torch.uint8, device=dev())
    base = raw.view(dtype)
    view = base[pad_elems:pad_elems + n].view(shape)

    def check():
        host = raw.cpu().numpy()
        assert (host[:pad_elems * elt] == fill_byte).all(), "write before the output buffer"
        assert (host[(pad_elems + n) * elt:] == fill_byte).all(), "write past the output buffer"

    return view, check
