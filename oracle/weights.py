"""Canonical weight entries built from BF16 master weights by the oracle's quantisers.

TEST INFRASTRUCTURE: part of the float64 CPU oracle (see oracle/__init__.py).

Formats per matrix group follow the mixed-precision recipe ("The Inference
Stack Behind OCRia", section "Reducing the data moved"): attention
projections in FP8 E4M3 with per-output-channel scales, MLP projections in
NVFP4, embeddings / lm_head in BF16 -- or everything BF16.
"""
from __future__ import annotations

import numpy as np

from . import quant
from .formats import bf16_bits_to_f64


def canonical_entry(fmt: str, bits: np.ndarray) -> dict:
    """BF16 master bits [N, K] (uint16) -> canonical entry in format `fmt`."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if fmt == "bf16":
        return {"fmt": "bf16", "w": bits}
    w = bf16_bits_to_f64(bits)
    if fmt == "fp8":
        q, s = quant.quantize_fp8_rowwise(w)
        return {"fmt": "fp8", "q": q, "s": s}
    if fmt == "nvfp4":
        q, sb, S = quant.quantize_nvfp4(w)
        return {"fmt": "nvfp4", "q": q, "sb": sb, "S": S}
    raise ValueError(f"unknown weight format {fmt!r}")


LAYER_FMT = {"wq": "attn", "wk": "attn", "wv": "attn", "wo": "attn",
             "wg": "mlp", "wu": "mlp", "wd": "mlp"}


def fmt_of(shape, name: str) -> str:
    return shape.attn_fmt if LAYER_FMT[name] == "attn" else shape.mlp_fmt
