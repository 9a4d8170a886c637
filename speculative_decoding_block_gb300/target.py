"""Builds the library's model object from BF16 master weights.

Uploads each master matrix, quantises it on the GPU with the library's own
round-to-nearest kernels (FP8 per-channel or NVFP4, as the shape's format
says), and hands the canonical bytes to vsd_model_create, which repacks
them into the GEMM tile layout.  Argument marshalling only.
"""
from __future__ import annotations

import torch

from . import binding as B

LAYER_NAMES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def model_config(shape, max_positions: int) -> B.ModelConfig:
    return B.ModelConfig(shape.layers, shape.hidden, shape.n_q, shape.n_kv, shape.head_dim, shape.ffn,
                         shape.vocab, float(shape.rope_theta), float(shape.eps), 1 if shape.tied else 0,
                         B.FMT[shape.attn_fmt], B.FMT[shape.mlp_fmt], int(max_positions))


def quantize(fmt: str, w_dev: torch.Tensor) -> dict:
    """Canonical entry of one BF16 matrix [N, K] on the device."""
    n, k = w_dev.shape
    if fmt == "bf16":
        return {"fmt": "bf16", "w": w_dev}
    if fmt == "fp8":
        q = torch.empty((n, k), dtype=torch.uint8, device=w_dev.device)
        s = torch.empty((n,), dtype=torch.float32, device=w_dev.device)
        B.vsd_quantize_fp8_rowwise(w_dev, q, s)
        return {"fmt": "fp8", "q": q, "s": s}
    if fmt == "nvfp4":
        q = torch.empty((n, k // 2), dtype=torch.uint8, device=w_dev.device)
        sb = torch.empty((n, k // 16), dtype=torch.uint8, device=w_dev.device)
        S = torch.empty((1,), dtype=torch.float32, device=w_dev.device)
        B.vsd_quantize_nvfp4(w_dev, q, sb, S)
        return {"fmt": "nvfp4", "q": q, "sb": sb, "S": S}
    raise ValueError(fmt)


def weight_of(entry: dict) -> B.Weight:
    if entry["fmt"] == "bf16":
        return B.weight_entry("bf16", entry["w"])
    if entry["fmt"] == "fp8":
        return B.weight_entry("fp8", entry["q"], entry["s"])
    return B.weight_entry("nvfp4", entry["q"], entry["sb"], entry["S"])


def build_target(shape, master: dict, max_positions: int, device="cuda", keep_canonical=False):
    """Returns (model, canonical) -- canonical is {layer: {name: entry}} when kept, else {}."""
    embed = master["embed"].to(device)
    lm = master["lm_head"].to(device) if not shape.tied else None
    weights, keep, canonical = [], [], {}
    for l in range(shape.layers):
        mats = master["layers"][l]
        canonical[l] = {}
        for name in LAYER_NAMES:
            fmt = shape.attn_fmt if name in ("wq", "wk", "wv", "wo") else shape.mlp_fmt
            e = quantize(fmt, mats[name].to(device))
            keep.append(e)
            canonical[l][name] = e
            weights.append(weight_of(e))
    model = B.vsd_model_create(model_config(shape, max_positions), embed, weights, lm_head=lm)
    del embed, lm, keep
    return model, (canonical if keep_canonical else {})
