"""Test glue that turns seeded workload inputs into oracle inputs.

Used only by tests (and the smoke / CPU-baseline code paths); it calls the
oracle's own quantisers, never the CUDA library.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import model as OM
from oracle import weights as OW
from workload import gen, linear_shapes


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 CPU tensor -> uint16 bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_model(shape, master: dict) -> OM.Model:
    layers = {}
    for l, mats in master["layers"].items():
        layers[l] = {n: OW.canonical_entry(OW.fmt_of(shape, n), bits(mats[n])) for n in mats}
    lm = None if shape.tied else OW.canonical_entry("bf16", bits(master["lm_head"]))
    return OM.Model(shape, bits(master["embed"]), layers, lm)


def oracle_state_from_kv(shape, k: torch.Tensor, v: torch.Tensor, pending: int) -> OM.RequestState:
    """BF16 K, V [layers, L, n_kv, d] -> oracle request state (exact values)."""
    kk = [bits(k[l]).astype(np.uint32) << 16 for l in range(shape.layers)]
    vv = [bits(v[l]).astype(np.uint32) << 16 for l in range(shape.layers)]
    kk = [a.view(np.float32).astype(np.float64) for a in kk]
    vv = [a.view(np.float32).astype(np.float64) for a in vv]
    return OM.RequestState(shape.layers, shape.n_kv, shape.head_dim, kk, vv, pending)


def near_tie_check(oracle_res: dict, acc_gpu: int, out_gpu, tol: float = 1e-3):
    """Compare one request's GPU accept/output with the oracle under the
    near-tie exemption: rows whose oracle top-2 logit gap is below `tol` may
    pick either token; everything before the first such row must match
    exactly.  Returns (ok, first_near_tie_row or None)."""
    a_o = int(oracle_res["accepted"])
    out_o = np.asarray(oracle_res["out"])
    out_gpu = np.asarray(out_gpu)
    gaps = np.asarray(oracle_res["top2_gap"])
    ties = np.flatnonzero(gaps[: a_o + 1] < tol)
    if len(ties) == 0:
        return (acc_gpu == a_o and np.array_equal(out_gpu, out_o)), None
    j = int(ties[0])
    ok = np.array_equal(out_gpu[:j], out_o[:j]) and acc_gpu >= j
    return ok, j
