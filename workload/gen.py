"""Seeded synthetic inputs for the verify step.

Everything here is input creation: random master weights, random prompt ids,
random KV contexts, context lengths and draft blocks.  No part of the
verification method (normalisation, projections, attention, quantisation,
argmax, acceptance) is computed here.  The oracle and the CUDA library both
consume these inputs; the greedy continuation used to plant a draft prefix is
passed in by the caller (from whichever model it trusts).

Recipes (stand-ins for the OmniDocBench / OCR workloads the pages measure on,
which are not available here):
  * weights: N(0, 0.02^2), rounded to BF16 -- the "BF16 master";
  * KV context (synthetic case): K, V ~ N(0, sigma^2) in BF16 with
    sigma = 0.02 * sqrt(hidden), the scale of a projection of a unit-RMS row;
  * planted prefix length k: geometric, capped at 16, with the capped mean
    equal to the stated mean (8.9; 7.7 / 8.6 / 10.4 mimic text, formula and
    table pages -- HunyuanOCR-1.5 summary, section two, item 4), or uniform
    on 0..16 for the tiny case;
  * the draft at index k differs from the target's greedy token there, and
    later drafts are uniform random ids.
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch

from .configs import BLOCK, ModelShape, Workload, linear_shapes


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little")


def _rng(*parts) -> np.random.Generator:
    return np.random.default_rng(_seed(*parts))


def normal_bf16(shape, std: float, *seed_parts) -> torch.Tensor:
    """N(0, std^2) samples drawn in float32 and rounded to BF16 (CPU tensor)."""
    a = _rng(*seed_parts).standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(std)
    return torch.from_numpy(a).to(torch.bfloat16)


def master_tensor(shape: ModelShape, seed: int, layer: int | None, name: str) -> torch.Tensor:
    """One BF16 master weight matrix [out, in] of the random-init target."""
    if name == "embed":
        dims = (shape.vocab, shape.hidden)
    elif name == "lm_head":
        dims = (shape.vocab, shape.hidden)
    else:
        n, k, _ = linear_shapes(shape)[name]
        dims = (n, k)
    return normal_bf16(dims, shape.init_std, "w", seed, layer, name)


def master_weights(shape: ModelShape, seed: int, layers=None) -> dict:
    """All BF16 master weights: {'embed', 'lm_head' (untied only), 'layers': [dict]}."""
    layers = range(shape.layers) if layers is None else layers
    out = {"embed": master_tensor(shape, seed, None, "embed"), "layers": {}}
    if not shape.tied:
        out["lm_head"] = master_tensor(shape, seed, None, "lm_head")
    for l in layers:
        out["layers"][l] = {n: master_tensor(shape, seed, l, n) for n in linear_shapes(shape)}
    return out


def context_lengths(w: Workload) -> np.ndarray:
    r = _rng("ctx", w.seed)
    return r.integers(w.ctx_lo, w.ctx_hi + 1, size=w.batch).astype(np.int32)


def prompt_ids(vocab: int, n: int, seed: int, req: int) -> np.ndarray:
    return _rng("prompt", seed, req).integers(0, vocab, size=n).astype(np.int32)


def pending_tokens(w: Workload) -> np.ndarray:
    """Last emitted token per request for a synthetic context (uniform ids)."""
    return _rng("pending", w.seed).integers(0, w.shape.vocab, size=w.batch).astype(np.int32)


def synthetic_kv(shape: ModelShape, length: int, seed: int, req: int):
    """Random BF16 K and V for one request: two tensors [layers, length, n_kv, head_dim]."""
    std = shape.init_std * float(np.sqrt(shape.hidden))
    dims = (shape.layers, length, shape.n_kv, shape.head_dim)
    return (normal_bf16(dims, std, "kv", seed, req, "k"),
            normal_bf16(dims, std, "kv", seed, req, "v"))


def geometric_ratio_for_capped_mean(mean: float, cap: int = BLOCK) -> float:
    """Ratio q with sum_{j=1..cap} q^j == mean (P(k >= j) = q^j, k capped at cap)."""
    if not 0.0 < mean < cap:
        raise ValueError("mean must lie strictly between 0 and the cap")
    lo, hi = 0.0, 1.0 - 1e-15
    for _ in range(200):
        q = 0.5 * (lo + hi)
        s = sum(q ** j for j in range(1, cap + 1))
        lo, hi = (q, hi) if s < mean else (lo, q)
    return 0.5 * (lo + hi)


def prefix_lengths(w: Workload, step: int = 0) -> np.ndarray:
    """Planted prefix length k per request for one step (k in 0..16)."""
    r = _rng("k", w.seed, step)
    if w.draft_dist == "uniform":
        return r.integers(0, BLOCK + 1, size=w.batch).astype(np.int32)
    means = [w.draft_means[b % len(w.draft_means)] for b in range(w.batch)]
    ks = np.empty(w.batch, np.int32)
    u = r.random(size=(w.batch, BLOCK))
    for b, m in enumerate(means):
        q = geometric_ratio_for_capped_mean(m)
        k = 0
        while k < BLOCK and u[b, k] < q:   # survive step k+1 with probability q
            k += 1
        ks[b] = k
    return ks


def plant_drafts(greedy: np.ndarray, k: int, vocab: int, *seed_parts) -> np.ndarray:
    """A 16-token draft block whose first k tokens are `greedy[:k]`.

    `greedy` holds the target's own greedy continuation (at least k+1 tokens
    when k < 16).  Index k is redrawn until it differs from greedy[k] so that
    exactly k drafts match; indices past k are uniform random ids.
    """
    r = _rng("draft", *seed_parts)
    d = r.integers(0, vocab, size=BLOCK).astype(np.int32)
    d[:k] = np.asarray(greedy[:k], np.int32)
    if k < BLOCK:
        while d[k] == greedy[k]:
            d[k] = r.integers(0, vocab)
    return d


def page_table(w: Workload, pages_per_req: int) -> np.ndarray:
    """Page table [batch, pages_per_req]: identity, or a seeded shuffle when paged."""
    n = w.batch * pages_per_req
    perm = np.arange(n, dtype=np.int32)
    if w.paged:
        perm = _rng("pages", w.seed).permutation(n).astype(np.int32)
    return perm.reshape(w.batch, pages_per_req)


def drafter_master(master: dict, target_layers: int, drafter_layers: int) -> dict:
    """The drafter's master weights: the target's embedding (and head) and its last layers, renumbered."""
    first = target_layers - drafter_layers
    out = {"embed": master["embed"], "layers": {i: master["layers"][first + i] for i in range(drafter_layers)}}
    if "lm_head" in master:
        out["lm_head"] = master["lm_head"]
    return out


def anchor_rows(hidden: int, batch: int, seed: int) -> torch.Tensor:
    """Synthetic drafter anchors [batch, hidden] float32: unit-RMS Gaussian rows (a residual row's scale)."""
    r = _rng("anchor", seed, hidden, batch)
    return torch.from_numpy(r.standard_normal((batch, hidden)).astype(np.float32))
