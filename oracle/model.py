"""Float64 forward of the decoder-only target and the greedy block-verify step.

TEST INFRASTRUCTURE: part of the float64 CPU oracle (see oracle/__init__.py).

What is computed, and where the pages fix it:
  * one target pass checks a whole drafted block (16 tokens) at once --
    "The Inference Stack Behind OCRia", section "Generate more tokens per
    target pass: speculative decoding"; HunyuanOCR-1.5 summary, section one,
    inference steps 2-3;
  * the accepted part is the longest prefix that matches the target's own
    choice, cut at the first mismatch from the left, and one target token is
    appended (the correction, or the bonus when all drafts match) --
    HunyuanOCR-1.5 summary, section one, inference step 4; the accept /
    correct / bonus branch of the speculative decoder in "LLM inference
    acceleration", section 3.2;
  * the result equals the target's own greedy output ("100% lossless") --
    OCRia post, speculative-decoding section;
  * previous tokens are not recomputed: their K and V sit in a cache --
    OCRia post, speculative-decoding section;
  * GQA, query heads share KV heads -- "LLM inference acceleration",
    section two.
Readings where the pages are silent (all listed in the design notes):
  * 17 rows per request: the pending token (last emitted token, not yet in
    the cache) followed by the 16 drafts, at positions L .. L+16;
  * pre-norm decoder layer, RMSNorm (gamma = 1, eps = 1e-6), no biases,
    rotate-half RoPE with inv_freq_i = theta^(-2i/head_dim), query head h
    reads KV head floor(h / group), SwiGLU MLP silu(x Wg^T) * (x Wu^T) Wd^T,
    final RMSNorm, tied or untied lm_head;
  * the KV cache holds BF16: every K and V row is rounded to BF16 (nearest,
    ties to even) where it is produced, and attention reads those values;
  * argmax ties go to the lowest token id;
  * commit writes rows 0..a (pending + accepted drafts) at positions
    L .. L+a; nothing else in the cache changes.
All arithmetic is float64; weights are the exact dequantised values.
"""
from __future__ import annotations

import numpy as np

from . import quant
from .formats import bf16_bits_to_f64, round_to_bf16

BLOCK = 16


# ------------------------------------------------------------------ weights
def dequantize(entry: dict) -> np.ndarray:
    """Canonical weight entry -> float64 [N, K].

    {'fmt': 'bf16', 'w': uint16 [N, K]}
    {'fmt': 'fp8', 'q': uint8 [N, K], 's': float32 [N]}
    {'fmt': 'nvfp4', 'q': uint8 [N, K/2], 'sb': uint8 [N, K/16], 'S': float32}
    """
    f = entry["fmt"]
    if f == "bf16":
        return bf16_bits_to_f64(entry["w"])
    if f == "fp8":
        return quant.dequantize_fp8_rowwise(entry["q"], entry["s"])
    if f == "nvfp4":
        return quant.dequantize_nvfp4(entry["q"], entry["sb"], entry["S"])
    raise ValueError(f"unknown weight format {f!r}")


class Model:
    """Float64 target: shape + canonical weights, dequantised on first use."""

    def __init__(self, shape, embed_bits, layers, lm_head=None):
        self.shape = shape
        self.embed = bf16_bits_to_f64(embed_bits)
        self._layers = layers              # {layer: {name: canonical entry}}
        self._lm_head = lm_head
        self._cache: dict = {}

    def w(self, layer: int, name: str) -> np.ndarray:
        key = (layer, name)
        if key not in self._cache:
            self._cache[key] = dequantize(self._layers[layer][name])
        return self._cache[key]

    def lm_head(self) -> np.ndarray:
        if self.shape.tied:
            return self.embed
        if "lm" not in self._cache:
            self._cache["lm"] = dequantize(self._lm_head)
        return self._cache["lm"]

    def drop_layer(self, layer: int) -> None:
        for name in list(self._layers[layer]):
            self._cache.pop((layer, name), None)


# ------------------------------------------------------------------ pieces
def rmsnorm(x: np.ndarray, eps: float, gamma=None) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gamma, over the last axis."""
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return y if gamma is None else y * gamma


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE of x [rows, heads, d] at integer positions pos [rows].

    Pair (i, i + d/2) rotates by angle pos * theta^(-2i/d).
    """
    d = x.shape[-1]
    half = d // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / d)
    ang = pos.astype(np.float64)[:, None] * inv_freq[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def softmax(s: np.ndarray) -> np.ndarray:
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    return e / np.sum(e, axis=-1, keepdims=True)


def block_attention(q, K, V, ctx_len: int, group: int) -> np.ndarray:
    """GQA attention of a block of rows over cached keys plus the block's own keys.

    q [R, n_q, d]; K, V [ctx_len + R, n_kv, d] (cache rows first, then the
    block rows).  Block row j sees keys t <= ctx_len + j.  Returns [R, n_q, d].
    """
    R, n_q, d = q.shape
    T = K.shape[0]
    visible = np.arange(T)[None, :] <= (ctx_len + np.arange(R))[:, None]
    out = np.empty_like(q)
    for h in range(n_q):
        kvh = h // group
        s = (q[:, h, :] @ K[:, kvh, :].T) / np.sqrt(d)
        s = np.where(visible, s, -np.inf)
        out[:, h, :] = softmax(s) @ V[:, kvh, :]
    return out


# ------------------------------------------------------------------ forward
def forward_block(m: Model, kc, vc, ctx_len: int, tokens, keep_hidden=False):
    """Run rows `tokens` at positions ctx_len.. through the target.

    kc, vc: per layer arrays [>= ctx_len, n_kv, d] of cached (BF16-valued) K, V.
    Returns dict with logits [R, V], new_k / new_v (per layer [R, n_kv, d],
    BF16-rounded) and, if asked, hidden (list of [R, H], entry 0 = embeddings,
    entry l+1 = residual stream after layer l).
    """
    tokens = np.asarray(tokens, np.int64)
    return forward_rows(m, kc, vc, ctx_len, m.embed[tokens], ctx_len + np.arange(len(tokens)), keep_hidden)


def forward_rows(m: Model, kc, vc, ctx_len: int, rows, pos, keep_hidden=False):
    """forward_block on given input rows [R, H] (the residual stream before
    layer 0) at given positions pos [R]; block row j sees the ctx_len cached
    rows and block rows 0..j."""
    s = m.shape
    h = np.array(rows, np.float64)
    R = h.shape[0]
    pos = np.asarray(pos, np.int64)
    hidden = [h.copy()] if keep_hidden else None
    new_k, new_v = [], []
    for l in range(s.layers):
        u = rmsnorm(h, s.eps)
        q = (u @ m.w(l, "wq").T).reshape(R, s.n_q, s.head_dim)
        k = (u @ m.w(l, "wk").T).reshape(R, s.n_kv, s.head_dim)
        v = (u @ m.w(l, "wv").T).reshape(R, s.n_kv, s.head_dim)
        q = rope(q, pos, s.rope_theta)
        k = round_to_bf16(rope(k, pos, s.rope_theta))
        v = round_to_bf16(v)
        K = np.concatenate([kc[l][:ctx_len], k], axis=0)
        V = np.concatenate([vc[l][:ctx_len], v], axis=0)
        a = block_attention(q, K, V, ctx_len, s.group).reshape(R, s.n_q * s.head_dim)
        h = h + a @ m.w(l, "wo").T
        x = rmsnorm(h, s.eps)
        h = h + (silu(x @ m.w(l, "wg").T) * (x @ m.w(l, "wu").T)) @ m.w(l, "wd").T
        new_k.append(k)
        new_v.append(v)
        if keep_hidden:
            hidden.append(h.copy())
    logits = rmsnorm(h, s.eps) @ m.lm_head().T
    return {"logits": logits, "new_k": new_k, "new_v": new_v, "hidden": hidden}


def greedy(logits: np.ndarray) -> np.ndarray:
    """Per-row argmax; ties resolve to the lowest token id."""
    return np.argmax(logits, axis=-1).astype(np.int64)


def accept_length(drafts, greedy_tokens) -> int:
    """Index of the first draft that differs from the target's greedy token, or 16."""
    for i in range(BLOCK):
        if int(drafts[i]) != int(greedy_tokens[i]):
            return i
    return BLOCK


# ------------------------------------------------------------------ state
class RequestState:
    """One request: BF16-valued KV rows per layer, committed length, pending token."""

    def __init__(self, layers: int, n_kv: int, d: int, k=None, v=None, pending: int = 0):
        if k is None:
            k = [np.zeros((0, n_kv, d)) for _ in range(layers)]
            v = [np.zeros((0, n_kv, d)) for _ in range(layers)]
        self.k = [np.asarray(a, np.float64) for a in k]
        self.v = [np.asarray(a, np.float64) for a in v]
        self.pending = int(pending)

    @property
    def length(self) -> int:
        return self.k[0].shape[0]

    def commit(self, new_k, new_v, rows: int) -> None:
        self.k = [np.concatenate([a, b[:rows]], axis=0) for a, b in zip(self.k, new_k)]
        self.v = [np.concatenate([a, b[:rows]], axis=0) for a, b in zip(self.v, new_v)]

    def copy(self) -> "RequestState":
        return RequestState(len(self.k), 0, 0, [a.copy() for a in self.k],
                            [a.copy() for a in self.v], self.pending)


def prefill(m: Model, prompt) -> RequestState:
    """Process the prompt rows causally, cache their K/V, pending = greedy next token."""
    s = m.shape
    st = RequestState(s.layers, s.n_kv, s.head_dim)
    r = forward_block(m, st.k, st.v, 0, prompt)
    st.commit(r["new_k"], r["new_v"], len(prompt))
    st.pending = int(greedy(r["logits"][-1:])[0])
    return st


def ar_step(m: Model, st: RequestState) -> int:
    """Plain autoregressive greedy step: run the pending row, commit it, return the next token."""
    r = forward_block(m, st.k, st.v, st.length, [st.pending])
    g = int(greedy(r["logits"])[0])
    st.commit(r["new_k"], r["new_v"], 1)
    st.pending = g
    return g


def ar_greedy(m: Model, st: RequestState, n: int) -> np.ndarray:
    """n greedy tokens continuing the request (state advanced in place)."""
    return np.array([ar_step(m, st) for _ in range(n)], np.int64)


def verify_step(m: Model, st: RequestState, drafts, keep_hidden=False) -> dict:
    """Greedy block verification of 16 drafts; commits the accepted rows in place.

    Rows are [pending, d_0 .. d_15] at positions L .. L+16.  Row j's greedy
    token g_j is the target's choice after that row.  a = first i with
    d_i != g_i (16 if none); the output is g_0 .. g_a (a+1 tokens, -1 padded
    to 17); rows 0..a are committed and the pending token becomes g_a.
    """
    drafts = np.asarray(drafts, np.int64)
    if drafts.shape != (BLOCK,):
        raise ValueError("a draft block has 16 tokens")
    L = st.length
    rows = np.concatenate([[st.pending], drafts])
    r = forward_block(m, st.k, st.v, L, rows, keep_hidden=keep_hidden)
    g = greedy(r["logits"])
    a = accept_length(drafts, g)
    out = np.full(BLOCK + 1, -1, np.int64)
    out[: a + 1] = g[: a + 1]
    st.commit(r["new_k"], r["new_v"], a + 1)
    st.pending = int(g[a])
    srt = np.sort(r["logits"], axis=-1)
    res = {"accepted": a, "out": out, "greedy": g, "logits": r["logits"],
           "top2_gap": srt[:, -1] - srt[:, -2], "new_k": r["new_k"],
           "new_v": r["new_v"], "hidden": r["hidden"], "ctx_len": L}
    if keep_hidden:  # the drafter's next conditioning row: last layer's residual at row a
        res["anchor"] = r["hidden"][-1][a].copy()
    return res


# ------------------------------------------------------------------ drafting
def draft_step(d: Model, anchor, seq_len: int, mask_token: int, keep_hidden=False) -> dict:
    """One pass of the block drafter over one request.

    The pages: the DFlash drafter is a small transformer (5 layers,
    initialised from the target's last five decoder layers) that takes the
    target's hidden state at the anchor and proposes a whole block of 16
    tokens in one forward pass -- HunyuanOCR-1.5 summary, section one; one
    drafter pass per drafted block -- "The Inference Stack Behind OCRia",
    speculative-decoding section.  Readings (the pages give no layer-level
    detail): input rows [anchor, E[mask] x 16] at positions seq_len ..
    seq_len+16, where anchor is the target's residual row (before the final
    norm) at the last accepted position; the drafter's layers are the
    target's kind of decoder layer; attention is causal among the 17 rows
    with no cache; draft j = argmax of row 1+j of the head (ties to the
    lowest id).  Returns drafts [16], logits [17, V] and, if asked, hidden.
    """
    s = d.shape
    anchor = np.asarray(anchor, np.float64).reshape(1, s.hidden)
    rows = np.concatenate([anchor, np.repeat(d.embed[[int(mask_token)]], BLOCK, axis=0)], axis=0)
    empty = [np.zeros((0, s.n_kv, s.head_dim)) for _ in range(s.layers)]
    r = forward_rows(d, empty, empty, 0, rows, seq_len + np.arange(BLOCK + 1), keep_hidden=keep_hidden)
    srt = np.sort(r["logits"], axis=-1)
    return {"drafts": greedy(r["logits"][1:]), "logits": r["logits"], "hidden": r["hidden"],
            "top2_gap": srt[:, -1] - srt[:, -2]}
