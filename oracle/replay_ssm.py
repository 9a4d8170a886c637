"""Float64 ReplaySSM-style verification and rollback of a recurrent layer.

TEST INFRASTRUCTURE: part of the CPU oracle (see oracle/__init__.py).

What the pages fix ("The Inference Stack Behind OCRia", section "Make
speculative verification cheaper"): GDN layers keep a fixed-size recurrent
state instead of a KV cache; under speculative decoding the state is kept as
a checkpoint plus a small buffer of recent inputs; outputs are computed from
the checkpoint and the buffered inputs; the full checkpoint is updated only
at periodic flushes; when drafted tokens are rejected, rollback moves the
buffer pointer so that only the accepted prefix is retained.

Readings (the pages give no update rule):
* The recurrence is the gated delta rule of Gated DeltaNet, per head with
  state S (d_v x d_k), and per token inputs q, k (d_k), v (d_v), a gate
  alpha in (0, 1] and a write strength beta in [0, 1]:
      S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
      o_t = S_t q_t.
* A verify step covers the 17 rows of a block (the pending token and the
  16 drafts).  Row t's output is S after the buffered tokens and rows
  0..t, applied to q_t; the block's inputs go into the buffer after the
  pointer, tentatively.
* The commit of a step moves the pointer past the accepted rows (a + 1 of
  them; a rejected request, a = -1, keeps its pointer).  A flush folds the
  buffered inputs into the checkpoint and empties the buffer; it runs at
  commit time when the next block would not fit (pointer + 17 > window).
"""
from __future__ import annotations

import numpy as np

ROWS = 17  # a verify block: the pending token and 16 drafts


def gdn_update(S: np.ndarray, k: np.ndarray, v: np.ndarray, alpha: float, beta: float) -> np.ndarray:
    """One gated delta rule update: alpha * S (I - beta k k^T) + beta v k^T."""
    d_k = S.shape[1]
    return alpha * (S @ (np.eye(d_k) - beta * np.outer(k, k))) + beta * np.outer(v, k)


def run_tokens(S: np.ndarray, ks, vs, alphas, betas) -> np.ndarray:
    """The state after the given tokens, in order."""
    S = np.array(S, np.float64)
    for k, v, a, b in zip(ks, vs, alphas, betas):
        S = gdn_update(S, k, v, a, b)
    return S


class ReplayState:
    """One request's recurrent state of one head, as checkpoint + input buffer."""

    def __init__(self, S0: np.ndarray, window: int):
        if window < ROWS:
            raise ValueError("the buffer must hold a block")
        self.ckpt = np.array(S0, np.float64)
        self.window = window
        d_v, d_k = self.ckpt.shape
        self.k = np.zeros((window, d_k))
        self.v = np.zeros((window, d_v))
        self.alpha = np.zeros(window)
        self.beta = np.zeros(window)
        self.ptr = 0

    def state(self) -> np.ndarray:
        """The effective state: the checkpoint replayed through the retained buffer."""
        n = self.ptr
        return run_tokens(self.ckpt, self.k[:n], self.v[:n], self.alpha[:n], self.beta[:n])

    def verify(self, q, k, v, alpha, beta) -> np.ndarray:
        """Outputs [17, d_v] of a block; its inputs are staged after the pointer."""
        q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
        alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
        if len(q) != ROWS or self.ptr + ROWS > self.window:
            raise ValueError("a block of 17 rows that fits the buffer")
        S = self.state()
        out = np.empty((ROWS, self.ckpt.shape[0]))
        for t in range(ROWS):
            S = gdn_update(S, k[t], v[t], alpha[t], beta[t])
            out[t] = S @ q[t]
        sl = slice(self.ptr, self.ptr + ROWS)
        self.k[sl], self.v[sl], self.alpha[sl], self.beta[sl] = k, v, alpha, beta
        return out

    def commit(self, accepted: int) -> bool:
        """Rollback by pointer: keep rows 0..accepted of the staged block
        (accepted = -1: none).  Then flush when the next block would not fit.
        Returns whether it flushed."""
        if accepted < -1 or accepted >= ROWS:
            raise ValueError("accepted in [-1, 16]")
        self.ptr += accepted + 1
        if self.ptr + ROWS > self.window:
            self.ckpt = self.state()
            self.ptr = 0
            return True
        return False
