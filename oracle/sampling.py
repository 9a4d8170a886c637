"""Float64 stochastic block verification (temperature sampling), one request.

TEST INFRASTRUCTURE: part of the CPU oracle (see oracle/__init__.py).

What the pages fix: verification with the correct procedure keeps the
accepted tokens distributed as the target's own output ("The Inference
Stack Behind OCRia", speculative-decoding section: "100% lossless"); the
serving code they print samples at temperature 0.7 and, after the accepted
drafts, emits a correction at the first rejection or a bonus token when all
drafts pass ("LLM inference acceleration", section 3.2, speculative
decoder).  The acceptance rule itself is not on the pages; it is the
standard speculative-sampling rule of the literature for a drafter that
proposes single tokens (its distribution q is a point mass on the draft):
draft d at row j is accepted with probability min(1, p_j(d) / q(d)) =
p_j(d), where p_j = softmax(logits_j / T); at the first rejection the
output is a sample of p_j with d removed and renormalised (max(0, p - q)
normalised); after 16 acceptances the bonus is a sample of p_16.
Readings: the random numbers are inputs -- u_accept[j] for the accept test
(accept iff u < p_j(d_j)) and u_sample[j] for the sample of row j, drawn by
inverse CDF over token ids in increasing order (the smallest v whose
cumulative mass reaches u times the total).
"""
from __future__ import annotations

import numpy as np

from .model import BLOCK, RequestState, forward_block


def inverse_cdf(weights: np.ndarray, u: float) -> int:
    """Smallest index v with sum(weights[:v+1]) >= u * sum(weights) (weights >= 0, u in (0, 1))."""
    c = np.cumsum(weights)
    return int(min(np.searchsorted(c, u * c[-1], side="left"), len(weights) - 1))


def sample_row(logits: np.ndarray, T: float, u: float, exclude: int = -1) -> tuple[int, float]:
    """Sample of softmax(logits / T) (without token `exclude`) by inverse CDF; also returns the
    distance of u * total to the nearest cumulative boundary, relative to the total (for near-tie reports)."""
    w = np.exp((logits - logits.max()) / T)
    if exclude >= 0:
        w[exclude] = 0.0
    v = inverse_cdf(w, u)
    c = np.cumsum(w)
    t = u * c[-1]
    lo = c[v - 1] if v > 0 else 0.0
    return v, float(min(t - lo, c[v] - t) / c[-1])


def decide(logits: np.ndarray, drafts, T: float, u_accept, u_sample) -> dict:
    """The acceptance rule on the 17 rows' logits: accepted count a, tokens out[0..a], near-tie margins."""
    drafts = np.asarray(drafts, np.int64)
    out = np.full(BLOCK + 1, -1, np.int64)
    margins = []  # |u - p| of every accept test made
    a = BLOCK
    for j in range(BLOCK):
        z = logits[j] / T
        p = np.exp(z - z.max())
        p = p / p.sum()
        d = int(drafts[j])
        pd = p[d] if 0 <= d < len(p) else 0.0
        margins.append(abs(float(u_accept[j]) - pd))
        if float(u_accept[j]) < pd:
            out[j] = d
            continue
        a = j
        break
    tok, margin = sample_row(logits[a], T, float(u_sample[a]), exclude=int(drafts[a]) if a < BLOCK else -1)
    out[a] = tok
    return {"accepted": a, "out": out, "accept_margins": np.array(margins), "sample_margin": margin}


def verify_step_sampled(m, st: RequestState, drafts, T: float, u_accept, u_sample) -> dict:
    """Stochastic block verification of 16 drafts; commits rows 0..a in place (as the greedy step)."""
    drafts = np.asarray(drafts, np.int64)
    L = st.length
    rows = np.concatenate([[st.pending], drafts])
    r = forward_block(m, st.k, st.v, L, rows)
    res = decide(r["logits"], drafts, T, u_accept, u_sample)
    a = res["accepted"]
    st.commit(r["new_k"], r["new_v"], a + 1)
    st.pending = int(res["out"][a])
    res["logits"] = r["logits"]
    return res
