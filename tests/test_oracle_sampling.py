"""Pins of the float64 stochastic verification (oracle.sampling).

* inverse CDF against a brute-force scan;
* losslessness in distribution: whatever the first draft (the target's
  favourite, a likely token, an unlikely one), the first output token is
  distributed as softmax(logits_0 / T) -- a chi-square test over 40000
  draws of the random inputs on a 64-token vocabulary (this is where a
  dropped or mis-weighted term of accept-or-resample shows);
* T -> 0 gives greedy verification (accepted length and tokens of the
  greedy rule);
* u_accept = 0 accepts every draft the target gives mass to; u_accept = 1
  accepts none.
"""
import numpy as np
import pytest

from oracle import model as OM
from oracle import sampling as S

T = 0.7


def test_inverse_cdf_brute_force():
    rng = np.random.default_rng(0)
    for _ in range(200):
        w = rng.random(rng.integers(1, 40)) * (rng.random() < 0.5 or 1e-3)
        w[rng.random(len(w)) < 0.3] = 0.0
        if w.sum() == 0:
            w[0] = 1.0
        u = rng.random() * 0.999 + 0.0005
        t = u * w.sum()
        acc, want = 0.0, len(w) - 1
        for v in range(len(w)):
            acc += w[v]
            if acc >= t:
                want = v
                break
        assert S.inverse_cdf(w, u) == want


@pytest.mark.parametrize("which", ["top", "second", "rare"])
def test_first_token_distribution(which):
    rng = np.random.default_rng(1)
    V = 64
    logits = rng.normal(0, 1.5, (17, V))
    p0 = np.exp(logits[0] / T - (logits[0] / T).max())
    p0 /= p0.sum()
    order = np.argsort(-p0)
    d0 = {"top": order[0], "second": order[1], "rare": order[-1]}[which]
    drafts = rng.integers(0, V, 16)
    drafts[0] = d0
    n = 40000
    ua, us = rng.random((n, 16)), rng.random((n, 17))
    counts = np.zeros(V)
    for i in range(n):
        counts[S.decide(logits, drafts, T, ua[i], us[i])["out"][0]] += 1
    expected = p0 * n
    big = expected > 5
    chi2 = float(((counts[big] - expected[big]) ** 2 / expected[big]).sum())
    dof = int(big.sum()) - 1
    assert chi2 < dof + 6 * np.sqrt(2 * dof), (chi2, dof)  # ~4 sigma of the chi-square
    assert counts[~big].sum() < expected[~big].sum() + 6 * np.sqrt(expected[~big].sum() + 1)


def test_zero_temperature_limit_is_greedy():
    rng = np.random.default_rng(2)
    logits = rng.normal(0, 1.0, (17, 50))
    g = OM.greedy(logits)
    for k in (0, 3, 16):
        drafts = rng.integers(0, 50, 16)
        drafts[:k] = g[:k]
        if k < 16 and drafts[k] == g[k]:
            drafts[k] = (g[k] + 1) % 50
        r = S.decide(logits, drafts, 1e-4, rng.random(16) * 0.98 + 0.01, rng.random(17) * 0.98 + 0.01)
        assert r["accepted"] == OM.accept_length(drafts, g) == k
        assert np.array_equal(r["out"][: k + 1], g[: k + 1])


def test_accept_all_or_none():
    rng = np.random.default_rng(3)
    logits = rng.normal(0, 1.0, (17, 30))
    drafts = rng.integers(0, 30, 16)
    r = S.decide(logits, drafts, T, np.zeros(16), rng.random(17))
    assert r["accepted"] == 16 and np.array_equal(r["out"][:16], drafts)
    r = S.decide(logits, drafts, T, np.ones(16), rng.random(17))
    assert r["accepted"] == 0 and r["out"][0] != drafts[0]
