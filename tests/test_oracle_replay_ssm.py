"""Pins of the float64 ReplaySSM oracle (oracle/replay_ssm.py).

The update rule against properties of the gated delta rule that do not
restate it: a unit-strength write under a unit key stores v at that key,
directions orthogonal to the key only decay, orthonormal keys act as an
associative memory.  The checkpoint / buffer / pointer machinery against the
plain recurrence over the accepted tokens only ("rollback == recompute"),
over random blocks, accepted lengths (rejections included) and flushes.
"""
import numpy as np
import pytest

from oracle.replay_ssm import ROWS, ReplayState, gdn_update, run_tokens


def _unit(x):
    return x / np.linalg.norm(x)


def test_unit_write_stores_v_under_its_key():
    rng = np.random.default_rng(1)
    S = rng.normal(size=(8, 6))
    k = _unit(rng.normal(size=6))
    v = rng.normal(size=8)
    S1 = gdn_update(S, k, v, 1.0, 1.0)
    assert np.allclose(S1 @ k, v, atol=1e-12)


def test_orthogonal_directions_only_decay():
    rng = np.random.default_rng(2)
    S = rng.normal(size=(5, 7))
    k = _unit(rng.normal(size=7))
    x = rng.normal(size=7)
    x -= (x @ k) * k  # orthogonal to k
    for alpha, beta in ((0.9, 0.5), (0.3, 1.0), (1.0, 0.0)):
        S1 = gdn_update(S, k, rng.normal(size=5), alpha, beta)
        assert np.allclose(S1 @ x, alpha * (S @ x), atol=1e-12)


def test_gate_alone_scales_the_state():
    rng = np.random.default_rng(3)
    S = rng.normal(size=(4, 4))
    S1 = gdn_update(S, _unit(rng.normal(size=4)), rng.normal(size=4), 0.25, 0.0)
    assert np.allclose(S1, 0.25 * S)


def test_orthonormal_keys_recall_their_values():
    rng = np.random.default_rng(4)
    d = 8
    Q, _ = np.linalg.qr(rng.normal(size=(d, d)))
    keys = Q.T[:5]
    vals = rng.normal(size=(5, 6))
    S = run_tokens(rng.normal(size=(6, d)), keys, vals, np.ones(5), np.ones(5))
    for k, v in zip(keys, vals):
        assert np.allclose(S @ k, v, atol=1e-10)


def _block(rng, d_k, d_v):
    q = rng.normal(size=(ROWS, d_k))
    k = np.stack([_unit(x) for x in rng.normal(size=(ROWS, d_k))])
    v = rng.normal(size=(ROWS, d_v))
    return q, k, v, rng.uniform(0.8, 1.0, ROWS), rng.uniform(0.0, 1.0, ROWS)


@pytest.mark.parametrize("window", [17, 40, 64])
def test_rollback_equals_recompute(window):
    rng = np.random.default_rng(window)
    d_k, d_v = 6, 5
    S0 = rng.normal(size=(d_v, d_k))
    rs = ReplayState(S0, window)
    S_ref = S0.copy()  # the plain recurrence over accepted tokens only
    flushes = 0
    for step in range(40):
        q, k, v, a, b = _block(rng, d_k, d_v)
        out = rs.verify(q, k, v, a, b)
        S = S_ref.copy()
        states = []
        for t in range(ROWS):
            S = gdn_update(S, k[t], v[t], a[t], b[t])
            states.append(S)
            assert np.allclose(out[t], S @ q[t], rtol=1e-10, atol=1e-10), (step, t)
        acc = int(rng.integers(-1, ROWS))  # -1: the request was rejected
        ptr_before = rs.ptr
        flushed = rs.commit(acc)
        flushes += flushed
        if acc >= 0:
            S_ref = states[acc]
        assert np.allclose(rs.state(), S_ref, rtol=1e-10, atol=1e-10), step
        assert flushed == (ptr_before + acc + 1 + ROWS > window)
        assert rs.ptr == (0 if flushed else ptr_before + acc + 1)
        if flushed:
            assert np.allclose(rs.ckpt, S_ref, rtol=1e-10, atol=1e-10)
    assert flushes > 0


def test_rejected_block_leaves_the_state():
    rng = np.random.default_rng(9)
    rs = ReplayState(rng.normal(size=(3, 4)), 64)
    before = rs.state().copy()
    rs.verify(*_block(rng, 4, 3))
    assert not rs.commit(-1)
    assert rs.ptr == 0 and np.array_equal(rs.state(), before)
    with pytest.raises(ValueError):
        rs.commit(17)


def test_flush_changes_no_result():
    """The same blocks and accepted lengths through buffers of different
    windows (so the flushes fall at different steps, or never) give the
    same outputs and states."""
    rng = np.random.default_rng(21)
    d_k, d_v = 5, 4
    S0 = rng.normal(size=(d_v, d_k))
    blocks = [_block(rng, d_k, d_v) for _ in range(12)]
    accs = [int(a) for a in rng.integers(-1, ROWS, size=12)]
    runs = []
    for window in (17, 30, 1000):
        rs = ReplayState(S0, window)
        outs, states = [], []
        for blk, acc in zip(blocks, accs):
            outs.append(rs.verify(*blk))
            rs.commit(acc)
            states.append(rs.state().copy())
        runs.append((outs, states))
    for outs, states in runs[1:]:
        for a, b in zip(outs, runs[0][0]):
            assert np.allclose(a, b, rtol=1e-10, atol=1e-10)
        for a, b in zip(states, runs[0][1]):
            assert np.allclose(a, b, rtol=1e-10, atol=1e-10)



def test_closed_form_of_the_buffered_state():
    """The closed form the library's buffer relies on: with corrected values
    u_t = beta_t (v_t - alpha_t S_{t-1} k_t) and L_t the sum of log alpha
    since the checkpoint (floored at -200 per token, which stands for a zero
    gate), S_t = e^{L_t} S_0 + sum_{s<=t} e^{L_t - L_s} u_s k_s^T -- checked
    against the oracle's step-by-step recurrence, a zero gate included."""
    rng = np.random.default_rng(33)
    d_k, d_v, n = 6, 5, 40
    S0 = rng.normal(size=(d_v, d_k))
    ks = np.stack([_unit(x) for x in rng.normal(size=(n, d_k))])
    vs = rng.normal(size=(n, d_v))
    alphas = rng.uniform(0.5, 1.0, n)
    alphas[7] = 0.0  # the state is forgotten at token 7
    betas = rng.uniform(0.0, 1.0, n)
    S = S0.copy()
    us, L = [], []
    for t in range(n):
        us.append(betas[t] * (vs[t] - alphas[t] * (S @ ks[t])))
        L.append((L[-1] if L else 0.0) + max(np.log(alphas[t]) if alphas[t] > 0 else -np.inf, -200.0))
        S = gdn_update(S, ks[t], vs[t], alphas[t], betas[t])
        closed = np.exp(L[t]) * S0 + sum(np.exp(L[t] - L[s]) * np.outer(us[s], ks[s]) for s in range(t + 1))
        assert np.allclose(closed, S, rtol=1e-10, atol=1e-10), t
