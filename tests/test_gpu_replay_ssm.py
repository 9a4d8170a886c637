"""GPU parity of the ReplaySSM rollback (vsd_ssm_*) against the float64 oracle
(oracle/replay_ssm.py): every verify block's outputs and, after every commit,
the effective state of every request and head, over consecutive steps with
random accepted lengths (rejections included) and the flushes they cause.
Tolerance: per-row relative L2 error <= 1e-4 (fp32 against float64 through
up to a window of gated-delta updates).
"""
import numpy as np
import pytest
import torch

from oracle.replay_ssm import ROWS, ReplayState
from tests.gpu_helpers import gpu, rel_rows, require_gpu

pytestmark = gpu
TOL = 1e-4


def _inputs(rng, B, H, d):
    q = rng.normal(size=(B, H, ROWS, d)).astype(np.float32)
    k = rng.normal(size=(B, H, ROWS, d))
    k = (k / np.linalg.norm(k, axis=-1, keepdims=True)).astype(np.float32)
    v = rng.normal(size=(B, H, ROWS, d)).astype(np.float32)
    alpha = rng.uniform(0.85, 1.0, size=(B, H, ROWS)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, size=(B, H, ROWS)).astype(np.float32)
    return q, k, v, alpha, beta


@pytest.mark.parametrize("d,window", [(64, 40), (128, 64), (128, 17)])
def test_replay_ssm_matches_oracle(d, window):
    B_ = require_gpu()
    rng = np.random.default_rng(d + window)
    B, H = 3, 2
    ssm = B_.SSM(4, H, d, window)
    S0 = (rng.normal(size=(B, H, d, d)) * 0.1).astype(np.float32)
    ref = [[ReplayState(S0[b, h].astype(np.float64), window) for h in range(H)] for b in range(B)]
    for b in range(B):
        ssm.set_state(b, torch.tensor(S0[b], device="cuda"))
    flushes = 0
    for step in range(14):
        q, k, v, alpha, beta = _inputs(rng, B, H, d)
        out = torch.empty((B, H, ROWS, d), dtype=torch.float32, device="cuda")
        dev = [torch.tensor(x, device="cuda") for x in (q, k, v, alpha, beta)]
        ssm.verify(B, *dev, out)
        got = out.cpu().numpy()
        for b in range(B):
            for h in range(H):
                want = ref[b][h].verify(q[b, h], k[b, h], v[b, h], alpha[b, h], beta[b, h])
                e = rel_rows(got[b, h], want)
                assert e.max() < TOL, (step, b, h, e.max())
        acc = rng.integers(-1, ROWS, size=B).astype(np.int32)
        ssm.commit(B, torch.tensor(acc, device="cuda"))
        for b in range(B):
            for h in range(H):
                flushes += ref[b][h].commit(int(acc[b]))
        st = torch.empty((H, d, d), dtype=torch.float32, device="cuda")
        for b in range(B):
            ssm.get_state(b, st)
            s = st.cpu().numpy()
            for h in range(H):
                e = rel_rows(s[h], ref[b][h].state())
                assert e.max() < TOL, (step, b, h, e.max())
        assert ssm.device_status() == 0
    assert flushes > 0


def test_bad_commit_count_rejects_the_block():
    B_ = require_gpu()
    rng = np.random.default_rng(7)
    d, H, window = 64, 1, 64
    ssm = B_.SSM(2, H, d, window)
    S0 = (rng.normal(size=(2, H, d, d)) * 0.1).astype(np.float32)
    for b in range(2):
        ssm.set_state(b, torch.tensor(S0[b], device="cuda"))
    before = torch.empty((H, d, d), dtype=torch.float32, device="cuda")
    ssm.get_state(1, before)
    q, k, v, alpha, beta = _inputs(rng, 2, H, d)
    out = torch.empty((2, H, ROWS, d), dtype=torch.float32, device="cuda")
    ssm.verify(2, *[torch.tensor(x, device="cuda") for x in (q, k, v, alpha, beta)], out)
    ssm.commit(2, torch.tensor([5, 17], dtype=torch.int32, device="cuda"))
    assert ssm.device_status() == B_.VSD_DEV_BAD_SEQLEN
    after = torch.empty_like(before)
    ssm.get_state(1, after)
    assert torch.equal(after, before)  # request 1 kept nothing of the block
    r0 = ReplayState(S0[0, 0].astype(np.float64), window)
    r0.verify(q[0, 0], k[0, 0], v[0, 0], alpha[0, 0], beta[0, 0])
    r0.commit(5)
    ssm.get_state(0, after)
    assert rel_rows(after.cpu().numpy()[0], r0.state()).max() < TOL


@pytest.mark.parametrize("d,window", [(64, 40), (128, 64)])
def test_extreme_gates_and_scales(d, window):
    """Gates of exactly 0 (the state is forgotten) and near 0 next to gates of
    1, a write strength of 0, and state, keys and values at very different
    magnitudes (the per-row power-of-2 operand scales), over enough steps to
    flush."""
    B_ = require_gpu()
    rng = np.random.default_rng(100 + d)
    B, H = 2, 2
    ssm = B_.SSM(B, H, d, window)
    S0 = (rng.normal(size=(B, H, d, d)) * 1e3).astype(np.float32)
    S0[0, 0, :3] = 0.0  # zero rows
    ref = [[ReplayState(S0[b, h].astype(np.float64), window) for h in range(H)] for b in range(B)]
    for b in range(B):
        ssm.set_state(b, torch.tensor(S0[b], device="cuda"))
    for step in range(8):
        q, k, v, alpha, beta = _inputs(rng, B, H, d)
        q *= 1e-3
        v *= 1e2
        alpha = rng.choice(np.array([0.0, 1e-6, 0.5, 1.0], np.float32), size=alpha.shape).astype(np.float32)
        beta[:, :, ::5] = 0.0
        out = torch.empty((B, H, ROWS, d), dtype=torch.float32, device="cuda")
        ssm.verify(B, *[torch.tensor(x, device="cuda") for x in (q, k, v, alpha, beta)], out)
        got = out.cpu().numpy()
        for b in range(B):
            for h in range(H):
                want = ref[b][h].verify(q[b, h], k[b, h], v[b, h], alpha[b, h], beta[b, h])
                assert rel_rows(got[b, h], want).max() < TOL, (step, b, h)
        acc = rng.integers(-1, ROWS, size=B).astype(np.int32)
        ssm.commit(B, torch.tensor(acc, device="cuda"))
        for b in range(B):
            for h in range(H):
                ref[b][h].commit(int(acc[b]))
        st = torch.empty((H, d, d), dtype=torch.float32, device="cuda")
        for b in range(B):
            ssm.get_state(b, st)
            s = st.cpu().numpy()
            for h in range(H):
                assert rel_rows(s[h], ref[b][h].state()).max() < TOL, (step, b, h)
    assert ssm.device_status() == 0


@pytest.mark.parametrize("d,window,B,H", [(64, 40, 16, 12), (128, 64, 10, 16)])
def test_more_items_than_sms(d, window, B, H):
    """More (request, head) items than SMs, so that persistent CTAs walk
    several items and each item's checkpoint and key images are the bulk
    copies its CTA issued during the previous one; requests keep different
    pointers (random accepted lengths), so consecutive items copy different
    numbers of retained rows."""
    B_ = require_gpu()
    rng = np.random.default_rng(1000 + d)
    ssm = B_.SSM(B, H, d, window)
    S0 = (rng.normal(size=(B, H, d, d)) * 0.1).astype(np.float32)
    ref = [[ReplayState(S0[b, h].astype(np.float64), window) for h in range(H)] for b in range(B)]
    for b in range(B):
        ssm.set_state(b, torch.tensor(S0[b], device="cuda"))
    for step in range(5):
        q, k, v, alpha, beta = _inputs(rng, B, H, d)
        out = torch.empty((B, H, ROWS, d), dtype=torch.float32, device="cuda")
        ssm.verify(B, *[torch.tensor(x, device="cuda") for x in (q, k, v, alpha, beta)], out)
        got = out.cpu().numpy()
        for b in range(B):
            for h in range(H):
                want = ref[b][h].verify(q[b, h], k[b, h], v[b, h], alpha[b, h], beta[b, h])
                assert rel_rows(got[b, h], want).max() < TOL, (step, b, h)
        acc = rng.integers(-1, ROWS, size=B).astype(np.int32)
        ssm.commit(B, torch.tensor(acc, device="cuda"))
        for b in range(B):
            for h in range(H):
                ref[b][h].commit(int(acc[b]))
    st = torch.empty((H, d, d), dtype=torch.float32, device="cuda")
    for b in (0, B // 2, B - 1):
        ssm.get_state(b, st)
        s = st.cpu().numpy()
        for h in range(H):
            assert rel_rows(s[h], ref[b][h].state()).max() < TOL, (b, h)
    assert ssm.device_status() == 0
