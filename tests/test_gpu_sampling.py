"""GPU parity of the stochastic (temperature) verification against the oracle.

Random numbers are inputs, so the GPU and the oracle take the same
decisions: accepted lengths and output tokens bit-exact, except where the
oracle's accept test is within 1e-6 of its threshold or its sample lies
within 2e-7 of the total mass from a cumulative boundary (logged); the
GPU's cumulative mass is a float32 sum of float32 weights, off by about
1e-8 of the total over a 152k-token vocabulary, where one token holds
about 7e-6 of it.
Covered: accepted prefixes of every length 0..16 (u_accept tiny on planted
rows, 0.5 where the draft should be rejected), the correction sample
without the rejected draft, the bonus sample after 16 acceptances; the
tiny shape at T = 0.7 and at temperatures low enough that logit / T far
exceeds the range of a float32 exponential (the weights must be taken
relative to the row maximum), and the benchmarked 0.5B mixed workload
(four requests checked against the oracle, all requests' outputs valid).
"""
import numpy as np
import pytest
import torch

from oracle import model as OM
from oracle import sampling as S
from tests.gpu_helpers import StepIO, gpu, load_state, require_gpu
from tests.oracle_helpers import oracle_model, oracle_state_from_kv
from workload import TINY, WORKLOADS, gen

pytestmark = gpu
T = 0.7


def _uniforms(drafts_k, seed):
    """u_accept: 1e-6 on the planted rows (accept if the target gives them mass), 0.5 after; u_sample uniform."""
    rng = np.random.default_rng(seed)
    ua = np.full((len(drafts_k), 16), 0.5, np.float32)
    for b, k in enumerate(drafts_k):
        ua[b, :k] = 1e-6
    us = (rng.random((len(drafts_k), 17)) * 0.98 + 0.01).astype(np.float32)
    return ua, us


def _check(ref, acc, out, report, b):
    a = ref["accepted"]
    tie = (len(ref["accept_margins"]) and ref["accept_margins"].min() < 1e-6) or ref["sample_margin"] < 2e-7
    if tie:
        report.append(b)
        return
    assert acc == a, (b, acc, a)
    assert np.array_equal(out[: a + 1], ref["out"][: a + 1]), (b, out, ref["out"])
    assert np.all(out[a + 1:] == -1)


@pytest.mark.parametrize("temp", [T, 0.01, 0.004])
def test_tiny_sampled_every_prefix(temp):
    B = require_gpu()
    from speculative_decoding_block_gb300.target import build_target
    master = gen.master_weights(TINY, seed=61)
    om = oracle_model(TINY, master)
    model, _ = build_target(TINY, master, max_positions=512)
    ks = [0, 1, 5, 16, 9, 3]
    states, drafts = [], []
    for b, k in enumerate(ks):
        st = OM.prefill(om, gen.prompt_ids(TINY.vocab, 30 + 17 * b, 62, b))
        g = OM.ar_greedy(om, st.copy(), 17)
        d = gen.plant_drafts(g, min(k, 16), TINY.vocab, "smp", b) if k < 16 else g[:16].copy()
        states.append(st)
        drafts.append(d)
    kv = B.vsd_kv_create(model, len(ks), 512)
    for b, st in enumerate(states):
        load_state(B, kv, b, st)
    ua, us = _uniforms(ks, 63)
    io = StepIO(len(ks), [s.length for s in states], [s.pending for s in states], np.stack(drafts))
    B.vsd_verify_step_sampled(model, kv, len(ks), io.seq, io.pending, io.drafts, io.acc, io.out,
                              torch.tensor(ua).cuda(), torch.tensor(us).cuda(), temp)
    torch.cuda.synchronize()
    assert B.vsd_get_device_status(kv) == 0
    ties = []
    top = []
    for b, st in enumerate(states):
        before = st.copy()
        ref = S.verify_step_sampled(om, st, drafts[b], temp, ua[b].astype(np.float64), us[b].astype(np.float64))
        top.append(float(ref["logits"].max()) / temp)
        _check(ref, int(io.acc[b]), io.out[b].cpu().numpy(), ties, b)
        if b not in ties:
            assert int(io.seq[b]) == before.length + ref["accepted"] + 1
            assert int(io.pending[b]) == int(ref["out"][ref["accepted"]])
    print("near ties", ties, "largest logit / T", max(top))
    # the planted full block with tiny u_accept reaches the bonus row
    assert int(io.acc[3]) == 16 or 3 in ties
    if temp < 0.1:  # the case is meant to exceed what exp() of a raw logit / T holds in float32
        assert max(top) > 88.0


def test_half_b_mixed_sampled_bench_workload():
    B = require_gpu()
    from speculative_decoding_block_gb300.target import build_target
    w = WORKLOADS["0.5b_mixed_b8_ctx512-4096"]
    shape = w.shape
    master = gen.master_weights(shape, w.seed)
    om = oracle_model(shape, master)
    model, _ = build_target(shape, master, max_positions=w.max_tokens_per_req())
    kv = B.vsd_kv_create(model, w.batch, w.max_tokens_per_req())
    lens, pend = gen.context_lengths(w), gen.pending_tokens(w)
    sampled = {0, 2, 5, w.batch - 1}
    states, drafts, ks = {}, [], []
    for b in range(w.batch):
        k, v = gen.synthetic_kv(shape, int(lens[b]), w.seed, b)
        B.vsd_kv_write(kv, b, 0, k.cuda().contiguous(), v.cuda().contiguous())
        st = oracle_state_from_kv(shape, k, v, int(pend[b]))
        if b in sampled:
            states[b] = st
            g = OM.ar_greedy(om, st.copy(), 4)
            drafts.append(gen.plant_drafts(g, 3, shape.vocab, "smp5", b))
            ks.append(3)
        else:
            drafts.append(gen._rng("smp5", b).integers(0, shape.vocab, 16))
            ks.append(0)
    ua, us = _uniforms(ks, 64)
    io = StepIO(w.batch, lens, pend, np.stack(drafts))
    B.vsd_verify_step_sampled(model, kv, w.batch, io.seq, io.pending, io.drafts, io.acc, io.out,
                              torch.tensor(ua).cuda(), torch.tensor(us).cuda(), T)
    torch.cuda.synchronize()
    assert B.vsd_get_device_status(kv) == 0
    out = io.out.cpu().numpy()
    acc = io.acc.cpu().numpy()
    assert np.all((acc >= 0) & (acc <= 16))
    for b in range(w.batch):
        assert np.all((out[b, : acc[b] + 1] >= 0) & (out[b, : acc[b] + 1] < shape.vocab))
    ties = []
    for b in sampled:
        ref = S.verify_step_sampled(om, states[b], drafts[b], T, ua[b].astype(np.float64), us[b].astype(np.float64))
        _check(ref, int(acc[b]), out[b], ties, b)
        print(b, "accept margin", ref["accept_margins"].min() if len(ref["accept_margins"]) else None,
              "sample margin", ref["sample_margin"])
    print("near ties", ties)
    assert len(ties) < len(sampled)  # at least one request compared
