"""GPU parity of the whole greedy verify step against the float64 oracle.

Accepted lengths, output tokens, committed positions and untouched cache
rows: bit-exact (except after an oracle near tie, top-2 gap < 1e-3, which is
logged).  Logits and hidden states: per-row relative L2 error <= 2e-2.
Committed K/V: per (layer, row, head) relative error <= 1e-2.
"""
import numpy as np
import pytest
import torch

from oracle import model as OM
from tests.gpu_helpers import StepIO, gpu, load_state, read_rows, rel_rows, require_gpu
from tests.oracle_helpers import near_tie_check, oracle_model
from tests.step_check import KV_TOL, check_request, run_step
from workload import TINY, WORKLOADS, gen

pytestmark = gpu


@pytest.fixture(scope="module")
def tiny_setup():
    B = require_gpu()
    from speculative_decoding_block_gb300.target import build_target
    w = WORKLOADS["tiny_b1_ctx128"]
    master = gen.master_weights(TINY, seed=w.seed)
    om = oracle_model(TINY, master)
    model, _ = build_target(TINY, master, max_positions=1024)
    return B, om, model


def test_tiny_workload_single_request(tiny_setup):
    B, om, model = tiny_setup
    w = WORKLOADS["tiny_b1_ctx128"]
    st = OM.prefill(om, gen.prompt_ids(TINY.vocab, 128, w.seed, 0))
    k = int(gen.prefix_lengths(w)[0])
    g = OM.ar_greedy(om, st.copy(), min(k + 1, 17))
    drafts = gen.plant_drafts(g, k, TINY.vocab, "tiny", w.seed)
    kv = B.vsd_kv_create(model, 1, 1024)
    load_state(B, kv, 0, st)
    res, logits, hidden = run_step(B, model, kv, TINY, [st], [drafts])
    ties = []
    ref = check_request(om, B, kv, TINY, 0, st, drafts, res[0], logits, hidden, ties)
    assert ref["accepted"] == k or ties


def test_tiny_batch_every_prefix_length(tiny_setup):
    """17 requests, planted k = 0..16, contexts of mixed length incl. empty."""
    B, om, model = tiny_setup
    lens = [0, 1, 15, 16, 17, 31, 64, 127, 128, 129, 200, 255, 256, 300, 40, 90, 5]
    states, drafts = [], []
    for b, L in enumerate(lens):
        st = OM.prefill(om, gen.prompt_ids(TINY.vocab, L, 77, b)) if L else OM.RequestState(
            TINY.layers, TINY.n_kv, TINY.head_dim, pending=int(gen.prompt_ids(TINY.vocab, 1, 78, b)[0]))
        g = OM.ar_greedy(om, st.copy(), min(b + 1, 17))
        drafts.append(gen.plant_drafts(g, b, TINY.vocab, "batch", b))
        states.append(st)
    kv = B.vsd_kv_create(model, len(lens), 400)
    for b, st in enumerate(states):
        load_state(B, kv, b, st)
    res, logits, hidden = run_step(B, model, kv, TINY, states, drafts)
    ties = []
    for b in range(len(lens)):
        check_request(om, B, kv, TINY, b, states[b], drafts[b], res[b], logits, hidden, ties)
    print("near ties:", ties)


def test_tiny_consecutive_steps_match_oracle(tiny_setup):
    """Eight committing steps in a row on a paged (shuffled) cache.

    The same device buffers serve every step (the step advances lengths and
    pending tokens in place), so steps after the first replay the step graph
    the library captured on the first."""
    B, om, model = tiny_setup
    Bn = 3
    states = [OM.prefill(om, gen.prompt_ids(TINY.vocab, 50 + 30 * b, 91, b)) for b in range(Bn)]
    kv = B.vsd_kv_create(model, Bn, 400)
    perm = gen._rng("pt", 91).permutation(kv.num_pages).astype(np.int32)
    B.vsd_kv_set_page_table(kv, torch.tensor(perm, device="cuda"))
    for b, st in enumerate(states):
        load_state(B, kv, b, st)
    io = None
    for step in range(8):
        drafts = []
        for b, st in enumerate(states):
            k = (step * 5 + b * 3) % 17
            g = OM.ar_greedy(om, st.copy(), min(k + 1, 17))
            drafts.append(gen.plant_drafts(g, k, TINY.vocab, "cons", step, b))
        if io is None:
            io = StepIO(Bn, [s.length for s in states], [s.pending for s in states], np.stack(drafts))
        else:
            io.drafts.copy_(torch.tensor(np.stack(drafts), dtype=torch.int32))
            io.acc.fill_(-7)
            io.out.fill_(-7)
        B.vsd_verify_step(model, kv, Bn, io.seq, io.pending, io.drafts, io.acc, io.out)
        torch.cuda.synchronize()
        assert B.vsd_get_device_status(kv) == 0
        for b, st in enumerate(states):
            ref = OM.verify_step(om, st, drafts[b])       # advances the oracle state
            ok, tie = near_tie_check(ref, int(io.acc[b]), io.out[b].cpu().numpy())
            assert ok and tie is None, (step, b)
            assert int(io.seq[b]) == st.length and int(io.pending[b]) == st.pending
    # the GPU cache now holds the same committed rows as the oracle state
    for b, st in enumerate(states):
        k_all, v_all = read_rows(B, kv, b, 0, st.length, TINY)
        for l in range(TINY.layers):
            assert rel_rows(k_all[l], st.k[l]).max() < KV_TOL
            assert rel_rows(v_all[l], st.v[l]).max() < KV_TOL


def test_tiny_host_buffer_steps_match_oracle(tiny_setup):
    """vsd_verify_step_host on numpy arrays: consecutive steps at batch 3,
    then a step of the first two requests alone (a different staging
    layout), each against the oracle."""
    B, om, model = tiny_setup
    states = [OM.prefill(om, gen.prompt_ids(TINY.vocab, 40 + 25 * b, 93, b)) for b in range(3)]
    kv = B.vsd_kv_create(model, 3, 400)
    for b, st in enumerate(states):
        load_state(B, kv, b, st)
    for step, Bn in enumerate([3, 3, 3, 2]):
        drafts = []
        for b in range(Bn):
            k = (step * 7 + b * 5) % 17
            g = OM.ar_greedy(om, states[b].copy(), min(k + 1, 17))
            drafts.append(gen.plant_drafts(g, k, TINY.vocab, "host", step, b))
        seq = np.array([s.length for s in states[:Bn]], dtype=np.int32)
        pend = np.array([s.pending for s in states[:Bn]], dtype=np.int32)
        dr = np.ascontiguousarray(np.stack(drafts).astype(np.int32))
        acc = np.full(Bn, -7, dtype=np.int32)
        out = np.full((Bn, 17), -7, dtype=np.int32)
        B.vsd_verify_step_host(model, kv, Bn, seq, pend, dr, acc, out)
        assert B.vsd_get_device_status(kv) == 0
        for b in range(Bn):
            ref = OM.verify_step(om, states[b], drafts[b])   # advances the oracle state
            ok, tie = near_tie_check(ref, int(acc[b]), out[b])
            assert ok and tie is None, (step, b)
            assert int(seq[b]) == states[b].length and int(pend[b]) == states[b].pending
    with pytest.raises(TypeError):
        B.vsd_verify_step_host(model, kv, 1, seq.astype(np.int64), pend, dr, acc, out)
