"""Device-side failure detection, with every fault made on the host.

Each case feeds one bad request among good ones to a tiny-model step: a
draft id >= vocab, a length with L + 17 > max_tokens, a page-table entry
outside the pool.  The status word must carry the matching bit; the bad
request must report accepted = -1 with its outputs -1 and its length,
pending token and cache rows byte-identical; the good requests must still
match the float64 oracle.  The bounded waits are exercised by a test-only
kernel whose waits can never succeed: it must give up with VSD_DEV_TIMEOUT
and leave the context usable, and a step that sees the timeout bit commits
nothing.  No case faults, traps or hangs the device: the bad values are ones
the kernels clamp before forming any address.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import model as OM
from tests.gpu_helpers import StepIO, gpu, load_state, read_rows, require_gpu
from tests.oracle_helpers import near_tie_check, oracle_model
from tests.step_check import check_request
from workload import ROWS, TINY, gen

pytestmark = gpu

LENS = (40, 70, 100)
MAX_TOKENS = 400
BAD = 1  # the request that carries the fault


@pytest.fixture(scope="module")
def tiny():
    B = require_gpu()
    from speculative_decoding_block_gb300.target import build_target
    master = gen.master_weights(TINY, seed=5)
    om = oracle_model(TINY, master)
    model, _ = build_target(TINY, master, max_positions=1024)
    return B, om, model


def _requests(om):
    states, drafts = [], []
    for b, L in enumerate(LENS):
        st = OM.prefill(om, gen.prompt_ids(TINY.vocab, L, 303, b))
        k = (5, 9, 3)[b]
        g = OM.ar_greedy(om, st.copy(), k + 1)
        drafts.append(gen.plant_drafts(g, k, TINY.vocab, "fail", b))
        states.append(st)
    return states, np.stack(drafts)


def _cache(B, model, states):
    kv = B.vsd_kv_create(model, len(states), MAX_TOKENS)
    for b, st in enumerate(states):
        load_state(B, kv, b, st)
    assert B.vsd_get_device_status(kv) == 0
    return kv


def _step(B, model, kv, seq, pending, drafts):
    Bn = len(seq)
    io = StepIO(Bn, seq, pending, drafts)
    M = ROWS * Bn
    logits = torch.full((M, TINY.vocab), float("nan"), dtype=torch.float32, device="cuda")
    hidden = torch.full((TINY.layers + 1, M, TINY.hidden), float("nan"), dtype=torch.float32, device="cuda")
    B.vsd_verify_step_debug(model, kv, Bn, io.seq, io.pending, io.drafts, io.acc, io.out, logits, hidden)
    torch.cuda.synchronize()
    status = B.vsd_get_device_status(kv)
    res = [(int(io.acc[b]), io.out[b].cpu().numpy(), int(io.seq[b]), int(io.pending[b])) for b in range(Bn)]
    return status, res, logits.cpu().numpy(), hidden.cpu().numpy()


def _check_rejected(B, kv, res_b, seq_b, pending_b, rows_before, n_rows):
    acc, out, seq, pend = res_b
    assert acc == -1 and np.all(out == -1), (acc, out)
    assert seq == seq_b and pend == pending_b
    k, v = read_rows(B, kv, BAD, 0, n_rows, TINY)
    assert np.array_equal(k, rows_before[0]) and np.array_equal(v, rows_before[1])


def _check_good(B, om, kv, states, drafts, res, logits, hidden):
    ties = []
    for b in range(len(states)):
        if b != BAD:
            check_request(om, B, kv, TINY, b, states[b], drafts[b], res[b], logits, hidden, ties)
    print("near ties:", ties)


def test_draft_id_beyond_vocab(tiny):
    B, om, model = tiny
    states, drafts = _requests(om)
    kv = _cache(B, model, states)
    bad = drafts.copy()
    bad[BAD, 4] = TINY.vocab + 5
    n = LENS[BAD] + ROWS
    before = read_rows(B, kv, BAD, 0, n, TINY)
    seq, pend = [s.length for s in states], [s.pending for s in states]
    status, res, logits, hidden = _step(B, model, kv, seq, pend, bad)
    assert status == B.VSD_DEV_BAD_TOKEN, status
    _check_rejected(B, kv, res[BAD], seq[BAD], pend[BAD], before, n)
    _check_good(B, om, kv, states, drafts, res, logits, hidden)


def test_pending_token_beyond_vocab(tiny):
    B, om, model = tiny
    states, drafts = _requests(om)
    kv = _cache(B, model, states)
    n = LENS[BAD] + ROWS
    before = read_rows(B, kv, BAD, 0, n, TINY)
    seq, pend = [s.length for s in states], [s.pending for s in states]
    pend[BAD] = -3
    status, res, logits, hidden = _step(B, model, kv, seq, pend, drafts)
    assert status == B.VSD_DEV_BAD_TOKEN, status
    _check_rejected(B, kv, res[BAD], seq[BAD], pend[BAD], before, n)
    _check_good(B, om, kv, states, drafts, res, logits, hidden)


def test_length_beyond_the_cache(tiny):
    B, om, model = tiny
    states, drafts = _requests(om)
    kv = _cache(B, model, states)
    before = read_rows(B, kv, BAD, 0, MAX_TOKENS, TINY)
    seq, pend = [s.length for s in states], [s.pending for s in states]
    seq[BAD] = MAX_TOKENS - ROWS + 1  # L + 17 = max_tokens + 1
    status, res, logits, hidden = _step(B, model, kv, seq, pend, drafts)
    assert status == B.VSD_DEV_BAD_SEQLEN, status
    _check_rejected(B, kv, res[BAD], seq[BAD], pend[BAD], before, MAX_TOKENS)
    _check_good(B, om, kv, states, drafts, res, logits, hidden)


@pytest.mark.parametrize("where", ["context", "committed"])
def test_page_outside_the_pool(tiny, where):
    """A context page (read by the attention) or the page the committed rows
    would go to lies outside the pool: only that request is rejected."""
    B, om, model = tiny
    states, drafts = _requests(om)
    kv = _cache(B, model, states)
    n = LENS[BAD] + ROWS
    before = read_rows(B, kv, BAD, 0, n, TINY)
    ppr, n_pages = kv.pages_per_req, kv.num_pages
    table = (np.arange(len(LENS) * ppr) % n_pages).astype(np.int32)
    page = 0 if where == "context" else (LENS[BAD] + 16) // 16
    table[BAD * ppr + page] = n_pages + 7
    B.vsd_kv_set_page_table(kv, torch.tensor(table, device="cuda"))
    seq, pend = [s.length for s in states], [s.pending for s in states]
    status, res, logits, hidden = _step(B, model, kv, seq, pend, drafts)
    assert status == B.VSD_DEV_BAD_PAGE, status
    # the pool is untouched: read the request's rows through the valid table again
    table[BAD * ppr + page] = BAD * ppr + page
    B.vsd_kv_set_page_table(kv, torch.tensor(table, device="cuda"))
    assert B.vsd_get_device_status(kv) == 0
    _check_rejected(B, kv, res[BAD], seq[BAD], pend[BAD], before, n)
    _check_good(B, om, kv, states, drafts, res, logits, hidden)


def test_wait_that_never_succeeds_times_out(tiny):
    B, om, model = tiny
    states, drafts = _requests(om)
    kv = _cache(B, model, states)
    with pytest.raises(B.VsdError):
        B.vsd_debug_wait_probe(kv, 0)
    B.vsd_debug_wait_probe(kv, 10_000)
    torch.cuda.synchronize()
    assert B.vsd_get_device_status(kv) == B.VSD_DEV_TIMEOUT
    # the context survives: a step right after matches the oracle
    seq, pend = [s.length for s in states], [s.pending for s in states]
    status, res, logits, hidden = _step(B, model, kv, seq, pend, drafts)
    assert status == 0
    ties = []
    for b in range(len(states)):
        check_request(om, B, kv, TINY, b, states[b], drafts[b], res[b], logits, hidden, ties)


def test_step_after_a_timeout_commits_nothing(tiny):
    """With VSD_DEV_TIMEOUT set (not yet read), the step's outputs cannot be
    trusted: every request is rejected and the cache keeps its rows."""
    B, om, model = tiny
    states, drafts = _requests(om)
    kv = _cache(B, model, states)
    befores = [read_rows(B, kv, b, 0, LENS[b] + ROWS, TINY) for b in range(len(LENS))]
    B.vsd_debug_wait_probe(kv, 10_000)
    seq, pend = [s.length for s in states], [s.pending for s in states]
    status, res, _, _ = _step(B, model, kv, seq, pend, drafts)
    assert status == B.VSD_DEV_TIMEOUT
    for b in range(len(LENS)):
        acc, out, s, p = res[b]
        assert acc == -1 and np.all(out == -1) and s == seq[b] and p == pend[b]
        k, v = read_rows(B, kv, b, 0, LENS[b] + ROWS, TINY)
        assert np.array_equal(k, befores[b][0]) and np.array_equal(v, befores[b][1])


def test_host_step_rejects_a_foreign_cache(tiny):
    """vsd_verify_step_host checks the model / cache pairing before it queues
    any copy; the staging stays usable for the next, valid call."""
    B, om, model = tiny
    from speculative_decoding_block_gb300.target import build_target
    other, _ = build_target(TINY, gen.master_weights(TINY, seed=6), max_positions=1024)
    states, drafts = _requests(om)
    kv = _cache(B, model, states)
    seq = np.array([s.length for s in states], np.int32)
    pend = np.array([s.pending for s in states], np.int32)
    acc = np.full(len(LENS), -7, np.int32)
    out = np.full((len(LENS), ROWS), -7, np.int32)
    L = B.lib()
    args = [B._host(seq, "seq_lens", 3), B._host(pend, "pending", 3), B._host(drafts.astype(np.int32), "drafts", 48,
                                                                                writable=False),
            B._host(acc, "accepted", 3), B._host(out, "out_tokens", 51)]
    st = L.vsd_verify_step_host(other.handle, kv.handle, 3, *args, None)
    assert st == B.VSD_ERR_ARG and b"another model" in L.vsd_last_error()
    assert np.all(acc == -7) and seq[0] == LENS[0]
    B.vsd_verify_step_host(model, kv, 3, seq, pend, drafts.astype(np.int32), acc, out)
    assert B.vsd_get_device_status(kv) == 0
    for b in range(len(LENS)):
        ref = OM.verify_step(om, states[b].copy(), drafts[b])
        ok, _ = near_tie_check(ref, int(acc[b]), out[b])
        assert ok, (b, acc[b], ref["accepted"])
        assert seq[b] == LENS[b] + acc[b] + 1
