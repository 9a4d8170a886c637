"""GPU check of the device-resident loop (vsd_spec_loop) against the oracle.

Tiny shape (2-layer target, its 2-layer drafter), 3 slots, 5 queued
requests with different context lengths and budgets, prefilled by the
oracle and written into cache slots 3..7 with their anchor rows:
  * every request's generated tokens equal the target's own greedy
    continuation (lossless), bit-exact (near ties of the oracle logged);
  * every request finishes with at least its budget, admissions follow the
    queue order, the queue is drained;
  * the same loop captured as a one-iteration CUDA graph and replayed gives
    the same outputs as the direct call.
"""
import numpy as np
import pytest
import torch

from oracle import model as OM
from tests.gpu_helpers import gpu, load_state, require_gpu
from tests.oracle_helpers import oracle_model
from workload import TINY, drafter_shape, gen, mask_token

pytestmark = gpu
SLOTS, LENS, BUDGETS, OUT_CAP, MAX_TOK = 3, [40, 0, 130, 7, 64], [20, 5, 33, 3, 12], 64, 400


@pytest.fixture(scope="module")
def setup():
    B = require_gpu()
    from speculative_decoding_block_gb300.target import build_target
    master = gen.master_weights(TINY, seed=41)
    om = oracle_model(TINY, master)
    ds = drafter_shape(TINY)
    target, _ = build_target(TINY, master, max_positions=MAX_TOK)
    drafter, _ = build_target(ds, gen.drafter_master(master, TINY.layers, ds.layers), max_positions=MAX_TOK)
    states, anchors = [], []
    for q, L in enumerate(LENS):
        prompt = gen.prompt_ids(TINY.vocab, max(L, 1), 43, q)
        st = OM.prefill(om, prompt)  # L == 0: one prompt token, cached
        r = OM.forward_block(om, [np.zeros((0, TINY.n_kv, TINY.head_dim))] * TINY.layers,
                             [np.zeros((0, TINY.n_kv, TINY.head_dim))] * TINY.layers, 0, prompt, keep_hidden=True)
        states.append(st)
        anchors.append(r["hidden"][-1][-1])
    greedy = [OM.ar_greedy(om, st.copy(), OUT_CAP) for st in states]
    return B, target, drafter, states, np.stack(anchors), greedy


def _run(B, target, drafter, states, anchors, n_iters, graph=False):
    kv = B.vsd_kv_create(target, SLOTS + len(states), MAX_TOK)
    for q, st in enumerate(states):
        load_state(B, kv, SLOTS + q, st)
    ls = B.LoopState(SLOTS, torch.tensor([s.length for s in states]), torch.tensor([s.pending for s in states]),
                     torch.tensor(BUDGETS), torch.tensor(anchors, dtype=torch.float32), OUT_CAP)
    if not graph:
        B.vsd_spec_loop(target, drafter, kv, ls, n_iters, mask_token(TINY))
    else:
        stream = torch.cuda.Stream()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            B.vsd_spec_loop(target, drafter, kv, ls, 1, mask_token(TINY), stream=stream)
        for _ in range(n_iters):
            g.replay()
    torch.cuda.synchronize()
    assert B.vsd_get_device_status(kv) == 0
    return {k: getattr(ls, k).cpu().numpy() for k in ("req_out", "req_generated", "req_admit_iter", "next_req",
                                                       "iter", "slot_req")}


def test_loop_is_lossless_and_drains_the_queue(setup):
    B, target, drafter, states, anchors, greedy = setup
    r = _run(B, target, drafter, states, anchors, 60)
    assert int(r["next_req"][0]) == len(states) and int(r["iter"][0]) == 60
    assert np.all(np.diff(r["req_admit_iter"]) >= 0) and np.all(r["req_admit_iter"] >= 0)
    for q in range(len(states)):
        g = int(r["req_generated"][q])
        assert g >= BUDGETS[q], (q, g)
        n = min(g, OUT_CAP)
        assert np.array_equal(r["req_out"][q][:n], greedy[q][:n]), (q, r["req_out"][q][:n], greedy[q][:n])
    assert np.all(r["slot_req"] == -1)  # everyone has left by iteration 60


def test_loop_in_a_graph_matches_direct(setup):
    B, target, drafter, states, anchors, greedy = setup
    a = _run(B, target, drafter, states, anchors, 25)
    b = _run(B, target, drafter, states, anchors, 25, graph=True)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
