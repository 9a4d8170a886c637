"""GPU parity of the block-drafter pass against the float64 oracle.

* tiny shape (2 layers, BF16): a drafter made of the target's layers; three
  requests at different start positions with given float32 anchors:
  drafts bit-exact (except after an oracle near tie, top-2 gap < 1e-3),
  logits and hidden rows <= 2e-2 relative (per row, L2);
* anchor export: after a committing verify step the cache holds, per
  request, the target's last residual row at its last accepted position
  (<= 2e-2 relative to the oracle's), and a draft pass on it (no explicit
  anchor) equals one given that row explicitly;
* 0.5B mixed (FP8 attention, NVFP4 MLP): the 5-layer drafter over the 8
  requests of the benchmarked workload: every request's drafts, two
  requests' logits;
* argument checks: a drafter whose shape does not fit the cache, a mask
  token outside the vocabulary.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import model as OM
from tests.gpu_helpers import gpu, load_state, rel_rows, require_gpu
from tests.oracle_helpers import oracle_model
from tests.step_check import HIDDEN_TOL as HID_TOL, LOGIT_TOL, run_step
from workload import HALF_B_MIXED, TINY, WORKLOADS, drafter_shape, gen, mask_token

pytestmark = gpu
TIE = 1e-3


def _drafts_match(ref: dict, got: np.ndarray) -> tuple[bool, int | None]:
    """Drafts equal up to the first row whose oracle top-2 gap is below TIE."""
    gaps = ref["top2_gap"][1:]
    ties = np.flatnonzero(gaps < TIE)
    j = int(ties[0]) if len(ties) else 16
    return bool(np.array_equal(got[:j], ref["drafts"][:j])), (j if j < 16 else None)


def _build(shape, master, drafter_layers, max_positions):
    from speculative_decoding_block_gb300.target import build_target
    ds = drafter_shape(shape, drafter_layers)
    dmaster = gen.drafter_master(master, shape.layers, ds.layers)
    target, _ = build_target(shape, master, max_positions=max_positions)
    drafter, _ = build_target(ds, dmaster, max_positions=max_positions)
    return target, drafter, oracle_model(ds, dmaster)


@pytest.fixture(scope="module")
def tiny():
    B = require_gpu()
    master = gen.master_weights(TINY, seed=21)
    target, drafter, od = _build(TINY, master, 2, 1024)
    return B, master, target, drafter, od


def _run_draft(B, drafter, kv, shape, lens, anchor, layers):
    Bn = len(lens)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    drafts = torch.full((Bn, 16), -7, dtype=torch.int32, device="cuda")
    logits = torch.full((17 * Bn, shape.vocab), float("nan"), device="cuda")
    hidden = torch.full((layers + 1, 17 * Bn, shape.hidden), float("nan"), device="cuda")
    B.vsd_draft_step_debug(drafter, kv, Bn, seq, mask_token(shape), drafts,
                           anchor=None if anchor is None else anchor.cuda().contiguous(),
                           logits=logits, hidden=hidden)
    torch.cuda.synchronize()
    assert B.vsd_get_device_status(kv) == 0
    return drafts.cpu().numpy(), logits.cpu().numpy(), hidden.cpu().numpy()


def test_tiny_drafts_given_anchors(tiny):
    B, master, target, drafter, od = tiny
    lens = [0, 37, 500]
    anchors = gen.anchor_rows(TINY.hidden, len(lens), 3)
    kv = B.vsd_kv_create(target, len(lens), 1024)
    drafts, logits, hidden = _run_draft(B, drafter, kv, TINY, lens, anchors, od.shape.layers)
    ties = []
    for b, L in enumerate(lens):
        ref = OM.draft_step(od, anchors[b].numpy().astype(np.float64), L, mask_token(TINY), keep_hidden=True)
        ok, tie = _drafts_match(ref, drafts[b])
        assert ok, (b, drafts[b], ref["drafts"])
        if tie is not None:
            ties.append((b, tie))
        rows = slice(17 * b, 17 * b + 17)
        assert rel_rows(logits[rows], ref["logits"]).max() < LOGIT_TOL
        for l in range(od.shape.layers + 1):
            assert rel_rows(hidden[l, rows], ref["hidden"][l]).max() < HID_TOL
    print("near ties", ties)


def test_tiny_anchor_export_and_draft(tiny):
    """verify (commits) -> anchor rows in the cache -> draft pass on them."""
    B, master, target, drafter, od = tiny
    om = oracle_model(TINY, master)
    lens = [64, 200]
    states, drafts_in = [], []
    for b, L in enumerate(lens):
        st = OM.prefill(om, gen.prompt_ids(TINY.vocab, L, 31, b))
        g = OM.ar_greedy(om, st.copy(), 6)
        drafts_in.append(gen.plant_drafts(g, 5, TINY.vocab, "anchor", b))
        states.append(st)
    kv = B.vsd_kv_create(target, len(lens), 1024)
    for b, st in enumerate(states):
        load_state(B, kv, b, st)
    res, _, _ = run_step(B, target, kv, TINY, states, drafts_in, debug=False)
    anchor = torch.empty((len(lens), TINY.hidden), dtype=torch.float32, device="cuda")
    B.vsd_kv_get_anchor(kv, len(lens), anchor)
    torch.cuda.synchronize()
    anchor = anchor.cpu()
    new_lens = []
    for b in range(len(lens)):
        ref = OM.verify_step(om, states[b].copy(), drafts_in[b], keep_hidden=True)
        assert res[b][0] == ref["accepted"]
        assert rel_rows(anchor[b].numpy(), ref["anchor"][None, :]).max() < HID_TOL
        new_lens.append(res[b][2])
    # the pass on the exported rows == the pass given the same rows explicitly
    d_cache, lg_cache, _ = _run_draft(B, drafter, kv, TINY, new_lens, None, od.shape.layers)
    d_given, lg_given, _ = _run_draft(B, drafter, kv, TINY, new_lens, anchor, od.shape.layers)
    assert np.array_equal(d_cache, d_given)
    assert np.array_equal(lg_cache, lg_given)
    for b, L in enumerate(new_lens):
        ref = OM.draft_step(od, anchor[b].numpy().astype(np.float64), L, mask_token(TINY))
        assert _drafts_match(ref, d_cache[b])[0]


def test_half_b_mixed_drafter_bench_workload():
    B = require_gpu()
    w = WORKLOADS["0.5b_mixed_b8_ctx512-4096"]
    shape = w.shape
    master = gen.master_weights(shape, w.seed)
    target, drafter, od = _build(shape, master, 5, w.max_tokens_per_req())
    kv = B.vsd_kv_create(target, w.batch, w.max_tokens_per_req())
    lens = [int(x) for x in gen.context_lengths(w)]
    anchors = gen.anchor_rows(shape.hidden, w.batch, w.seed)
    drafts, logits, _ = _run_draft(B, drafter, kv, shape, lens, anchors, od.shape.layers)
    ties = []
    for b in range(w.batch):
        ref = OM.draft_step(od, anchors[b].numpy().astype(np.float64), lens[b], mask_token(shape))
        ok, tie = _drafts_match(ref, drafts[b])
        assert ok, (b, drafts[b], ref["drafts"])
        if tie is not None:
            ties.append((b, tie))
        if b in (0, w.batch - 1):
            assert rel_rows(logits[17 * b: 17 * b + 17], ref["logits"]).max() < LOGIT_TOL
    print("near ties", ties)


def test_draft_argument_checks(tiny):
    B, master, target, drafter, od = tiny
    kv = B.vsd_kv_create(target, 1, 256)
    seq = torch.zeros(1, dtype=torch.int32, device="cuda")
    drafts = torch.empty((1, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(B.VsdError):
        B.vsd_draft_step(drafter, kv, 1, seq, TINY.vocab, drafts)
    other = dataclasses.replace(TINY, name="tiny-wide", ffn=TINY.ffn + 64)
    from speculative_decoding_block_gb300.target import build_target
    wide, _ = build_target(other, gen.master_weights(other, seed=1), max_positions=256)
    with pytest.raises(B.VsdError):
        B.vsd_draft_step(wide, kv, 1, seq, mask_token(TINY), drafts)
