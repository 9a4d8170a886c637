"""Pins of the float64 block-drafter pass (oracle.model.draft_step).

The drafter runs the target's kind of decoder layer (forward_rows, the same
code as the pinned verify forward) over rows [anchor, E[mask] x 16] with no
cache.  What pins the draft-specific parts:
  * no layers: the head alone, drafts = argmax(rmsnorm(E[mask]) E^T) for
    every row (closed form; checks the row indexing 1..16 and the head);
  * with no cache, RoPE rotates all rows' q and k by one offset, so the pass
    depends on the start position only through the BF16 rounding of the
    rotated keys (relative 2^-9; catches absolute positions where relative
    ones belong, or RoPE on V, which move the logits by O(1));
  * block-causal attention: rows 0..j of the full pass equal a pass over the
    first j+1 rows alone;
  * 17 identical input rows (anchor = E[mask]) give 17 identical outputs
    (every key holds the same value vector, whatever the weights);
  * a draft pass over the target's own layers equals forward_block of the
    same rows when they are token embeddings (the shared forward code).
"""
import dataclasses

import numpy as np
import pytest

from oracle import model as OM
from tests.oracle_helpers import oracle_model
from workload import TINY, drafter_shape, gen, mask_token

SHAPE = dataclasses.replace(TINY, name="tiny-draft", vocab=512)


@pytest.fixture(scope="module")
def drafter():
    master = gen.master_weights(SHAPE, seed=11)
    ds = drafter_shape(SHAPE, 2)
    return oracle_model(ds, gen.drafter_master(master, SHAPE.layers, ds.layers)), master


def _anchor(seed=0):
    return gen.anchor_rows(SHAPE.hidden, 1, seed).numpy()[0].astype(np.float64)


def test_zero_layer_drafter_is_the_head(drafter):
    d, master = drafter
    d0 = oracle_model(dataclasses.replace(SHAPE, layers=0),
                      {"embed": master["embed"], "layers": {}})
    mt = mask_token(SHAPE)
    r = OM.draft_step(d0, _anchor(), 40, mt)
    e = d0.embed
    want = np.argmax(OM.rmsnorm(e[mt][None, :], SHAPE.eps) @ e.T, axis=-1)[0]
    assert np.array_equal(r["drafts"], np.full(16, want))
    row0 = np.argmax(OM.rmsnorm(_anchor()[None, :], SHAPE.eps) @ e.T)
    assert int(np.argmax(r["logits"][0])) == int(row0)


def test_no_dependence_on_start_position(drafter):
    d, _ = drafter
    a = OM.draft_step(d, _anchor(1), 0, mask_token(SHAPE))
    b = OM.draft_step(d, _anchor(1), 777, mask_token(SHAPE))
    assert np.abs(a["logits"] - b["logits"]).max() < 5e-3 * np.abs(a["logits"]).max()
    clear = a["top2_gap"][1:] > 1e-2
    assert np.array_equal(a["drafts"][clear], b["drafts"][clear])


def test_block_causal(drafter):
    d, _ = drafter
    s = d.shape
    full = OM.draft_step(d, _anchor(2), 5, mask_token(SHAPE))
    rows = np.concatenate([_anchor(2)[None, :], np.repeat(d.embed[[mask_token(SHAPE)]], 16, axis=0)], 0)
    empty = [np.zeros((0, s.n_kv, s.head_dim)) for _ in range(s.layers)]
    for j in (0, 3, 9):
        part = OM.forward_rows(d, empty, empty, 0, rows[: j + 1], 5 + np.arange(j + 1))
        assert np.abs(part["logits"] - full["logits"][: j + 1]).max() < 1e-10


def test_identical_rows_identical_outputs(drafter):
    d, _ = drafter
    mt = mask_token(SHAPE)
    r = OM.draft_step(d, d.embed[mt], 9, mt)
    assert np.abs(r["logits"] - r["logits"][0][None, :]).max() < 1e-10
    assert len(set(r["drafts"].tolist())) == 1


def test_draft_pass_is_the_shared_forward(drafter):
    d, _ = drafter
    toks = gen.prompt_ids(SHAPE.vocab, 17, 5, 0)
    s = d.shape
    empty = [np.zeros((0, s.n_kv, s.head_dim)) for _ in range(s.layers)]
    a = OM.forward_block(d, empty, empty, 0, toks)
    b = OM.forward_rows(d, empty, empty, 0, d.embed[toks], np.arange(17))
    assert np.array_equal(a["logits"], b["logits"])
