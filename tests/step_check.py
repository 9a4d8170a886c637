"""Shared checks of a finished GPU verify step against the float64 oracle.

Accepted lengths, output tokens, committed positions and untouched cache
rows: bit-exact (except after an oracle near tie, top-2 gap < 1e-3, which is
reported).  Logits and hidden states: per-row relative L2 error <= 2e-2.
Committed K/V: per (layer, row, head) relative error <= 1e-2.
"""
import numpy as np
import torch

from oracle import model as OM
from tests.gpu_helpers import StepIO, read_rows, rel_rows
from tests.oracle_helpers import near_tie_check

LOGIT_TOL, HIDDEN_TOL, KV_TOL = 2e-2, 2e-2, 1e-2


def check_request(om, B, kv, shape, b, st_before, drafts, res_gpu, logits, hidden, report):
    """Compares request b of a finished GPU step with the oracle model `om` (advances nothing)."""
    st = st_before.copy()
    L = st.length
    ref = OM.verify_step(om, st, drafts, keep_hidden=hidden is not None)
    acc, out, seq, pend = res_gpu
    ok, tie = near_tie_check(ref, acc, out)
    assert ok, (b, acc, out, ref["accepted"], ref["out"])
    if tie is not None:
        report.append((b, tie))
    rows = slice(b * 17, b * 17 + 17)
    if logits is not None:
        e = rel_rows(logits[rows], ref["logits"])
        assert e.max() < LOGIT_TOL, e.max()
    if hidden is not None:
        for l in range(shape.layers + 1):
            e = rel_rows(hidden[l, rows], ref["hidden"][l])
            assert e.max() < HIDDEN_TOL, (l, e.max())
    if tie is None:
        a = ref["accepted"]
        assert seq == L + a + 1 and pend == ref["out"][a]
        k_all, v_all = read_rows(B, kv, b, 0, L + 17, shape)
        # untouched: rows before L and the 16 - a rows after the committed ones
        for l in range(shape.layers):
            assert np.array_equal(k_all[l, :L], st_before.k[l][:L])
            assert np.array_equal(v_all[l, :L], st_before.v[l][:L])
            assert not np.any(k_all[l, L + a + 1:]) and not np.any(v_all[l, L + a + 1:])
            for kvref, got in ((ref["new_k"][l], k_all[l]), (ref["new_v"][l], v_all[l])):
                e = rel_rows(got[L: L + a + 1], kvref[: a + 1])
                assert e.max() < KV_TOL, (l, e.max())
    return ref


def run_step(B, model, kv, shape, states, drafts, debug=True):
    Bn = len(states)
    io = StepIO(Bn, [s.length for s in states], [s.pending for s in states], np.stack(drafts))
    M = 17 * Bn
    logits = hidden = None
    if debug:
        logits = torch.full((M, shape.vocab), float("nan"), dtype=torch.float32, device="cuda")
        hidden = torch.full((shape.layers + 1, M, shape.hidden), float("nan"), dtype=torch.float32, device="cuda")
        B.vsd_verify_step_debug(model, kv, Bn, io.seq, io.pending, io.drafts, io.acc, io.out, logits, hidden)
    else:
        B.vsd_verify_step(model, kv, Bn, io.seq, io.pending, io.drafts, io.acc, io.out)
    torch.cuda.synchronize()
    assert B.vsd_get_device_status(kv) == 0
    res = [(int(io.acc[b]), io.out[b].cpu().numpy(), int(io.seq[b]), int(io.pending[b])) for b in range(Bn)]
    return res, (logits.cpu().numpy() if debug else None), (hidden.cpu().numpy() if debug else None)


