"""The allocation-free attention entry point against the regular one.

vsd_block_attention_static exists for callers that must not allocate device
memory while they run (a server whose memory another allocator hands out
up front, or code running where an allocation is forbidden): it keeps its
scratch in a fixed array inside the library instead.  These tests call it
through the C ABI twice in a row, with different batches, and compare each
result with vsd_block_attention on the same inputs, within the tolerance
used by the other attention tests.  The file is named so that pytest
collects it last.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests.gpu_helpers import rel_rows, require_gpu
from workload import TINY, gen

pytestmark = pytest.mark.gpu


def _model(shape):
    from speculative_decoding_block_gb300.target import build_target
    master = gen.master_weights(shape, seed=5)
    return build_target(shape, master, max_positions=4096)[0]


def _inputs(shape, lens, tag):
    q = torch.stack([gen.normal_bf16((17, shape.n_q, shape.head_dim), 0.6, tag + "q", b) for b in range(len(lens))])
    kn = torch.stack([gen.normal_bf16((17, shape.n_kv, shape.head_dim), 0.6, tag + "k", b) for b in range(len(lens))])
    vn = torch.stack([gen.normal_bf16((17, shape.n_kv, shape.head_dim), 0.6, tag + "v", b) for b in range(len(lens))])
    return q.cuda().contiguous(), kn.cuda().contiguous(), vn.cuda().contiguous()


def test_static_scratch_attention_matches_regular_entry_point():
    B = require_gpu()
    shape = TINY
    model = _model(shape)
    max_batch, max_tokens = 5, 2200
    kv = B.vsd_kv_create(model, max_batch, max_tokens)
    tab = gen._rng("nopt", 4).permutation(kv.num_pages).astype(np.int32)
    B.vsd_kv_set_page_table(kv, torch.tensor(tab[: max_batch * kv.pages_per_req], device="cuda"))
    full = [1900, 0, 640, 17, 1111]
    for b, L in enumerate(full):
        kc = gen.normal_bf16((shape.layers, L, shape.n_kv, shape.head_dim), 0.6, "nak", b, L)
        vc = gen.normal_bf16((shape.layers, L, shape.n_kv, shape.head_dim), 0.6, "nav", b, L)
        if L:
            B.vsd_kv_write(kv, b, 0, kc.cuda().contiguous(), vc.cuda().contiguous())
    # two calls in a row: a larger batch, then a smaller one whose scratch
    # layout differs, so the second sees what the first left behind
    for call, (layer, lens) in enumerate([(1, full), (0, [640, 0, 3])]):
        Bn = len(lens)
        q, kn, vn = _inputs(shape, lens, f"c{call}")
        seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
        ref = torch.full((Bn * 17, shape.n_q * shape.head_dim), float("nan"), dtype=torch.float16, device="cuda")
        got = torch.full_like(ref, float("nan"))
        B.vsd_block_attention(model, kv, layer, Bn, seq, q, kn, vn, ref)
        B.vsd_block_attention_static(model, kv, layer, Bn, seq, q, kn, vn, got)
        torch.cuda.synchronize()
        assert B.vsd_get_device_status(kv) == 0
        g = got.float().cpu().numpy()
        r = ref.float().cpu().numpy()
        assert np.isfinite(g).all(), call
        err = rel_rows(g.reshape(-1, shape.head_dim), r.reshape(-1, shape.head_dim))
        assert err.max() < 1e-2, (call, err.max())


def test_static_scratch_attention_rejects_oversize_batches():
    B = require_gpu()
    shape = TINY
    model = _model(shape)
    Bn = 200  # 400 query tiles of 16 KiB plus their partials: more than the 16 MiB array
    kv = B.vsd_kv_create(model, Bn, 64)
    q, kn, vn = _inputs(shape, [0] * Bn, "big")
    seq = torch.zeros(Bn, dtype=torch.int32, device="cuda")
    out = torch.empty((Bn * 17, shape.n_q * shape.head_dim), dtype=torch.float16, device="cuda")
    with pytest.raises(B.VsdError, match="static array"):
        B.vsd_block_attention_static(model, kv, 0, Bn, seq, q, kn, vn, out)
