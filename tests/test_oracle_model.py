"""Pins of the oracle's forward and verify step against closed forms, a
library attention, special cases and the losslessness property (no GPU)."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import model as OM
from oracle.formats import round_to_bf16
from tests.oracle_helpers import oracle_model, oracle_state_from_kv
from workload import TINY, gen


def _bf16_bits_of(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _custom_model(shape, embed, mats: dict, lm=None):
    layers = {l: {n: {"fmt": "bf16", "w": _bf16_bits_of(w)} for n, w in m.items()}
              for l, m in mats.items()}
    lm_e = None if lm is None else {"fmt": "bf16", "w": _bf16_bits_of(lm)}
    return OM.Model(shape, _bf16_bits_of(embed), layers, lm_e)


# ------------------------------------------------------------- pieces
def test_rope_is_complex_rotation_by_position_times_frequency():
    rng = np.random.default_rng(0)
    d, theta = 8, 1e4
    x = rng.standard_normal((5, 3, d))
    pos = np.array([0, 1, 7, 100, 4095])
    got = OM.rope(x, pos, theta)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    freq = theta ** (-np.arange(0, d, 2) / d)
    zr = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    assert np.allclose(got[..., : d // 2], zr.real, atol=1e-12)
    assert np.allclose(got[..., d // 2:], zr.imag, atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((1, 1, 64)), rng.standard_normal((1, 1, 64))
    assert np.allclose(OM.rope(q, np.array([0]), 1e4), q)
    assert np.isclose(np.linalg.norm(OM.rope(q, np.array([37]), 1e4)), np.linalg.norm(q))
    dots = [np.sum(OM.rope(q, np.array([p + 5]), 1e4) * OM.rope(k, np.array([p]), 1e4))
            for p in (0, 11, 1000)]
    assert np.allclose(dots, dots[0], rtol=1e-10)


def test_rmsnorm_closed_form():
    x = np.full((2, 8), 3.0)
    x[1] = -0.5
    y = OM.rmsnorm(x, 1e-6)
    assert np.allclose(y[0], 3.0 / np.sqrt(9.0 + 1e-6))
    assert np.allclose(y[1], -0.5 / np.sqrt(0.25 + 1e-6))


def test_block_attention_matches_torch_sdpa_with_gqa_and_causal_block():
    rng = np.random.default_rng(2)
    L, R, n_q, n_kv, d = 23, 17, 6, 2, 16
    q = rng.standard_normal((R, n_q, d))
    K = rng.standard_normal((L + R, n_kv, d))
    V = rng.standard_normal((L + R, n_kv, d))
    got = OM.block_attention(q, K, V, L, n_q // n_kv)
    mask = torch.ones(R, L + R, dtype=torch.bool)
    mask[:, L:] = torch.tril(torch.ones(R, R, dtype=torch.bool))
    qt = torch.from_numpy(q).permute(1, 0, 2)                      # [n_q, R, d]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(n_q // n_kv, dim=0)
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(n_q // n_kv, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    assert np.allclose(got, ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_zero_query_gives_mean_of_visible_values():
    rng = np.random.default_rng(3)
    L, R, n_q, n_kv, d = 9, 4, 4, 2, 8
    K = rng.standard_normal((L + R, n_kv, d))
    V = rng.standard_normal((L + R, n_kv, d))
    got = OM.block_attention(np.zeros((R, n_q, d)), K, V, L, 2)
    for j in range(R):
        for h in range(n_q):
            assert np.allclose(got[j, h], V[: L + j + 1, h // 2].mean(axis=0), atol=1e-13)


def test_single_row_block_is_plain_decode_attention():
    rng = np.random.default_rng(4)
    L, d = 31, 16
    q = rng.standard_normal((1, 2, d))
    K, V = rng.standard_normal((L + 1, 1, d)), rng.standard_normal((L + 1, 1, d))
    got = OM.block_attention(q, K, V, L, 2)
    for h in range(2):
        s = K[:, 0] @ q[0, h] / np.sqrt(d)
        p = np.exp(s - s.max())
        assert np.allclose(got[0, h], (p / p.sum()) @ V[:, 0], atol=1e-13)


def test_accept_length_is_longest_matching_prefix():
    rng = np.random.default_rng(5)
    for _ in range(2000):
        g = rng.integers(0, 3, 16)
        d = np.where(rng.random(16) < 0.8, g, rng.integers(0, 3, 16))
        longest = max(i for i in range(17) if np.array_equal(d[:i], g[:i]))
        assert OM.accept_length(d, g) == longest
    assert OM.accept_length(np.arange(16), np.arange(16)) == 16
    assert OM.accept_length(np.arange(16) + 1, np.arange(16)) == 0


def test_greedy_ties_go_to_lowest_id():
    lg = np.array([[0.0, 2.0, 2.0, 1.0], [5.0, 5.0, 5.0, 5.0]])
    assert OM.greedy(lg).tolist() == [1, 0]


# ------------------------------------------------------------- special-case models
def _shape(**kw):
    base = dict(name="t", layers=1, hidden=4, n_q=2, n_kv=1, head_dim=2, ffn=2, vocab=3,
                rope_theta=1e4, tied=True, attn_fmt="bf16", mlp_fmt="bf16")
    base.update(kw)
    from workload import ModelShape
    return ModelShape(**base)


def test_zero_layers_reduce_to_normed_embedding_times_lm_head():
    s = _shape()
    rng = np.random.default_rng(6)
    emb = np.round(rng.standard_normal((3, 4)) * 8) / 8
    z = lambda n, k: np.zeros((n, k))
    m = _custom_model(s, emb, {0: {"wq": z(4, 4), "wk": z(2, 4), "wv": z(2, 4), "wo": z(4, 4),
                                   "wg": z(2, 4), "wu": z(2, 4), "wd": z(4, 2)}})
    st = OM.RequestState(1, 1, 2)
    r = OM.forward_block(m, st.k, st.v, 0, [2, 0, 1])
    e = emb[[2, 0, 1]]
    expect = (e / np.sqrt(np.mean(e ** 2, axis=1, keepdims=True) + 1e-6)) @ emb.T
    assert np.allclose(r["logits"], expect, atol=1e-12)


def test_silu_applies_to_the_gate_and_multiplies_the_up_projection():
    s = _shape()
    z = lambda n, k: np.zeros((n, k))
    emb = np.ones((3, 4))
    wg = np.array([[-12.5] * 4, [0.25] * 4])     # gate pre-activations ~ (-50, 1)
    wu = np.full((2, 4), 0.25)                    # up ~ (1, 1)
    wd = np.array([[1.0, 0.0], [0.0, 1.0], [0.0, 2.0], [0.0, 0.0]])
    m = _custom_model(s, emb, {0: {"wq": z(4, 4), "wk": z(2, 4), "wv": z(2, 4), "wo": z(4, 4),
                                   "wg": wg, "wu": wu, "wd": wd}})
    st = OM.RequestState(1, 1, 2)
    r = OM.forward_block(m, st.k, st.v, 0, [0], keep_hidden=True)
    c = 1.0 / np.sqrt(1.0 + 1e-6)                 # rmsnorm of an all-ones row
    silu1 = 0.7310585786300049 * c                # silu(c) ~ c * sigmoid(1)
    mlp = r["hidden"][1][0] - r["hidden"][0][0]
    # gate -50c: silu ~ -1e-20 -> that feature contributes nothing
    assert abs(mlp[0]) < 1e-15
    assert np.allclose(mlp[1:3], [silu1 * c, 2 * silu1 * c], rtol=1e-6)


def test_attention_with_zero_queries_adds_wo_times_mean_value():
    s = _shape(hidden=4, n_q=2, n_kv=1, head_dim=2)
    rng = np.random.default_rng(7)
    emb = np.round(rng.standard_normal((3, 4)) * 4) / 4
    z = lambda n, k: np.zeros((n, k))
    wv = np.round(rng.standard_normal((2, 4)) * 4) / 4
    wo = np.round(rng.standard_normal((4, 4)) * 4) / 4
    m = _custom_model(s, emb, {0: {"wq": z(4, 4), "wk": z(2, 4), "wv": wv, "wo": wo,
                                   "wg": z(2, 4), "wu": z(2, 4), "wd": z(4, 2)}})
    st = OM.RequestState(1, 1, 2)
    toks = [1, 2, 0, 2]
    r = OM.forward_block(m, st.k, st.v, 0, toks, keep_hidden=True)
    e = emb[toks]
    u = e / np.sqrt(np.mean(e ** 2, axis=1, keepdims=True) + 1e-6)
    v = round_to_bf16(u @ wv.T)                     # cache dtype
    for j in range(4):
        head = v[: j + 1].mean(axis=0)              # both query heads read KV head 0
        delta = np.concatenate([head, head]) @ wo.T
        assert np.allclose(r["hidden"][1][j] - e[j], delta, atol=1e-12)


# ------------------------------------------------------------- losslessness
@pytest.fixture(scope="module")
def tiny():
    master = gen.master_weights(TINY, seed=7)
    return oracle_model(TINY, master)


def test_prefill_equals_token_by_token_decode(tiny):
    prompt = gen.prompt_ids(TINY.vocab, 12, 7, 0)
    st_p = OM.prefill(tiny, prompt)
    st_a = OM.RequestState(TINY.layers, TINY.n_kv, TINY.head_dim, pending=int(prompt[0]))
    for t in prompt[1:]:
        OM.ar_step(tiny, st_a)
        st_a.pending = int(t)
    nxt = OM.ar_step(tiny, st_a)
    assert nxt == st_p.pending
    for l in range(TINY.layers):
        assert np.allclose(st_a.k[l], st_p.k[l], rtol=1e-10, atol=1e-12)
        assert np.allclose(st_a.v[l], st_p.v[l], rtol=1e-10, atol=1e-12)


def test_verify_with_greedy_drafts_reproduces_autoregressive_decode(tiny):
    prompt = gen.prompt_ids(TINY.vocab, 128, 7, 1)
    st0 = OM.prefill(tiny, prompt)
    st_ar = st0.copy()
    g = OM.ar_greedy(tiny, st_ar, 17)
    st_v = st0.copy()
    res = OM.verify_step(tiny, st_v, g[:16])
    assert res["accepted"] == 16
    assert res["out"].tolist() == g.tolist()
    assert st_v.pending == st_ar.pending and st_v.length == st_ar.length == 128 + 17
    for l in range(TINY.layers):
        assert np.allclose(st_v.k[l], st_ar.k[l], rtol=1e-10, atol=1e-12)
        assert np.allclose(st_v.v[l], st_ar.v[l], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("k", [0, 1, 5, 15])
def test_planted_prefix_is_accepted_exactly(tiny, k):
    prompt = gen.prompt_ids(TINY.vocab, 128, 7, 2)
    st0 = OM.prefill(tiny, prompt)
    g = OM.ar_greedy(tiny, st0.copy(), k + 1)
    d = gen.plant_drafts(g, k, TINY.vocab, "test", k)
    st = st0.copy()
    res = OM.verify_step(tiny, st, d)
    assert res["accepted"] == k
    assert res["out"][: k + 1].tolist() == g[: k + 1].tolist()
    assert np.all(res["out"][k + 1:] == -1)
    assert st.length == 128 + k + 1 and st.pending == g[k]
    # untouched: the cache rows that existed before the step
    for l in range(TINY.layers):
        assert np.array_equal(st.k[l][:128], st0.k[l])


def test_verify_from_synthetic_kv_state(tiny):
    k, v = gen.synthetic_kv(TINY, 40, 3, 0)
    st = oracle_state_from_kv(TINY, k, v, pending=5)
    ref = st.copy()
    g = OM.ar_greedy(tiny, ref, 4)
    res = OM.verify_step(tiny, st, gen.plant_drafts(g, 3, TINY.vocab, "syn"))
    assert res["accepted"] == 3 and res["out"][:4].tolist() == g.tolist()
