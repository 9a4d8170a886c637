"""GPU parity of the single kernels of the step against the float64 oracle:
quantisers (bit-exact), the GEMM in every weight format, block attention,
and the argmax / accept / commit tail (bit-exact)."""
import numpy as np
import pytest
import torch

from oracle import formats as OF
from oracle import model as OM
from oracle import quant as OQ
from tests.gpu_helpers import StepIO, f64_to_bf16_tensor, gpu, read_rows, rel_rows, require_gpu
from tests.oracle_helpers import bits
from workload import ModelShape, TINY, gen

pytestmark = gpu


def _master(n, k, std, seed):
    return gen.normal_bf16((n, k), std, "comp", seed, n, k)


def _edge_matrix():
    """Rows exercising ties, saturation, zero rows / blocks and signed zeros."""
    w = np.zeros((6, 64), np.float32)
    w[0, :8] = [448.0, -448.0, 1.0, -1.0, 2 ** -9, -(2 ** -9), 0.0, -0.0]
    w[1, :16] = np.linspace(-6, 6, 16)
    w[2, 16:32] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -6.0]
    w[4, 3] = 1e-6
    w[5] = np.linspace(-0.02, 0.02, 64)
    return torch.from_numpy(w).to(torch.bfloat16)


@pytest.mark.parametrize("case", ["random_896", "random_ragged", "edge"])
def test_quantisers_match_oracle_bytes(case):
    B = require_gpu()
    if case == "random_896":
        w = _master(1152, 896, 0.02, 1)
    elif case == "random_ragged":
        w = _master(300, 688 - 688 % 16, 1.0, 2)
    else:
        w = _edge_matrix()
    n, k = w.shape
    wd = w.cuda().contiguous()
    q = torch.empty((n, k), dtype=torch.uint8, device="cuda")
    s = torch.empty((n,), dtype=torch.float32, device="cuda")
    B.vsd_quantize_fp8_rowwise(wd, q, s)
    q4 = torch.empty((n, k // 2), dtype=torch.uint8, device="cuda")
    sb = torch.empty((n, k // 16), dtype=torch.uint8, device="cuda")
    S = torch.empty((1,), dtype=torch.float32, device="cuda")
    B.vsd_quantize_nvfp4(wd, q4, sb, S)
    torch.cuda.synchronize()
    w64 = OF.bf16_bits_to_f64(bits(w))
    rq, rs = OQ.quantize_fp8_rowwise(w64)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)
    rq4, rsb, rS = OQ.quantize_nvfp4(w64)
    assert S.item() == rS
    assert np.array_equal(sb.cpu().numpy(), rsb)
    assert np.array_equal(q4.cpu().numpy(), rq4)


def _canonical_dev(fmt, w):
    from speculative_decoding_block_gb300.target import quantize
    return quantize(fmt, w.cuda().contiguous())


def _dequant_dev_entry(e):
    if e["fmt"] == "bf16":
        return OF.bf16_bits_to_f64(bits(e["w"].cpu()))
    if e["fmt"] == "fp8":
        return OQ.dequantize_fp8_rowwise(e["q"].cpu().numpy(), e["s"].cpu().numpy())
    return OQ.dequantize_nvfp4(e["q"].cpu().numpy(), e["sb"].cpu().numpy(), np.float32(e["S"].item()))


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "nvfp4"])
@pytest.mark.parametrize("n,k,m", [(300, 896, 17), (1152, 896, 136), (256, 688, 1), (896, 4864, 40),
                                   (640, 256, 300)])
def test_linear_matches_oracle(fmt, n, k, m):
    B = require_gpu()
    from speculative_decoding_block_gb300.target import weight_of
    if fmt == "nvfp4" and k % 16:
        pytest.skip("NVFP4 needs k % 16 == 0")
    w = _master(n, k, 0.02, 3)
    e = _canonical_dev(fmt, w)
    x = (torch.randn((m, k), generator=torch.Generator().manual_seed(n + k + m)) * 1.0).to(torch.float16)
    y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    B.vsd_linear(weight_of(e), n, k, x.cuda().contiguous(), y)
    torch.cuda.synchronize()
    ref = x.double().numpy() @ _dequant_dev_entry(e).T
    err = rel_rows(y.cpu().numpy(), ref)
    assert np.all(np.isfinite(y.cpu().numpy()))
    assert err.max() < 1e-4, err.max()


def _attn_model(shape):
    from speculative_decoding_block_gb300.target import build_target
    master = gen.master_weights(shape, seed=5)
    return build_target(shape, master, max_positions=4096)[0]


@pytest.mark.parametrize("lens,paged", [((0, 5, 128), False), ((300, 1000, 17), False), ((2100, 63, 777), True)])
def test_block_attention_matches_oracle(lens, paged):
    B = require_gpu()
    shape = TINY
    model = _attn_model(shape)
    Bn = len(lens)
    kv = B.vsd_kv_create(model, Bn, 2200)
    if paged:
        tab = gen._rng("pt", 9).permutation(kv.num_pages).astype(np.int32)
        B.vsd_kv_set_page_table(kv, torch.tensor(tab[: Bn * kv.pages_per_req], device="cuda"))
    rng = np.random.default_rng(7)
    layer = 1
    ctx, q, kn, vn = [], [], [], []
    for b, L in enumerate(lens):
        kc = gen.normal_bf16((shape.layers, L, shape.n_kv, shape.head_dim), 0.6, "ak", b, L)
        vc = gen.normal_bf16((shape.layers, L, shape.n_kv, shape.head_dim), 0.6, "av", b, L)
        if L:
            B.vsd_kv_write(kv, b, 0, kc.cuda().contiguous(), vc.cuda().contiguous())
        ctx.append((kc[layer].double().numpy(), vc[layer].double().numpy()))
        q.append(gen.normal_bf16((17, shape.n_q, shape.head_dim), 0.6, "aq", b))
        kn.append(gen.normal_bf16((17, shape.n_kv, shape.head_dim), 0.6, "akn", b))
        vn.append(gen.normal_bf16((17, shape.n_kv, shape.head_dim), 0.6, "avn", b))
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.full((Bn * 17, shape.n_q * shape.head_dim), float("nan"), dtype=torch.float16, device="cuda")
    B.vsd_block_attention(model, kv, layer, Bn, seq, torch.stack(q).cuda().contiguous(),
                          torch.stack(kn).cuda().contiguous(), torch.stack(vn).cuda().contiguous(), out)
    torch.cuda.synchronize()
    assert B.vsd_get_device_status(kv) == 0
    got = out.float().cpu().numpy().reshape(Bn, 17, shape.n_q, shape.head_dim)
    for b, L in enumerate(lens):
        K = np.concatenate([ctx[b][0], kn[b].double().numpy()], axis=0)
        V = np.concatenate([ctx[b][1], vn[b].double().numpy()], axis=0)
        ref = OM.block_attention(q[b].double().numpy(), K, V, L, shape.group)
        err = rel_rows(got[b], ref)
        assert err.max() < 1e-2, (b, L, err.max())


def test_accept_commit_is_bit_exact():
    B = require_gpu()
    shape = TINY
    model = _attn_model(shape)
    Bn = 5
    kv = B.vsd_kv_create(model, Bn, 512)
    rng = np.random.default_rng(3)
    lens = np.array([0, 16, 100, 250, 495 - 17], np.int32)
    ks = [0, 16, 7, 1, 15]
    V = shape.vocab
    logits = rng.standard_normal((Bn, 17, V)).astype(np.float32)
    drafts = np.zeros((Bn, 16), np.int32)
    pending = rng.integers(0, V, Bn).astype(np.int32)
    for b in range(Bn):
        g = np.argmax(logits[b], axis=-1)
        drafts[b] = gen.plant_drafts(g, ks[b], V, "ac", b)
    logits[1, 3, 5] = logits[1, 3].max()            # exact tie: lowest id wins
    logits[1, 3, 9] = logits[1, 3].max()
    drafts[1, 3] = np.argmax(logits[1, 3])
    # existing cache contents
    pre_k, pre_v = [], []
    for b in range(Bn):
        k0 = gen.normal_bf16((shape.layers, 512, shape.n_kv, shape.head_dim), 1.0, "pk", b)
        v0 = gen.normal_bf16((shape.layers, 512, shape.n_kv, shape.head_dim), 1.0, "pv", b)
        B.vsd_kv_write(kv, b, 0, k0.cuda().contiguous(), v0.cuda().contiguous())
        pre_k.append(k0.double().numpy())
        pre_v.append(v0.double().numpy())
    kn = gen.normal_bf16((shape.layers, Bn, 17, shape.n_kv, shape.head_dim), 1.0, "kn")
    vn = gen.normal_bf16((shape.layers, Bn, 17, shape.n_kv, shape.head_dim), 1.0, "vn")
    io = StepIO(Bn, lens, pending, drafts)
    B.vsd_accept_commit(model, kv, Bn, torch.from_numpy(logits).cuda().contiguous(), kn.cuda().contiguous(),
                        vn.cuda().contiguous(), io.seq, io.pending, io.drafts, io.acc, io.out)
    torch.cuda.synchronize()
    assert B.vsd_get_device_status(kv) == 0
    acc, out = io.acc.cpu().numpy(), io.out.cpu().numpy()
    for b in range(Bn):
        g = OM.greedy(logits[b].astype(np.float64))
        a = OM.accept_length(drafts[b], g)
        assert acc[b] == a == (ks[b] if b != 1 else a)
        ref_out = np.full(17, -1)
        ref_out[: a + 1] = g[: a + 1]
        assert np.array_equal(out[b], ref_out)
        assert io.seq[b].item() == lens[b] + a + 1 and io.pending[b].item() == g[a]
        k_all, v_all = read_rows(B, kv, b, 0, 512, shape)
        exp_k, exp_v = pre_k[b].copy(), pre_v[b].copy()
        exp_k[:, lens[b]: lens[b] + a + 1] = kn[:, b, : a + 1].double().numpy()
        exp_v[:, lens[b]: lens[b] + a + 1] = vn[:, b, : a + 1].double().numpy()
        assert np.array_equal(k_all, exp_k) and np.array_equal(v_all, exp_v)
    assert OM.greedy(logits[1, 3:4].astype(np.float64))[0] == 5
