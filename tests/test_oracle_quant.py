"""Pins of the oracle's round-to-nearest quantisers: exact round trips on
hand-built blocks, brute-force nearest codes, zero blocks, error bounds."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q


def test_fp8_rowwise_roundtrip_on_representable_rows():
    rng = np.random.default_rng(0)
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    codes = rng.choice(finite, size=(6, 64)).astype(np.uint8)
    codes[:, 0] = 0x7E                        # every row reaches amax = 448 * 2^k
    scales = np.float32(2.0) ** np.arange(-9, -3, dtype=np.float32)
    w = F.e4m3_to_f64(codes) * scales.astype(np.float64)[:, None]
    q, s = Q.quantize_fp8_rowwise(w)
    assert np.array_equal(s, scales)
    nz = F.e4m3_to_f64(codes) != 0            # +0 / -0 both decode to 0
    assert np.array_equal(q[nz], codes[nz])
    assert np.array_equal(Q.dequantize_fp8_rowwise(q, s), w)


def test_fp8_codes_are_nearest_to_scaled_weight():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((8, 48)) * 0.02).astype(np.float32).astype(np.float64)
    q, s = Q.quantize_fp8_rowwise(w)
    vals = F.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    r = (w.astype(np.float32) / s[:, None]).astype(np.float64)
    for i in range(w.shape[0]):
        for j in range(w.shape[1]):
            d = np.abs(vals - abs(r[i, j]))
            assert abs(F.e4m3_to_f64(q[i, j])) in vals[d == d.min()]
    assert np.all(np.abs(F.e4m3_to_f64(q)) <= 448)
    assert np.max(np.abs(F.e4m3_to_f64(q)), axis=1).tolist() == [448.0] * 8


def test_fp8_zero_row():
    w = np.zeros((2, 32))
    w[1, 3] = 0.5 * 448           # scale 0.5 exactly
    q, s = Q.quantize_fp8_rowwise(w)
    assert s[0] == 0 and np.all(q[0] == 0)
    assert s[1] == 0.5
    assert Q.dequantize_fp8_rowwise(q, s)[1, 3] == 224.0


def _nvfp4_exact_tensor(rng, n, k, S):
    """Weights that NVFP4 represents exactly, with the largest block scale 448."""
    blk = rng.integers(0x08, 0x7F, size=(n, k // 16)).astype(np.uint8)
    blk[0, 0] = 0x7E
    codes = rng.integers(0, 16, size=(n, k)).astype(np.uint8)
    codes.reshape(n, k // 16, 16)[:, :, 5] = 0x7      # +6 in every block: amax_blk = 6*sblk*S
    v = F.e2m1_to_f64(codes).reshape(n, k // 16, 16)
    w = (v * (F.e4m3_to_f64(blk) * S)[:, :, None]).reshape(n, k)
    return w, codes, blk


def test_nvfp4_roundtrip_on_hand_built_blocks():
    rng = np.random.default_rng(2)
    S = np.float32(2.0 ** -12)
    w, codes, blk = _nvfp4_exact_tensor(rng, 4, 64, float(S))
    q, sb, S2 = Q.quantize_nvfp4(w)
    assert S2 == S
    assert np.array_equal(sb, blk)
    got = Q.unpack_e2m1(q)
    nz = F.e2m1_to_f64(codes) != 0
    assert np.array_equal(got[nz], codes[nz])
    assert np.array_equal(Q.dequantize_nvfp4(q, sb, S2), w)


def test_nvfp4_packing_low_nibble_is_even_element():
    w = np.zeros((1, 16))
    unit = 448 * 2.0 ** -10                 # S = 2^-10, block scale 448
    w[0, 0], w[0, 1] = 6.0 * unit, -3.0 * unit   # codes 0x7 and 0xD
    q, sb, S = Q.quantize_nvfp4(w)
    assert S == 2.0 ** -10 and sb[0, 0] == 0x7E
    assert q[0, 0] == (0x7 | (0xD << 4))
    assert Q.dequantize_nvfp4(q, sb, S)[0, :2].tolist() == [6.0 * unit, -3.0 * unit]


def test_nvfp4_zero_block_and_zero_tensor():
    w = np.zeros((2, 32))
    w[0, 20] = 1.0
    q, sb, S = Q.quantize_nvfp4(w)
    assert sb[0, 0] == 0 and np.all(Q.unpack_e2m1(q)[0, :16] == 0)
    assert np.all(sb[1] == 0) and np.all(q[1] == 0)
    q, sb, S = Q.quantize_nvfp4(np.zeros((3, 16)))
    assert S == 0 and not q.any() and not sb.any()


def test_nvfp4_codes_are_nearest_given_block_scale():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((4, 64)) * 0.02).astype(np.float32).astype(np.float64)
    q, sb, S = Q.quantize_nvfp4(w)
    # the block scale is the nearest E4M3 to amax_blk / (6 S), computed in fp32
    amax = np.max(np.abs(w.reshape(4, 4, 16)), axis=2).astype(np.float32)
    target = (amax / np.float32(np.float32(6) * S)).astype(np.float64)
    vals = F.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    for i, j in np.ndindex(4, 4):
        d = np.abs(vals - target[i, j])
        assert F.e4m3_to_f64(sb[i, j]) in vals[d == d.min()]
    grid = F.e2m1_to_f64(np.arange(8, dtype=np.uint8))
    scale = (F.e4m3_to_f64(sb).astype(np.float32) * S).astype(np.float32)
    codes = Q.unpack_e2m1(q).reshape(4, 4, 16)
    r = (w.reshape(4, 4, 16).astype(np.float32) / scale[:, :, None]).astype(np.float64)
    for i, j, e in np.ndindex(4, 4, 16):
        d = np.abs(grid - min(abs(r[i, j, e]), 6.0))
        assert abs(F.e2m1_to_f64(codes[i, j, e])) in grid[d == d.min()]


@pytest.mark.parametrize("std", [0.02, 1.0])
def test_quantisation_error_bounds(std):
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((16, 256)) * std).astype(np.float32).astype(np.float64)
    q, s = Q.quantize_fp8_rowwise(w)
    err = np.abs(Q.dequantize_fp8_rowwise(q, s) - w)
    # E4M3: half a spacing -- relative 2^-4 for normals, absolute 2^-10 * s for subnormals
    assert np.all(err <= np.maximum(np.abs(w) * 2.0 ** -4, s[:, None] * 2.0 ** -10) * (1 + 1e-6))
    q4, sb, S = Q.quantize_nvfp4(w)
    err4 = np.abs(Q.dequantize_nvfp4(q4, sb, S) - w)
    scale = (F.e4m3_to_f64(sb) * float(S)).repeat(16, axis=1)
    # E2M1: at most one unit (spacing 2 between 4 and 6, halved) per block scale,
    # plus the block scale's own E4M3 rounding (<= 1/16 relative of 6*scale)
    assert np.all(err4 <= scale * 1.0 + 6 * scale / 16 + 1e-12)
