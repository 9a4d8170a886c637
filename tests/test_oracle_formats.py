"""Pins of the oracle's number formats against torch casts, bit-field closed
forms and brute-force nearest-value search (no GPU)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_table_matches_torch_all_256_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = F.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_format_golden_points():
    with open(os.path.join(GOLDEN, "formats.json")) as f:
        g = json.load(f)
    for code, val in g["e4m3"]:
        assert F.e4m3_to_f64(np.uint8(code)) == val
    for code, val in g["e2m1"]:
        assert F.e2m1_to_f64(np.uint8(code)) == val
    for x, code in g["e2m1_rne"]:
        assert int(F.f64_to_e2m1(np.float64(x))) == code, x


def test_e2m1_closed_form_from_bit_fields():
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        mag = (m * 0.5) if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        assert F.e2m1_to_f64(np.uint8(c)) == (-mag if s else mag)


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(F.f64_to_e4m3(F.e4m3_to_f64(codes)), codes)


def test_e2m1_roundtrip_every_code():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(F.f64_to_e2m1(F.e2m1_to_f64(codes)), codes)


def _nearest_bruteforce(x, table_codes, table_vals):
    """Nearest value by exhaustive search; ties -> even code."""
    out = []
    for xv in x:
        d = np.abs(table_vals - abs(xv))
        best = np.flatnonzero(d == d.min())
        c = [int(table_codes[i]) for i in best]
        c = [k for k in c if k % 2 == 0] or c
        out.append(c[0] | ((0x80 if table_codes.max() > 15 else 0x8) if np.signbit(xv) else 0))
    return np.array(out, np.uint8)


def test_e4m3_encoder_is_nearest_even_bruteforce():
    rng = np.random.default_rng(0)
    pos_codes = np.arange(0x7F, dtype=np.uint8)
    vals = F.e4m3_to_f64(pos_codes)
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([rng.uniform(-448, 448, 500), rng.uniform(-0.02, 0.02, 500),
                        mids, -mids, vals, [0.0, -0.0, 1e-12, -1e-12]])
    x = x.astype(np.float32).astype(np.float64)
    assert np.array_equal(F.f64_to_e4m3(x), _nearest_bruteforce(x, pos_codes, vals))


def test_e4m3_encoder_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(20000) * 0.01])
    x = np.clip(x, -448, 448).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.f64_to_e4m3(x.astype(np.float64)), ref)


def test_e4m3_saturates():
    assert int(F.f64_to_e4m3(np.float64(1e6))) == 0x7E
    assert int(F.f64_to_e4m3(np.float64(-470.0))) == 0xFE


def test_e2m1_encoder_is_nearest_even_bruteforce():
    codes = np.arange(8, dtype=np.uint8)
    vals = F.e2m1_to_f64(codes)
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([np.linspace(-7, 7, 1001), mids, -mids, vals, [0.1, -0.1]])
    x = np.clip(x, -6, 6)
    assert np.array_equal(F.f64_to_e2m1(x), _nearest_bruteforce(x, codes, vals))


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ours = F.bf16_bits_to_f64(bits)
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_round_to_bf16_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(100000) * rng.choice([1e-3, 1.0, 300.0], 100000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.round_to_bf16(x.astype(np.float64)), ref)
