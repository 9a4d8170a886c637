"""Number formats of the mixed-precision weights, from their bit fields.

TEST INFRASTRUCTURE: part of the float64 CPU oracle.  Only tests/, the smoke
check and the CPU-baseline leg of the bench may import anything under
oracle/; the CUDA library never does, and the oracle never imports it.

Formats named by "The Inference Stack Behind OCRia", section "Reducing the
data moved: workload-aware quantization" (BF16, FP8, NVFP4 weights):
  * BF16: sign, 8 exponent bits (bias 127), 7 fraction bits -- the upper half
    of an IEEE binary32;
  * FP8 E4M3 ("fn" variant): sign, 4 exponent bits (bias 7), 3 fraction
    bits, no infinities, S.1111.111 is NaN, largest finite 448;
  * FP4 E2M1 (NVFP4 values): sign, 2 exponent bits (bias 1), 1 fraction bit,
    magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
Encoders round to nearest, ties to the even code (even fraction LSB), and
saturate to the largest finite magnitude; the sign bit follows the input's
sign, so a negative input that rounds to zero gives a negative-zero code.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------- BF16
def bf16_bits_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest BF16 value (ties to even), as float64.

    One rounding step straight from float64 (no detour through float32):
    a BF16 significand has 8 bits, so x = m * 2^e with 0.5 <= |m| < 1 rounds
    to rint(m * 2^8) * 2^(e-8).  Values stay far inside the normal range here.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


# ---------------------------------------------------------------- E4M3
def _e4m3_magnitudes() -> np.ndarray:
    """Magnitude of every code 0x00..0x7F (0x7F is NaN)."""
    v = np.empty(128, dtype=np.float64)
    for c in range(128):
        e, m = (c >> 3) & 0xF, c & 0x7
        v[c] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    v[0x7F] = np.nan
    return v


E4M3_MAG = _e4m3_magnitudes()
E4M3_MAX = 448.0


def e4m3_to_f64(codes) -> np.ndarray:
    c = np.asarray(codes).astype(np.uint8)
    mag = E4M3_MAG[c & 0x7F]
    return np.where(c & 0x80, -mag, mag)


# ---------------------------------------------------------------- E2M1
E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E2M1_MAX = 6.0


def e2m1_to_f64(codes) -> np.ndarray:
    c = np.asarray(codes).astype(np.uint8) & 0xF
    mag = E2M1_MAG[c & 0x7]
    return np.where(c & 0x8, -mag, mag)


# ---------------------------------------------------------------- rounding
def _encode_rne(x, finite_mags: np.ndarray, sign_bit: int, nan_code: int | None) -> np.ndarray:
    """Nearest code to each x among `finite_mags` (ascending, code = index),
    ties to the even code, saturating to the largest finite magnitude."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    top = len(finite_mags) - 1
    i = np.clip(np.searchsorted(finite_mags, a, side="right") - 1, 0, top)
    lo = finite_mags[i]
    hi = finite_mags[np.minimum(i + 1, top)]
    dlo, dhi = a - lo, hi - a
    up = (dhi < dlo) | ((dhi == dlo) & (i % 2 == 1))
    code = np.where(up & (i < top), i + 1, i)
    code = np.where(a >= finite_mags[top], top, code)          # satfinite
    code = code.astype(np.uint8) | np.where(np.signbit(x), sign_bit, 0).astype(np.uint8)
    if nan_code is not None:
        code = np.where(np.isnan(x), nan_code, code).astype(np.uint8)
    return code


def _encode_chunked(x, finite_mags, sign_bit, nan_code, chunk=1 << 16):
    """_encode_rne over slices of a flattened array (keeps temporaries small)."""
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, np.uint8)
    for i in range(0, flat.size, chunk):
        out[i:i + chunk] = _encode_rne(flat[i:i + chunk], finite_mags, sign_bit, nan_code)
    return out.reshape(x.shape)


def f64_to_e4m3(x) -> np.ndarray:
    """Round to nearest E4M3 code (ties to even), saturating at +-448."""
    return _encode_chunked(x, E4M3_MAG[:0x7F], 0x80, 0x7F)


def f64_to_e2m1(x) -> np.ndarray:
    """Round to nearest E2M1 code (ties to even), saturating at +-6 (low nibble)."""
    return _encode_chunked(x, E2M1_MAG, 0x8, None)
