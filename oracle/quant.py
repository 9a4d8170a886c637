"""Round-to-nearest weight quantisers and exact dequantisation.

TEST INFRASTRUCTURE: part of the float64 CPU oracle (see oracle/__init__.py).

"The Inference Stack Behind OCRia", section "Reducing the data moved:
workload-aware quantization", names the weight formats (FP8, NVFP4 next to
BF16) but not the scale recipe; its activation-aware calibration needs a
dataset and is replaced by plain round-to-nearest.  Readings taken here
(each one also listed in the design notes):

  FP8 E4M3, one fp32 scale per output channel (row):
      s_row = amax_row / 448                      (fp32 division)
      q     = E4M3_RNE_sat(w / s_row)             (fp32 division)
      w'    = e4m3(q) * s_row
  NVFP4: E2M1 values, one E4M3 scale per 16 consecutive input elements of a
  row, one fp32 scale per tensor:
      S     = amax_tensor / (6 * 448)             (fp32)
      s_blk = E4M3_RNE_sat(amax_blk / (6 * S))    (fp32: 6*S, then the division)
      q     = E2M1_RNE_sat(w / (e4m3(s_blk) * S)) (fp32: the product, then the division)
      w'    = e2m1(q) * e4m3(s_blk) * S
  Codes are packed two per byte, even element in the low nibble.  A scale
  that is zero (all-zero row / block / tensor) stores code 0 for every value.
The arithmetic that decides a code is float32 with one rounding per
operation, so that any implementation that follows the same sequence of
IEEE operations reaches the same bytes.  Dequantisation is exact in float64.
"""
from __future__ import annotations

import numpy as np

from .formats import e2m1_to_f64, e4m3_to_f64, f64_to_e2m1, f64_to_e4m3

F32 = np.float32


def quantize_fp8_rowwise(w) -> tuple[np.ndarray, np.ndarray]:
    """w [N, K] (values exact in float32) -> (q uint8 [N, K], s float32 [N])."""
    w32 = np.asarray(w, dtype=np.float64).astype(F32)
    amax = np.max(np.abs(w32), axis=1)
    s = (amax / F32(448.0)).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (w32 / s[:, None]).astype(F32)
    q = f64_to_e4m3(r.astype(np.float64))
    q[s == 0, :] = 0
    return q, s


def dequantize_fp8_rowwise(q, s) -> np.ndarray:
    return e4m3_to_f64(q) * np.asarray(s, np.float32).astype(np.float64)[:, None]


def quantize_nvfp4(w) -> tuple[np.ndarray, np.ndarray, np.float32]:
    """w [N, K], K % 16 == 0 -> (q uint8 [N, K/2], s_blk uint8 [N, K/16], S float32)."""
    w32 = np.asarray(w, dtype=np.float64).astype(F32)
    n, k = w32.shape
    if k % 16:
        raise ValueError("NVFP4 needs the input dimension to be a multiple of 16")
    S = F32(np.max(np.abs(w32)) / F32(2688.0)) if w32.size else F32(0.0)
    blocks = w32.reshape(n, k // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=2)
    if S == 0:
        return (np.zeros((n, k // 2), np.uint8), np.zeros((n, k // 16), np.uint8), F32(0.0))
    den = F32(F32(6.0) * S)
    sb = f64_to_e4m3((amax_b / den).astype(F32).astype(np.float64))
    scale = (e4m3_to_f64(sb).astype(F32) * S).astype(F32)          # exact e4m3 -> fp32, one product
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (blocks / scale[:, :, None]).astype(F32)
    codes = f64_to_e2m1(r.astype(np.float64))
    codes[np.broadcast_to((scale == 0)[:, :, None], codes.shape)] = 0
    codes = codes.reshape(n, k)
    packed = (codes[:, 0::2] & 0xF) | ((codes[:, 1::2] & 0xF) << 4)
    return packed.astype(np.uint8), sb, S


def unpack_e2m1(q) -> np.ndarray:
    """Packed bytes [N, K/2] -> codes [N, K] (even element from the low nibble)."""
    q = np.asarray(q, np.uint8)
    out = np.empty((q.shape[0], q.shape[1] * 2), np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def dequantize_nvfp4(q, sb, S) -> np.ndarray:
    v = e2m1_to_f64(unpack_e2m1(q))
    n, k = v.shape
    scale = e4m3_to_f64(sb) * float(np.float32(S))
    return (v.reshape(n, k // 16, 16) * scale[:, :, None]).reshape(n, k)
