"""Shared set-up of the GPU parity tests: library targets built from the same
seeded master weights the oracle uses, and cache loading."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import model as OM
from workload import ROWS

gpu = pytest.mark.gpu


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_block_gb300 import binding as B
    B.lib()  # fails loudly if the library is missing
    return B


def f64_to_bf16_tensor(a: np.ndarray) -> torch.Tensor:
    """Values that are exact BF16 numbers (oracle cache rows) -> BF16 tensor."""
    t = torch.tensor(np.asarray(a), dtype=torch.float64)
    out = t.to(torch.float32).to(torch.bfloat16)
    assert torch.equal(out.to(torch.float64), t), "value not representable in BF16"
    return out


def load_state(B, kv, req: int, st: OM.RequestState):
    """Copy an oracle request state's cache rows into cache slot `req`."""
    if st.length == 0:
        return
    k = f64_to_bf16_tensor(np.stack(st.k)).cuda().contiguous()
    v = f64_to_bf16_tensor(np.stack(st.v)).cuda().contiguous()
    B.vsd_kv_write(kv, req, 0, k, v)


def read_rows(B, kv, req: int, start: int, count: int, shape):
    k = torch.empty((shape.layers, count, shape.n_kv, shape.head_dim), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    if count:
        B.vsd_kv_read(kv, req, start, k, v)
    return k.float().cpu().numpy().astype(np.float64), v.float().cpu().numpy().astype(np.float64)


def rel_rows(x: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per-row relative L2 error (last axis)."""
    x = np.asarray(x, np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, ref.shape[-1])
    return np.linalg.norm(x - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)


class StepIO:
    """Device tensors of one verify step for B requests."""

    def __init__(self, B_: int, seq, pending, drafts):
        self.seq = torch.tensor(np.asarray(seq), dtype=torch.int32, device="cuda")
        self.pending = torch.tensor(np.asarray(pending), dtype=torch.int32, device="cuda")
        self.drafts = torch.tensor(np.asarray(drafts), dtype=torch.int32, device="cuda").reshape(B_, 16)
        self.acc = torch.full((B_,), -7, dtype=torch.int32, device="cuda")
        self.out = torch.full((B_, ROWS), -7, dtype=torch.int32, device="cuda")
