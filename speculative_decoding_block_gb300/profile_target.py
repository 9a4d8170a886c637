"""A few verify steps of one synthetic workload through the library, as a
target for an external profiler (ncu) or a plain timing run.

    python -m speculative_decoding_block_gb300.profile_target WORKLOAD [layered|persistent] [STEPS]
    python -m speculative_decoding_block_gb300.profile_target replay_ssm [LAYERS] [STEPS]

Builds the seeded random-init target of the workload's shape, loads its
synthetic contexts, and runs STEPS steps (default 3) from the same inputs
with random drafts, flushing L2 (a 256 MiB write) before each step.  Each
step is one vsd_verify_step call: the library captures the step as a CUDA
graph on the first call and replays it on the later ones.
"""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from workload import ROWS, WORKLOADS, gen  # noqa: E402

from speculative_decoding_block_gb300 import binding as B  # noqa: E402
from speculative_decoding_block_gb300.target import build_target  # noqa: E402


def replay_ssm(argv):
    """STEPS verify + commit rounds of LAYERS recurrent-state rollback objects
    at 32 requests, 16 heads, d = 128, window 64 (17 rows accepted per
    request and step, so every third commit flushes)."""
    layers = int(argv[0]) if argv else 2
    steps = int(argv[1]) if len(argv) > 1 else 3
    batch, heads, d, window = 32, 16, 128, 64
    rng = np.random.default_rng(11)
    objs = [B.SSM(batch, heads, d, window) for _ in range(layers)]
    for o in objs:
        for b in range(batch):
            o.set_state(b, torch.tensor((rng.normal(size=(heads, d, d)) * 0.05).astype(np.float32), device="cuda"))
    n = batch * heads * ROWS
    q, k, v = (torch.tensor(rng.normal(size=(n, d)).astype(np.float32), device="cuda") for _ in range(3))
    k = k / k.norm(dim=1, keepdim=True)
    alpha = torch.tensor(rng.uniform(0.9, 1.0, n).astype(np.float32), device="cuda")
    beta = torch.tensor(rng.uniform(0.0, 1.0, n).astype(np.float32), device="cuda")
    out = torch.empty((n, d), dtype=torch.float32, device="cuda")
    acc = torch.full((batch,), 16, dtype=torch.int32, device="cuda")
    for _ in range(steps):
        for o in objs:
            o.verify(batch, q, k, v, alpha, beta, out)
            o.commit(batch, acc)
    torch.cuda.synchronize()
    if any(o.device_status() for o in objs):
        raise SystemExit("device status set")
    print("ok replay_ssm", layers, steps)


def main(argv):
    if argv[0] == "replay_ssm":
        return replay_ssm(argv[1:])
    w = WORKLOADS[argv[0]]
    mode = argv[1] if len(argv) > 1 else "layered"
    steps = int(argv[2]) if len(argv) > 2 else 3
    shape = w.shape
    master = gen.master_weights(shape, w.seed)
    model, _ = build_target(shape, master, max_positions=w.max_tokens_per_req())
    del master
    Bn = w.batch
    kv = B.vsd_kv_create(model, Bn, w.max_tokens_per_req())
    B.vsd_kv_set_step_kernel(kv, B.STEP_PERSISTENT if mode == "persistent" else B.STEP_LAYERED)
    if w.paged:
        B.vsd_kv_set_page_table(kv, torch.tensor(gen.page_table(w, kv.pages_per_req), device="cuda").contiguous())
    lens, pend = gen.context_lengths(w), gen.pending_tokens(w)
    for b in range(Bn):
        k, v = gen.synthetic_kv(shape, int(lens[b]), w.seed, b)
        B.vsd_kv_write(kv, b, 0, k.cuda().contiguous(), v.cuda().contiguous())
        del k, v
    seq0 = torch.tensor(lens, dtype=torch.int32, device="cuda")
    pen0 = torch.tensor(pend, dtype=torch.int32, device="cuda")
    seq, pen = seq0.clone(), pen0.clone()
    acc = torch.empty(Bn, dtype=torch.int32, device="cuda")
    out = torch.empty((Bn, ROWS), dtype=torch.int32, device="cuda")
    drafts = torch.tensor(np.random.default_rng(1).integers(0, shape.vocab, (Bn, 16)), dtype=torch.int32,
                          device="cuda")
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    for _ in range(steps):
        seq.copy_(seq0)
        pen.copy_(pen0)
        flush.fill_(1.0)
        B.vsd_verify_step(model, kv, Bn, seq, pen, drafts, acc, out)
        torch.cuda.synchronize()
    status = B.vsd_get_device_status(kv)
    if status:
        raise SystemExit(f"device status {status:#x}")
    print("ok", w.name, mode, steps)


if __name__ == "__main__":
    main(sys.argv[1:])
