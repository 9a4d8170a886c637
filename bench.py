"""Throughput of the greedy block-verify step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one vsd_verify_step over the whole batch of the workload (every
request: pending token + 16 drafts through the target, argmax, prefix accept,
KV commit).  The step is replayed from a CUDA graph with seq_lens / pending
restored before each replay (the step is deterministic, so the re-committed
rows get identical values); L2 is flushed between timed steps.  value =
verified tokens (sum of accepted+1) per second over all ranks.

N > 1 runs N independent replicas (one per GPU, launched by torchrun): the
verify step has no cross-request exchange, so there is no collective on the
data path; the barrier and the max over ranks are for timing only.

--impl reference times the float64 CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import atexit
import hashlib
import json
import multiprocessing as mp
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workload import ROWS, WORKLOADS, drafter_shape, gen, linear_shapes, mask_token  # noqa: E402

DEFAULT_WORKLOAD = "0.5b_mixed_b8_ctx512-4096"
METRIC = "verified tokens/sec per GB300, 0.5B target, block 16; verify-step HBM % peak"


# ------------------------------------------------------------------ byte accounting
def weight_bytes(shape, name: str) -> int:
    n, k, fmt = linear_shapes(shape)[name]
    if fmt == "bf16":
        return 2 * n * k
    if fmt == "fp8":
        return n * k + 4 * n
    return n * k // 2 + n * k // 16 + 4


def kernel_bytes(shape, lens, accepted):
    """Algorithmic HBM bytes per launch of each kernel kind (weights / KV that must be read,
    results that must be written; intermediates that can stay on chip are not counted)."""
    B = len(lens)
    M = ROWS * B
    H = shape.hidden
    kv_row = 2 * shape.n_kv * shape.head_dim * 2            # K + V of one token, one layer
    act = lambda k: M * k * 2
    d = {
        "embed": M * H * 2 + M * H * 6 + M * 4,
        "qkv_gemm": sum(weight_bytes(shape, n) for n in ("wq", "wk", "wv")) + act(H),
        "attention": int(np.sum(lens)) * kv_row + M * shape.n_q * shape.head_dim * 2 * 2,
        "o_proj_gemm": weight_bytes(shape, "wo") + act(shape.n_q * shape.head_dim) + 2 * M * H * 4 + act(H),
        "gate_up_gemm": weight_bytes(shape, "wg") + weight_bytes(shape, "wu") + act(H) + act(shape.ffn),
        "down_gemm": weight_bytes(shape, "wd") + act(shape.ffn) + 2 * M * H * 4 + act(H),
        "lm_head_gemm": shape.vocab * H * 2 + act(H),
        "accept_commit": int(np.sum(np.asarray(accepted) + 1)) * kv_row * shape.layers + B * 4 * 60,
    }
    # the persistent launch: every layer's GEMMs and attention, then the head
    per_layer = sum(d[k] for k in ("qkv_gemm", "attention", "o_proj_gemm", "gate_up_gemm", "down_gemm"))
    d["step"] = per_layer * shape.layers + d["lm_head_gemm"]
    return d


def step_bytes(shape, lens, accepted) -> int:
    """Algorithmic bytes of one whole step: every weight once (incl. scales), the lm_head,
    17*B embedding rows, the KV context, the committed rows, ids and outputs."""
    B = len(lens)
    w = sum(weight_bytes(shape, n) for n in linear_shapes(shape)) * shape.layers
    w += shape.vocab * shape.hidden * 2
    emb = ROWS * B * shape.hidden * 2
    kv_row = 2 * shape.n_kv * shape.head_dim * 2 * shape.layers
    kv = int(np.sum(lens)) * kv_row
    commit = int(np.sum(np.asarray(accepted) + 1)) * kv_row
    io = B * (16 * 4 + 8) + B * (4 + 17 * 4 + 8)
    return w + emb + kv + commit + io


def draft_pass_bytes(shape, B: int) -> int:
    """Algorithmic bytes of one drafter pass: its layers' weights once, the head, 17*B rows in, drafts out."""
    ds = drafter_shape(shape)
    w = sum(weight_bytes(ds, n) for n in linear_shapes(ds)) * ds.layers + shape.vocab * shape.hidden * 2
    return w + ROWS * B * shape.hidden * 2 + B * shape.hidden * 4 + B * (4 + 16 * 4)


def step_flops(shape, lens) -> float:
    B = len(lens)
    M = ROWS * B
    params = sum(n * k for n, k, _ in linear_shapes(shape).values()) * shape.layers + shape.vocab * shape.hidden
    attn = 4 * ROWS * shape.n_q * shape.head_dim * (float(np.sum(lens)) + 9) * shape.layers
    return 2.0 * M * params + attn


_CODE_TOKENS = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'', re.S)


def code_only(src: str) -> str:
    """C++ source without comments and blank lines (string and char literals kept)."""
    src = _CODE_TOKENS.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", src)
    return "\n".join(l.rstrip() for l in src.splitlines() if l.strip())


SSM_SOURCES = ("replay_ssm.cuh", "replay_ssm.cu")  # the recurrent-state rollback, outside the verify step


def kernel_source_sha(ssm: bool = False) -> str:
    """Hash of the library's code (comments and blank lines excluded), naming
    the build an ncu capture was taken on: the verify step's sources, or
    (ssm) the recurrent-state rollback kernels' own."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "speculative_decoding_block_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if (f in SSM_SOURCES) != ssm:
            continue
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(f.encode() + code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha()
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == kind and parts[1] == workload \
                and parts[3] == sha:
            return int(parts[2])
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 10 ms from before the warm-up; the summary keeps
    the samples whose timestamps fall inside the timed region (or, when the
    region is shorter than the sampling interval, the two nearest)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        proc, self.proc = self.proc, None
        if proc is not None:
            proc.terminate()
            try:
                out, _ = proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                proc.kill()
                out, _ = proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t0: float, t1: float):
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[1]), float(f[2]), [n for n, v in zip(names, f[5:9]) if v.lower() == "active"]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside and rows:  # region shorter than the interval: the nearest samples on either side
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:2]
        sm = [r[1] for r in inside]
        reasons = sorted({n for r in inside for n in r[3]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": inside[0][2] if inside else None,
                "samples": len(sm), "samples_in_region": sum(t0 <= r[0] <= t1 for r in rows),
                "region_s": round(t1 - t0, 4), "reasons": reasons}


# ------------------------------------------------------------------ oracle (CPU) sample
def _oracle_worker(name: str, n_requests: int, budget_s: float, go, q):
    """Runs in a spawned process: oracle set-up, then (after `go`) a timed sample."""
    try:
        import torch  # noqa: F401  (CPU only)
        from oracle import model as OM
        from tests.oracle_helpers import oracle_model, oracle_state_from_kv
        w = WORKLOADS[name]
        shape = w.shape
        master = gen.master_weights(shape, w.seed)
        om = oracle_model(shape, master)
        del master
        lens = gen.context_lengths(w)
        pend = gen.pending_tokens(w)
        ks = gen.prefix_lengths(w)
        reqs = []
        for b in range(min(n_requests, w.batch)):
            kk, vv = gen.synthetic_kv(shape, int(lens[b]), w.seed, b)
            st = oracle_state_from_kv(shape, kk, vv, int(pend[b]))
            g = OM.ar_greedy(om, st.copy(), min(int(ks[b]) + 1, 16))
            reqs.append((st, gen.plant_drafts(g, int(ks[b]), shape.vocab, "bench", w.seed, b)))
        q.put(("ready", None))
        go.wait()
        tokens, steps, t0 = 0, 0, time.perf_counter()
        while True:
            st, d = reqs[steps % len(reqs)]
            r = OM.verify_step(om, st.copy(), d)
            tokens += r["accepted"] + 1
            steps += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        q.put(("done", {"tokens": tokens, "steps": steps, "seconds": dt,
                        "cores": len(os.sched_getaffinity(0))}))
    except Exception as e:  # report, never hang the parent
        q.put(("error", repr(e)))


def start_oracle(name: str, n_requests: int, budget_s: float):
    ctx = mp.get_context("spawn")
    go, q = ctx.Event(), ctx.Queue()
    p = ctx.Process(target=_oracle_worker, args=(name, n_requests, budget_s, go, q), daemon=True)
    p.start()
    return p, go, q


def finish_oracle(handle, timeout=900):
    p, go, q = handle
    go.set()
    res = None
    t_end = time.time() + timeout
    while time.time() < t_end:
        try:
            kind, val = q.get(timeout=5)
        except Exception:
            if not p.is_alive():
                break
            continue
        if kind == "done":
            res = val
            break
        if kind == "error":
            res = {"error": val}
            break
    p.join(timeout=10)
    if p.is_alive():
        p.kill()
    return res


# ------------------------------------------------------------------ GPU arm
def job_totals(seconds: float, units: float, world: int, device: str = "cpu"):
    """Whole-job figures of a replicated run: the slowest rank's time and the
    units all ranks processed (the replicas exchange nothing else)."""
    if world == 1:
        return seconds, units
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


class Step:
    """One workload's cache, inputs and planted drafts on the device, and the
    one-step CUDA graph on a side stream (inputs reset and L2 flushed before
    every replay)."""

    def __init__(self, B, w, model, flush, stream):
        import torch
        self.B, self.w, self.shape, self.model, self.flush, self.stream = B, w, w.shape, model, flush, stream
        dev = "cuda"
        self.max_tok = w.max_tokens_per_req()
        Bn = self.Bn = w.batch
        kv = self.kv = B.vsd_kv_create(model, Bn, self.max_tok)
        if w.paged:
            pt = gen.page_table(w, kv.pages_per_req)
            B.vsd_kv_set_page_table(kv, torch.tensor(pt, device=dev).contiguous())
        self.lens = gen.context_lengths(w)
        self.pend = gen.pending_tokens(w)
        for b in range(Bn):
            kk, vv = gen.synthetic_kv(self.shape, int(self.lens[b]), w.seed, b)
            B.vsd_kv_write(kv, b, 0, kk.to(dev).contiguous(), vv.to(dev).contiguous())
            del kk, vv
        torch.cuda.synchronize()
        self.seq0 = torch.tensor(self.lens, dtype=torch.int32, device=dev)
        self.pend0 = torch.tensor(self.pend, dtype=torch.int32, device=dev)
        self.seq, self.pen = self.seq0.clone(), self.pend0.clone()
        self.acc = torch.empty(Bn, dtype=torch.int32, device=dev)
        self.out = torch.empty((Bn, ROWS), dtype=torch.int32, device=dev)
        self.drafts = torch.zeros((Bn, 16), dtype=torch.int32, device=dev)
        # greedy trace of every request from the library itself (verify steps with
        # arbitrary drafts advance the greedy continuation by a+1 >= 1 tokens)
        trace = [[] for _ in range(Bn)]
        rnd = np.random.default_rng(12345)
        while min(len(t) for t in trace) < ROWS:
            self.drafts.copy_(torch.tensor(rnd.integers(0, self.shape.vocab, (Bn, 16)), dtype=torch.int32))
            B.vsd_verify_step(model, kv, Bn, self.seq, self.pen, self.drafts, self.acc, self.out)
            o = self.out.cpu().numpy()
            for b in range(Bn):
                trace[b].extend(int(x) for x in o[b] if x >= 0)
        ks = gen.prefix_lengths(w)
        self.planted = np.stack([gen.plant_drafts(np.array(trace[b]), int(ks[b]), self.shape.vocab, "bench", w.seed, b)
                                 for b in range(Bn)])
        self.drafts.copy_(torch.tensor(self.planted, dtype=torch.int32))
        self.reset()
        B.vsd_verify_step(model, kv, Bn, self.seq, self.pen, self.drafts, self.acc, self.out)
        torch.cuda.synchronize()
        assert B.vsd_get_device_status(kv) == 0
        self.accepted = self.acc.cpu().numpy()
        self.tokens_per_step = int(np.sum(self.accepted + 1))
        self.reset()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            B.vsd_verify_step(model, kv, Bn, self.seq, self.pen, self.drafts, self.acc, self.out, stream=stream)

    def reset(self):
        self.seq.copy_(self.seq0)
        self.pen.copy_(self.pend0)

    def replay(self, ev=None):
        import torch
        with torch.cuda.stream(self.stream):
            self.reset()
            self.flush.fill_(1.0)
            if ev:
                ev[0].record(self.stream)
            self.graph.replay()
            if ev:
                ev[1].record(self.stream)

    def timed(self, warmup, steps):
        """Per-step device times (ms) of `steps` replays after `warmup`."""
        import torch
        for _ in range(warmup):
            self.replay()
        torch.cuda.synchronize()
        if not np.array_equal(self.acc.cpu().numpy(), self.accepted):
            raise RuntimeError("graph replay gave different accepted lengths than the direct call")
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for ev in evs:
            self.replay(ev)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def direct(self):
        """One step launched directly on the side stream (inputs reset, L2 flushed)."""
        import torch
        with torch.cuda.stream(self.stream):
            self.reset()
            self.flush.fill_(1.0)
        self.B.vsd_verify_step(self.model, self.kv, self.Bn, self.seq, self.pen, self.drafts, self.acc, self.out,
                               stream=self.stream)

    def profiled(self, reps=3):
        """Per-kind launch counts and device times (us, summed over the kind's
        launches) of one step: each launch bracketed by CUDA events on the side
        stream (inputs reset, L2 flushed); medians over reps."""
        import torch
        runs = []
        for _ in range(reps):
            with torch.cuda.stream(self.stream):
                self.reset()
                self.flush.fill_(1.0)
            per = {}
            for kind, ms in self.B.vsd_verify_step_profiled(self.model, self.kv, self.Bn, self.seq, self.pen,
                                                            self.drafts, self.acc, self.out, stream=self.stream):
                n, t = per.get(kind, (0, 0.0))
                per[kind] = (n + 1, t + ms * 1e3)
            runs.append(per)
        return {k: (runs[0][k][0], float(np.median([r[k][1] for r in runs]))) for k in runs[0]}

    def recapture(self):
        """Captures the step graph again (after a change of the cache's step kernel)."""
        import torch
        self.reset()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self.B.vsd_verify_step(self.model, self.kv, self.Bn, self.seq, self.pen, self.drafts, self.acc, self.out,
                                   stream=self.stream)


def kernel_report(shape, lens, accepted, kern, ms_per_step):
    """`kernels` key of the bench line: per launch its share of the step, that
    share of the event-timed step, and its algorithmic bytes."""
    kb = kernel_bytes(shape, lens, accepted)
    tot = sum(us for _, us in kern.values())
    kernels = {}
    for k, (n, us) in kern.items():
        us_ev = ms_per_step * 1e3 * us / tot / n  # per launch, scaled to the event-timed step
        kernels[k] = {"launches": n, "us_bracketed": round(us / n, 2), "us_avg": round(us_ev, 2),
                      "ms_total": round(us_ev * n / 1e3, 4), "share": round(us / tot, 4),
                      "bytes_per_launch": kb[k], "gbs": round(kb[k] / (us_ev * 1e-6) / 1e9, 1)}
    return kernels


def run_gpu(args, rank: int, world: int):
    import torch
    from speculative_decoding_block_gb300 import binding as B
    from speculative_decoding_block_gb300.build import build
    from speculative_decoding_block_gb300.target import build_target

    w = WORKLOADS[args.workload]
    shape = w.shape
    build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dev = "cuda"
    max_tok = w.max_tokens_per_req()
    # the RoPE table also covers the other configurations of the same shape, which reuse this target
    max_pos = max([max_tok] + [x.max_tokens_per_req() for x in WORKLOADS.values() if x.shape == shape])
    master = gen.master_weights(shape, w.seed)
    model, _ = build_target(shape, master, max_positions=max_pos)
    drafter = None
    if not args.no_draft:
        ds = drafter_shape(shape)
        drafter, _ = build_target(ds, gen.drafter_master(master, shape.layers, ds.layers), max_positions=max_tok)
    del master
    stream = torch.cuda.Stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    S = Step(B, w, model, flush, stream)
    Bn, kv, lens, pend, accepted = S.Bn, S.kv, S.lens, S.pend, S.accepted
    seq, pen, acc, out, drafts, seq0, pend0 = S.seq, S.pen, S.acc, S.out, S.drafts, S.seq0, S.pend0
    tokens_per_step = S.tokens_per_step

    clk = ClockSampler(torch.cuda.current_device()).start()
    atexit.register(clk.stop)  # never leave the sampler running
    for _ in range(args.warmup):
        S.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_region0 = time.time()
    step_ms = S.timed(0, args.steps)
    t_region1 = time.time()
    clk.stop()
    if world > 1:
        torch.distributed.barrier()
    total_s, job_tokens = job_totals(sum(step_ms) / 1e3, tokens_per_step * args.steps, world, dev)
    ms_per_step = total_s * 1e3 / args.steps

    # per-kernel times of the same step (event-bracketed launches)
    kern = S.profiled()
    kernels = kernel_report(shape, lens, accepted, kern, ms_per_step)
    dominant = max(kernels, key=lambda k: kernels[k]["ms_total"])

    # end to end through the public host-buffer call: inputs up, the step,
    # outputs down, all inside vsd_verify_step_host
    h_seq0 = np.asarray(lens, dtype=np.int32)
    h_pen0 = np.asarray(pend, dtype=np.int32)
    h_dr = np.ascontiguousarray(np.asarray(S.planted, dtype=np.int32))
    h_seq, h_pen = h_seq0.copy(), h_pen0.copy()
    h_acc = np.empty(Bn, dtype=np.int32)
    h_out = np.empty((Bn, ROWS), dtype=np.int32)
    e2e_times = []
    e2e_tokens = 0
    for i in range(args.warmup + args.steps):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
        stream.synchronize()
        h_seq[:] = h_seq0
        h_pen[:] = h_pen0
        t0 = time.perf_counter()
        B.vsd_verify_step_host(model, kv, Bn, h_seq, h_pen, h_dr, h_acc, h_out, stream=stream)
        if i >= args.warmup:
            e2e_times.append(time.perf_counter() - t0)
            e2e_tokens += int(np.sum(h_acc + 1))
    if not np.array_equal(h_acc, accepted):
        raise RuntimeError("the host-buffer step gave different accepted lengths than the device step")
    h2d = 4 * Bn * (16 + 2)
    d2h = 4 * Bn * (3 + ROWS)
    e2e_s, e2e_job_tokens = job_totals(sum(e2e_times), e2e_tokens, world, dev)
    e2e_value = e2e_job_tokens / e2e_s

    hbm, tf_burst, tf_sust, peak_src = peaks()
    sb = step_bytes(shape, lens, accepted)
    value = job_tokens / total_s
    dk = kernels[dominant]
    achieved = dk["bytes_per_launch"] / (dk["us_avg"] * 1e-6) / 1e9
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded random-init weights, random KV context, planted draft prefixes)",
        "config": {
            "workload": w.name,
            "shape": {"name": shape.name, "layers": shape.layers, "hidden": shape.hidden,
                      "heads": f"{shape.n_q}q/{shape.n_kv}kv/{shape.head_dim}", "ffn": shape.ffn,
                      "vocab": shape.vocab,
                      "weights": f"attn {shape.attn_fmt}, mlp {shape.mlp_fmt}, embed/lm_head bf16"},
            "batch": Bn, "rows_per_request": ROWS, "ctx_lens": [int(x) for x in lens],
            "paged": w.paged, "accepted": [int(a) for a in accepted],
            "tokens_per_step": tokens_per_step, "mean_accepted_plus_1": round(tokens_per_step / Bn, 3),
            "parallelism": f"replicas x{world}", "l2": "flushed between steps (256 MiB write)",
            "graph": "one CUDA graph per step", "step_bytes": sb, "step_gflop": round(step_flops(shape, lens) / 1e9, 2),
        },
        "verify_steps_per_s": round(args.steps * world / total_s, 2),
        "step_hbm_frac": round(sb / (ms_per_step * 1e-3) / 1e9 / hbm, 4),
        "step_hbm_frac_nominal_8tbs": round(sb / (ms_per_step * 1e-3) / 1e9 / 8000.0, 4),
        "roofline": {"kernel": dominant, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": recorded_traffic(dominant, w.name),
                     "bytes_per_launch": dk["bytes_per_launch"], "us_avg": dk["us_avg"],
                     "time": "event-timed step x the kernel's share of the event-bracketed launches"},
        "kernels": kernels,
        "kernel_times": "each launch of one step bracketed by CUDA events (median of 3, L2 flushed); us_avg is "
                        "the event-timed step x the launch's share of those times",
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * statistics.mean(e2e_times), 4),
                "ms_per_step_median": round(1e3 * statistics.median(e2e_times), 4),
                "ms_per_step_max": round(1e3 * max(e2e_times), 4),
                "call": "vsd_verify_step_host (one packed copy each way; replays the step graph the library captured on its first call)"},
        "gpu_launches": sum(n for n, _ in kern.values()),
        "clocks": clk.summary(t_region0, t_region1),
    }
    result["persistent"] = time_persistent(B, S, args)
    result["replay_ssm"] = time_replay_ssm(B, flush, stream)
    result["sampled"] = time_sampled(B, model, kv, Bn, seq, pen, drafts, acc, out, seq0, pend0, flush, stream, args)
    if w.steps > 1:
        result["consecutive"] = time_consecutive(B, model, kv, shape, w, Bn, seq, pen, seq0, pend0, max_tok, flush,
                                                 stream)
    if drafter is not None:
        result["draft"] = time_draft(B, model, drafter, kv, shape, Bn, seq, pen, drafts, acc, out, seq0, pend0,
                                     S.graph, flush, stream, args)
        result["loop"] = time_loop(B, model, drafter, shape, w, max_tok, flush, stream)
    del S, kv, drafter
    # the other configurations' own units, measured in the same run
    for key, name in (("config4", "0.5b_mixed_b32_ctx1024-8192_paged16_64steps"), ("config5", "7b_mixed_b16_ctx4096")):
        if args.no_extra or name == w.name or name not in WORKLOADS:
            continue
        try:
            result[key] = measure_extra(B, WORKLOADS[name], model if WORKLOADS[name].shape == shape else None,
                                        flush, stream, args)
        except Exception as e:  # report, keep the main line
            result[key] = {"workload": name, "error": repr(e)[:300]}
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle's set-up and its timed sample start after the GPU arm
        r = finish_oracle(start_oracle(args.workload, n_requests=2, budget_s=args.cpu_budget))
        if r and "tokens" in r:
            result["cpu_baseline"] = {
                "value": round(r["tokens"] / r["seconds"], 3), "unit": "tokens/s", "cores": r["cores"],
                "kind": "oracle",
                "sample": f"{r['steps']} float64 verify steps of requests 0-1 of this workload "
                          f"(one request per step) in {r['seconds']:.1f} s"}
        else:
            result["cpu_baseline"] = {"value": None, "unit": "tokens/s", "kind": "oracle",
                                      "error": (r or {}).get("error", "no result")}
    if rank == 0:
        print(json.dumps(result), flush=True)


def time_replay_ssm(B, flush, stream, layers=24, batch=32, heads=16, d=128, window=64, steps=40):
    """The ReplaySSM verify + commit of a recurrent layer stack at 32 requests
    (the pages profile 24 GDN layers at 32 concurrent requests): each layer's
    own state object, one CUDA graph of all layers' verify and commit, the
    accepted counts of a planted-prefix mix (mean k + 1 about 9.9), L2
    flushed before each replay.  The pointers advance from replay to replay,
    so the flushes (about one commit in four) are in the mean."""
    import torch
    rng = np.random.default_rng(11)
    objs = [B.SSM(batch, heads, d, window) for _ in range(layers)]
    for o in objs:
        for b in range(batch):
            o.set_state(b, torch.tensor((rng.normal(size=(heads, d, d)) * 0.05).astype(np.float32), device="cuda"))
    n = batch * heads * ROWS
    q = torch.tensor(rng.normal(size=(n, d)).astype(np.float32), device="cuda")
    k = rng.normal(size=(n, d))
    k = torch.tensor((k / np.linalg.norm(k, axis=1, keepdims=True)).astype(np.float32), device="cuda")
    v = torch.tensor(rng.normal(size=(n, d)).astype(np.float32), device="cuda")
    alpha = torch.tensor(rng.uniform(0.9, 1.0, n).astype(np.float32), device="cuda")
    beta = torch.tensor(rng.uniform(0.0, 1.0, n).astype(np.float32), device="cuda")
    out = torch.empty((n, d), dtype=torch.float32, device="cuda")
    acc = torch.tensor(np.minimum(rng.geometric(1.0 / 9.9, batch) - 1, 16).astype(np.int32), device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for o in objs:
            o.verify(batch, q, k, v, alpha, beta, out, stream=stream)
            o.commit(batch, acc, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(5 + steps):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
            if i >= 5:
                evs[i - 5][0].record(stream)
            g.replay()
            if i >= 5:
                evs[i - 5][1].record(stream)
    torch.cuda.synchronize()
    if any(o.device_status() for o in objs):
        raise RuntimeError("replay verify reported a device error")
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    us = ms * 1e3 / layers
    hb = batch * heads
    mean_ptr = (window - ROWS) / 2  # the retained buffer grows from 0 to at most window - 17 between flushes
    per_layer = (hb * d * d * 4                            # checkpoint read
                 + hb * mean_ptr * (8 * d + 8)             # retained keys, corrected values (fp32), log sums (f64)
                 + hb * ROWS * (3 * d + 2) * 4              # block inputs read
                 + hb * ROWS * d * 4                        # outputs written
                 + hb * ROWS * (8 * d + 8))                 # the block's keys, corrected values, log sums staged
    return {"layers": layers, "requests": batch, "heads": heads, "d": d, "window": window,
            "us_per_layer": round(us, 2), "ms_all_layers": round(ms, 4),
            "bytes_per_layer_est": int(per_layer), "hbm_frac_est": round(per_layer / (us * 1e-6) / 1e9 / peaks()[0], 4),
            "accepted_plus_1_mean": round(float((acc + 1).float().mean().item()), 2),
            "note": "verify + commit (with its periodic flush) of every layer in one graph; bytes without flushes"}


def time_persistent(B, S, args):
    """The same step with the single persistent launch (graph replays, L2
    flushed), then the cache goes back to the default launches."""
    B.vsd_kv_set_step_kernel(S.kv, B.STEP_PERSISTENT)
    try:
        S.recapture()
        ms = S.timed(args.warmup, max(10, min(args.steps, 100)))
        kern = S.profiled()
    finally:
        B.vsd_kv_set_step_kernel(S.kv, B.STEP_LAYERED)
        S.recapture()
    m = statistics.mean(ms)
    kernels = kernel_report(S.shape, S.lens, S.accepted, kern, m)
    return {"ms_per_step": round(m, 4), "tokens_per_s": round(S.tokens_per_step / (m * 1e-3), 1),
            "step_hbm_frac": round(step_bytes(S.shape, S.lens, S.accepted) / (m * 1e-3) / 1e9 / peaks()[0], 4),
            "kernels": kernels, "gpu_launches": sum(n for n, _ in kern.values()),
            "note": "vsd_kv_set_step_kernel(VSD_STEP_PERSISTENT): the layers and the head in one cooperative launch"}


def measure_extra(B, w, model, flush, stream, args):
    """Another configuration's unit on the same GPU: its step (graph replays,
    L2 flushed), the per-kernel split and, for a multi-step workload, its
    consecutive committing steps as one graph.  `model`: the already built
    target when the shape is the same (random-init weights either way)."""
    import torch
    from speculative_decoding_block_gb300.target import build_target
    t_setup = time.time()
    shape = w.shape
    if model is None:
        master = gen.master_weights(shape, w.seed)
        model, _ = build_target(shape, master, max_positions=w.max_tokens_per_req())
        del master
    S = Step(B, w, model, flush, stream)
    setup_s = time.time() - t_setup
    steps = max(10, min(args.steps, 50))
    ms = S.timed(args.warmup, steps)
    ms_step = statistics.mean(ms)
    kern = S.profiled()
    kernels = kernel_report(shape, S.lens, S.accepted, kern, ms_step)
    hbm = peaks()[0]
    sb = step_bytes(shape, S.lens, S.accepted)
    r = {"workload": w.name, "batch": S.Bn, "steps": steps, "warmup": args.warmup,
         "ms_per_step": round(ms_step, 4), "tokens_per_step": S.tokens_per_step,
         "tokens_per_s": round(S.tokens_per_step / (ms_step * 1e-3), 1),
         "verify_steps_per_s": round(1e3 / ms_step, 2), "step_bytes": sb,
         "step_hbm_frac": round(sb / (ms_step * 1e-3) / 1e9 / hbm, 4),
         "accepted": [int(a) for a in S.accepted], "kernels": kernels,
         "gpu_launches": sum(n for n, _ in kern.values()), "setup_s": round(setup_s, 1)}
    r["persistent"] = time_persistent(B, S, args)
    if w.steps > 1:
        r["consecutive"] = time_consecutive(B, model, S.kv, shape, w, S.Bn, S.seq, S.pen, S.seq0, S.pend0,
                                            S.max_tok, flush, stream)
    return r


def time_consecutive(B, model, kv, shape, w, Bn, seq, pen, seq0, pend0, max_tok, flush, stream, runs=3):
    """The workload's consecutive committing steps as one timed unit.  Drafts
    are planted per step and request (prefix lengths drawn per step) from the
    library's own greedy trace, taken by a pre-pass from the same start with
    random drafts (every such step emits the target's greedy tokens, at least
    one per request).  All steps run as one CUDA graph; lengths and pending
    tokens are restored before each replay, which recommits identical rows."""
    import torch
    S = w.steps
    ks = np.stack([gen.prefix_lengths(w, s) for s in range(S)])      # [S, B]
    need = (ks + 1).sum(axis=0) + ROWS                                  # trace tokens per request
    acc1 = torch.empty(Bn, dtype=torch.int32, device="cuda")
    out1 = torch.empty((Bn, ROWS), dtype=torch.int32, device="cuda")
    dr1 = torch.empty((Bn, 16), dtype=torch.int32, device="cuda")
    seq.copy_(seq0)
    pen.copy_(pend0)
    torch.cuda.synchronize()
    L0 = seq0.cpu().numpy()
    trace = [[] for _ in range(Bn)]
    rnd = np.random.default_rng(54321)
    while any(len(t) < n for t, n in zip(trace, need)):
        if max(int(L0[b]) + len(trace[b]) for b in range(Bn)) + ROWS > max_tok:
            raise RuntimeError("greedy trace would outgrow the cache")
        dr1.copy_(torch.tensor(rnd.integers(0, shape.vocab, (Bn, 16)), dtype=torch.int32))
        B.vsd_verify_step(model, kv, Bn, seq, pen, dr1, acc1, out1)
        o = out1.cpu().numpy()
        for b in range(Bn):
            trace[b].extend(int(x) for x in o[b] if x >= 0)
    planted = np.zeros((S, Bn, 16), np.int32)
    pos = np.zeros(Bn, np.int64)
    for st in range(S):
        for b in range(Bn):
            t = np.asarray(trace[b][pos[b]:pos[b] + ROWS])
            planted[st, b] = gen.plant_drafts(t, int(ks[st, b]), shape.vocab, "consecutive", w.seed, st, b)
            pos[b] += int(ks[st, b]) + 1
    drafts_all = torch.tensor(planted, device="cuda")
    acc_all = torch.full((S, Bn), -1, dtype=torch.int32, device="cuda")
    out_all = torch.empty((S, Bn, ROWS), dtype=torch.int32, device="cuda")
    seq.copy_(seq0)
    pen.copy_(pend0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for st in range(S):
            B.vsd_verify_step(model, kv, Bn, seq, pen, drafts_all[st], acc_all[st], out_all[st], stream=stream)

    def replay(ev=None):
        with torch.cuda.stream(stream):
            seq.copy_(seq0)
            pen.copy_(pend0)
            flush.fill_(1.0)
            if ev:
                ev[0].record(stream)
            g.replay()
            if ev:
                ev[1].record(stream)

    replay()
    torch.cuda.synchronize()
    if B.vsd_get_device_status(kv) != 0:
        raise RuntimeError("consecutive steps reported a device error")
    accs = acc_all.cpu().numpy()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
    for ev in evs:
        replay(ev)
    torch.cuda.synchronize()
    if not np.array_equal(acc_all.cpu().numpy(), accs):
        raise RuntimeError("consecutive replays disagree")
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    tokens = int((accs + 1).sum())
    return {"steps": S, "replays": runs, "ms_total": round(ms, 3), "ms_per_step": round(ms / S, 4),
            "tokens": tokens, "tokens_per_s": round(tokens / (ms * 1e-3), 1),
            "mean_accepted_plus_1": round(float((accs + 1).mean()), 3),
            "planted_mean_k_plus_1": round(float((ks + 1).mean()), 3),
            "steps_as_planted": round(float((accs == ks).mean()), 4),
            "kv_tokens_first_last": [int(L0.sum()), int(L0.sum() + (accs[:-1] + 1).sum())],
            "graph": f"{S} committing steps in one CUDA graph, L2 flushed before each replay"}


def time_sampled(B, model, kv, Bn, seq, pen, drafts, acc, out, seq0, pend0, flush, stream, args, temperature=0.7):
    """The stochastic verification step at temperature 0.7 on the same inputs (graph replay, L2 flushed);
    uniforms from a fixed generator (they are inputs of the step)."""
    import torch
    rng = np.random.default_rng(7)
    ua = torch.tensor(rng.random((Bn, 16)), dtype=torch.float32, device="cuda")
    us = torch.tensor(rng.random((Bn, 17)), dtype=torch.float32, device="cuda")
    gs = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gs, stream=stream):
        B.vsd_verify_step_sampled(model, kv, Bn, seq, pen, drafts, acc, out, ua, us, temperature, stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.warmup + args.steps):
        with torch.cuda.stream(stream):
            seq.copy_(seq0)
            pen.copy_(pend0)
            flush.fill_(1.0)
            if i >= args.warmup:
                ev[i - args.warmup][0].record(stream)
            gs.replay()
            if i >= args.warmup:
                ev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    if B.vsd_get_device_status(kv) != 0:
        raise RuntimeError("sampled step reported a device error")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    tokens = int((acc + 1).sum().item())
    return {"temperature": temperature, "ms_per_step": round(ms, 4), "tokens_per_step": tokens,
            "tokens_per_s": round(tokens / (ms * 1e-3), 1),
            "accepted": [int(x) for x in acc.cpu().numpy()],
            "note": "random-init target: at T = 0.7 a planted draft has p(d) ~ 1e-4, so almost every step emits "
                    "one sampled token per request; ms_per_step is the cost of the sampled step"}


def time_draft(B, model, drafter, kv, shape, Bn, seq, pen, drafts, acc, out, seq0, pend0, g_verify, flush, stream,
               args):
    """The drafter pass alone (graph replay, L2 flushed between passes) and one
    speculative iteration (verify step, then a draft pass on its anchor rows)."""
    import torch
    mask = mask_token(shape)
    dout = torch.empty((Bn, 16), dtype=torch.int32, device="cuda")
    # anchor rows and lengths of a committed verify step
    with torch.cuda.stream(stream):
        seq.copy_(seq0)
        pen.copy_(pend0)
        g_verify.replay()
    stream.synchronize()
    seq_after = seq.clone()
    gd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gd, stream=stream):
        B.vsd_draft_step(drafter, kv, Bn, seq_after, mask, dout, stream=stream)
    gi = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gi, stream=stream):
        B.vsd_verify_step(model, kv, Bn, seq, pen, drafts, acc, out, stream=stream)
        B.vsd_draft_step(drafter, kv, Bn, seq, mask, dout, stream=stream)

    def timed(graph, reset):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                if reset:
                    seq.copy_(seq0)
                    pen.copy_(pend0)
                flush.fill_(1.0)
                if i >= args.warmup:
                    ev[i - args.warmup][0].record(stream)
                graph.replay()
                if i >= args.warmup:
                    ev[i - args.warmup][1].record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    ms_draft = timed(gd, False)
    ms_iter = timed(gi, True)
    if B.vsd_get_device_status(kv) != 0:
        raise RuntimeError("draft pass reported a device error")
    pb = draft_pass_bytes(shape, Bn)
    hbm = peaks()[0]
    return {"layers": drafter_shape(shape).layers, "weights": "the target's last layers (random init), its head",
            "mask_token": mask, "ms_per_pass": round(ms_draft, 4),
            "drafted_tokens_per_s": round(Bn * 16 / (ms_draft * 1e-3), 1),
            "pass_bytes": pb, "pass_hbm_frac": round(pb / (ms_draft * 1e-3) / 1e9 / hbm, 4),
            "ms_per_iteration": round(ms_iter, 4),
            "iteration": "one CUDA graph: verify step, then a draft pass on its anchor rows"}


def time_loop(B, model, drafter, shape, w, max_tok, flush, stream, queued=16, iters=64, budget=48, runs=3):
    """The device-resident loop: w.batch slots, `queued` requests with synthetic contexts of the workload's
    length mix and synthetic anchor rows, `iters` iterations of schedule -> draft -> verify -> collect in one
    CUDA graph (L2 flushed before each run)."""
    import torch
    slots = w.batch
    kv = B.vsd_kv_create(model, slots + queued, max_tok)
    rng = np.random.default_rng(w.seed)
    lens = rng.integers(w.ctx_lo, min(w.ctx_hi, max_tok - budget - 40) + 1, size=queued)
    for q in range(queued):
        kk, vv = gen.synthetic_kv(shape, int(lens[q]), w.seed + 1, q)
        B.vsd_kv_write(kv, slots + q, 0, kk.cuda().contiguous(), vv.cuda().contiguous())
        del kk, vv
    pend = rng.integers(0, shape.vocab, size=queued)
    anchors = gen.anchor_rows(shape.hidden, queued, w.seed)
    ls = B.LoopState(slots, torch.tensor(lens), torch.tensor(pend), torch.full((queued,), budget),
                     anchors, budget + 17)
    fresh = {k: getattr(ls, k).clone() for k in ("slot_req", "next_req", "iter", "req_generated",
                                                  "req_admit_iter", "req_out")}

    def reset():
        for k, v in fresh.items():
            getattr(ls, k).copy_(v)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        B.vsd_spec_loop(model, drafter, kv, ls, iters, mask_token(shape), stream=stream)
    times = []
    for r in range(runs + 1):
        with torch.cuda.stream(stream):
            reset()
            flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        if r:
            times.append(e0.elapsed_time(e1))
    if B.vsd_get_device_status(kv) != 0:
        raise RuntimeError("loop reported a device error")
    gen_tok = int(ls.req_generated.sum().item())
    busy = int((ls.req_admit_iter >= 0).sum().item())
    ms = statistics.mean(times)
    return {"slots": slots, "queued": queued, "iterations": iters, "budget": budget,
            "requests_admitted": busy, "requests_finished": int((ls.req_generated >= budget).sum().item()),
            "generated_tokens": gen_tok, "ms_total": round(ms, 3), "ms_per_iteration": round(ms / iters, 4),
            "tokens_per_s": round(gen_tok / (ms * 1e-3), 1),
            "drafter": "random weights: drafts are accepted about as often as chance, ~1 token per slot-iteration",
            "graph": f"{iters} iterations in one CUDA graph, L2 flushed before each run"}


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The float64 oracle on the host cores: each step = one request's verify step."""
    import torch  # noqa: F401
    from oracle import model as OM
    from tests.oracle_helpers import oracle_model, oracle_state_from_kv
    w = WORKLOADS[args.workload]
    shape = w.shape
    master = gen.master_weights(shape, w.seed)
    om = oracle_model(shape, master)
    del master
    lens, pend, ks = gen.context_lengths(w), gen.pending_tokens(w), gen.prefix_lengths(w)
    reqs = []
    for b in range(min(2, w.batch)):
        kk, vv = gen.synthetic_kv(shape, int(lens[b]), w.seed, b)
        st = oracle_state_from_kv(shape, kk, vv, int(pend[b]))
        g = OM.ar_greedy(om, st.copy(), min(int(ks[b]) + 1, 16))
        reqs.append((st, gen.plant_drafts(g, int(ks[b]), shape.vocab, "bench", w.seed, b)))
    for i in range(args.warmup):
        st, d = reqs[i % len(reqs)]
        OM.verify_step(om, st.copy(), d)
    tokens, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        st, d = reqs[i % len(reqs)]
        tokens += OM.verify_step(om, st.copy(), d)["accepted"] + 1
    dt = time.perf_counter() - t0
    value = tokens / dt
    cores = len(os.sched_getaffinity(0))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded random-init weights, random KV context, planted draft prefixes)",
        "config": {"workload": w.name, "batch_sample": "one request per step, requests 0-1",
                   "parallelism": "none (host cores)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} float64 verify steps (one request each), {dt:.1f} s"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)  # ~0.6 s timed: clock samples land inside
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-draft", action="store_true", help="skip the drafter-pass measurement")
    ap.add_argument("--no-extra", action="store_true", help="skip the other configurations' keys")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of timed oracle work")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    try:
        run_gpu(args, rank, world)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
