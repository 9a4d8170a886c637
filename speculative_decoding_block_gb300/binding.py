"""ctypes binding of libvsd.so (include/vsd.h): the same names, torch tensors in.

Argument marshalling only -- every step of the verify path runs in the
library's CUDA kernels.  Tensors must be CUDA, contiguous, of the dtype the
header states; BF16 data may be passed as torch.bfloat16 or int16/uint16
bit patterns.  The stream is torch's current stream unless one is given.
Loading fails loudly if the shared library is missing: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvsd.so")

VSD_OK, VSD_ERR_ARG, VSD_ERR_CUDA, VSD_ERR_OOM, VSD_ERR_CAPACITY, VSD_ERR_DEVICE, VSD_ERR_UNSUPPORTED = range(7)
VSD_DEV_BAD_TOKEN, VSD_DEV_BAD_SEQLEN, VSD_DEV_BAD_PAGE, VSD_DEV_TIMEOUT = 1, 2, 4, 8
FMT = {"bf16": 0, "fp8": 1, "nvfp4": 2}

EXPORTS = [
    "vsd_version", "vsd_last_error", "vsd_quantize_fp8_rowwise", "vsd_quantize_nvfp4",
    "vsd_model_create", "vsd_model_destroy", "vsd_kv_create", "vsd_kv_destroy",
    "vsd_kv_pages_per_req", "vsd_kv_num_pages", "vsd_kv_set_page_table", "vsd_kv_write",
    "vsd_kv_read", "vsd_get_device_status", "vsd_verify_step", "vsd_verify_step_debug",
    "vsd_linear", "vsd_block_attention", "vsd_block_attention_static", "vsd_accept_commit",
    "vsd_verify_step_profiled", "vsd_draft_step", "vsd_draft_step_debug", "vsd_kv_get_anchor", "vsd_spec_loop", "vsd_verify_step_sampled",
    "vsd_verify_step_host",
    "vsd_trace_enable", "vsd_trace_read", "vsd_debug_wait_probe", "vsd_kv_set_step_kernel",
    "vsd_ssm_create", "vsd_ssm_destroy", "vsd_ssm_set_state", "vsd_ssm_get_state", "vsd_ssm_verify",
    "vsd_ssm_commit", "vsd_ssm_get_device_status",
]
KERNEL_KINDS = ["embed", "qkv_gemm", "attention", "o_proj_gemm", "gate_up_gemm", "down_gemm",
                "lm_head_gemm", "accept_commit", "step"]


class VsdError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"vsd status {status}: {msg}")
        self.status = status


class ModelConfig(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_q", ctypes.c_int32),
                ("n_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rope_theta", ctypes.c_float), ("eps", ctypes.c_float),
                ("tied", ctypes.c_int32), ("attn_fmt", ctypes.c_int32), ("mlp_fmt", ctypes.c_int32),
                ("max_positions", ctypes.c_int32)]


class Weight(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("data_dev", ctypes.c_void_p), ("scale_dev", ctypes.c_void_p),
                ("tensor_scale_dev", ctypes.c_void_p)]


class Weights(ctypes.Structure):
    _fields_ = [("embed_dev", ctypes.c_void_p), ("lm_head_dev", ctypes.c_void_p),
                ("layers", ctypes.POINTER(Weight))]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m speculative_decoding_block_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        c_int, p = ctypes.c_int32, ctypes.c_void_p
        sig = {
            "vsd_version": ([], ctypes.c_char_p),
            "vsd_last_error": ([], ctypes.c_char_p),
            "vsd_quantize_fp8_rowwise": ([p, c_int, c_int, p, p, p], c_int),
            "vsd_quantize_nvfp4": ([p, c_int, c_int, p, p, p, p], c_int),
            "vsd_model_create": ([ctypes.POINTER(ModelConfig), ctypes.POINTER(Weights), p,
                                  ctypes.POINTER(p)], c_int),
            "vsd_model_destroy": ([p], None),
            "vsd_kv_create": ([p, c_int, c_int, c_int, c_int, ctypes.POINTER(p)], c_int),
            "vsd_kv_destroy": ([p], None),
            "vsd_kv_pages_per_req": ([p], c_int),
            "vsd_kv_num_pages": ([p], c_int),
            "vsd_kv_set_page_table": ([p, p, p], c_int),
            "vsd_kv_write": ([p, c_int, c_int, c_int, p, p, p], c_int),
            "vsd_kv_read": ([p, c_int, c_int, c_int, p, p, p], c_int),
            "vsd_get_device_status": ([p, p, ctypes.POINTER(c_int)], c_int),
            "vsd_verify_step": ([p, p, c_int, p, p, p, p, p, p], c_int),
            "vsd_verify_step_host": ([p, p, c_int, p, p, p, p, p, p], c_int),
            "vsd_verify_step_debug": ([p, p, c_int, p, p, p, p, p, p, p, p], c_int),
            "vsd_verify_step_profiled": ([p, p, c_int, p, p, p, p, p, c_int, p, p, ctypes.POINTER(c_int)],
                                         c_int),
            "vsd_draft_step": ([p, p, c_int, p, c_int, p, p], c_int),
            "vsd_verify_step_sampled": ([p, p, c_int, p, p, p, p, p, p, p, ctypes.c_float, p, p], c_int),
            "vsd_draft_step_debug": ([p, p, c_int, p, c_int, p, p, p, p, p], c_int),
            "vsd_kv_get_anchor": ([p, c_int, p, p], c_int),
            "vsd_spec_loop": ([p, p, p, c_int, c_int, p, p, p, p, p, p, p, p, p, p, c_int, c_int, c_int, p], c_int),
            "vsd_linear": ([ctypes.POINTER(Weight), c_int, c_int, p, c_int, p, p], c_int),
            "vsd_trace_enable": ([p, c_int], c_int),
            "vsd_debug_wait_probe": ([p, ctypes.c_int64, p], c_int),
            "vsd_kv_set_step_kernel": ([p, c_int], c_int),
            "vsd_ssm_create": ([c_int, c_int, c_int, c_int, ctypes.POINTER(p)], c_int),
            "vsd_ssm_destroy": ([p], None),
            "vsd_ssm_set_state": ([p, c_int, p, p], c_int),
            "vsd_ssm_get_state": ([p, c_int, p, p], c_int),
            "vsd_ssm_verify": ([p, c_int, p, p, p, p, p, p, p], c_int),
            "vsd_ssm_commit": ([p, c_int, p, p], c_int),
            "vsd_ssm_get_device_status": ([p, p, ctypes.POINTER(c_int)], c_int),
            "vsd_trace_read": ([p, p, c_int, ctypes.POINTER(c_int), p], c_int),
            "vsd_block_attention": ([p, p, c_int, c_int, p, p, p, p, p, p], c_int),
            "vsd_block_attention_static": ([p, p, c_int, c_int, p, p, p, p, p, p], c_int),
            "vsd_accept_commit": ([p, p, c_int, p, p, p, p, p, p, p, p, p], c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != VSD_OK:
        raise VsdError(status, lib().vsd_last_error().decode())


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _host(t, name: str, numel: int, writable: bool = True):
    """Address of a contiguous int32 host array (numpy array or CPU tensor) of at least numel elements;
    writable for the arrays the call writes."""
    if isinstance(t, torch.Tensor):
        if t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int32 CPU tensor")
        n, ptr = t.numel(), t.data_ptr()
    else:
        import numpy as np
        if not isinstance(t, np.ndarray) or t.dtype != np.int32 or not t.flags.c_contiguous:
            raise TypeError(f"{name} must be a contiguous int32 numpy array")
        if writable and not t.flags.writeable:
            raise TypeError(f"{name} is written by the call and must be writeable")
        n, ptr = t.size, t.ctypes.data
    if n < numel:
        raise ValueError(f"{name} holds {n} elements, needs {numel}")
    return ctypes.c_void_p(ptr)


def _dev(t: torch.Tensor | None, dtypes, name: str, numel: int | None = None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return ctypes.c_void_p(t.data_ptr())


B16 = (torch.bfloat16, torch.int16, torch.uint16, torch.float16)
U8 = (torch.uint8,)
I32 = (torch.int32,)
F32 = (torch.float32,)


def vsd_version() -> str:
    return lib().vsd_version().decode()


def vsd_quantize_fp8_rowwise(w, q, scale, stream=None) -> None:
    n, k = w.shape
    _check(lib().vsd_quantize_fp8_rowwise(_dev(w, B16, "w"), n, k, _dev(q, U8, "q", n * k),
                                          _dev(scale, F32, "scale", n), _stream(stream)))


def vsd_quantize_nvfp4(w, q, block_scale, tensor_scale, stream=None) -> None:
    n, k = w.shape
    _check(lib().vsd_quantize_nvfp4(_dev(w, B16, "w"), n, k, _dev(q, U8, "q", n * k // 2),
                                    _dev(block_scale, U8, "block_scale", n * k // 16),
                                    _dev(tensor_scale, F32, "tensor_scale", 1), _stream(stream)))


class Model:
    """Owns a vsd_model handle."""

    def __init__(self, handle: ctypes.c_void_p, cfg: ModelConfig):
        self.handle, self.cfg = handle, cfg

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.vsd_model_destroy(self.handle)
            self.handle = None


class KV:
    """Owns a vsd_kv handle (paged cache + step workspace)."""

    def __init__(self, handle, model: Model, max_batch: int, max_tokens: int):
        self.handle, self.model = handle, model
        self.max_batch, self.max_tokens = max_batch, max_tokens

    @property
    def pages_per_req(self) -> int:
        return lib().vsd_kv_pages_per_req(self.handle)

    @property
    def num_pages(self) -> int:
        return lib().vsd_kv_num_pages(self.handle)

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.vsd_kv_destroy(self.handle)
            self.handle = None


def weight_entry(fmt: str, data, scale=None, tensor_scale=None) -> Weight:
    f = FMT[fmt]
    dd = {0: B16, 1: U8, 2: U8}[f]
    sd = {0: None, 1: F32, 2: U8}[f]
    return Weight(f, _dev(data, dd, "data"), _dev(scale, sd, "scale") if sd else None,
                  _dev(tensor_scale, F32, "tensor_scale") if f == 2 else None)


def vsd_model_create(cfg: ModelConfig, embed, layer_weights: list, lm_head=None, stream=None) -> Model:
    """layer_weights: layers*7 Weight entries (wq, wk, wv, wo, wg, wu, wd per layer)."""
    arr = (Weight * len(layer_weights))(*layer_weights)
    w = Weights(_dev(embed, B16, "embed"), _dev(lm_head, B16, "lm_head"), arr)
    h = ctypes.c_void_p()
    _check(lib().vsd_model_create(ctypes.byref(cfg), ctypes.byref(w), _stream(stream), ctypes.byref(h)))
    return Model(h, cfg)


def vsd_kv_create(model: Model, max_batch: int, max_tokens_per_req: int, page_size: int = 16,
                  num_pages: int = 0) -> KV:
    h = ctypes.c_void_p()
    _check(lib().vsd_kv_create(model.handle, max_batch, max_tokens_per_req, page_size, num_pages,
                               ctypes.byref(h)))
    return KV(h, model, max_batch, max_tokens_per_req)


def vsd_kv_set_page_table(kv: KV, table, stream=None) -> None:
    _check(lib().vsd_kv_set_page_table(kv.handle, _dev(table, I32, "table", kv.max_batch * kv.pages_per_req),
                                       _stream(stream)))


def vsd_kv_write(kv: KV, req: int, start: int, k, v, stream=None) -> None:
    count = k.shape[1]
    _check(lib().vsd_kv_write(kv.handle, req, start, count, _dev(k, B16, "k"), _dev(v, B16, "v"),
                              _stream(stream)))


def vsd_kv_read(kv: KV, req: int, start: int, k, v, stream=None) -> None:
    count = k.shape[1]
    _check(lib().vsd_kv_read(kv.handle, req, start, count, _dev(k, B16, "k"), _dev(v, B16, "v"),
                             _stream(stream)))


def vsd_trace_enable(kv: KV, max_launches: int) -> None:
    _check(lib().vsd_trace_enable(kv.handle, max_launches))


TRACE_CTAS, TRACE_TAGS = 1024, 64


def vsd_trace_read(kv: KV, max_launches: int = 256, stream=None):
    """Timestamp table as a numpy array [launches, 1024 CTAs, 64 tags] of uint64 ns (0 = not reached)."""
    import numpy as np
    buf = np.zeros((max_launches, TRACE_CTAS, TRACE_TAGS), dtype=np.uint64)
    n = ctypes.c_int32()
    _check(lib().vsd_trace_read(kv.handle, ctypes.c_void_p(buf.ctypes.data), max_launches, ctypes.byref(n),
                                _stream(stream)))
    return buf[: n.value]


STEP_LAYERED, STEP_PERSISTENT = 0, 1


class SSM:
    """A recurrent layer's ReplaySSM state (checkpoint + input buffer) for max_batch requests."""

    def __init__(self, max_batch: int, heads: int, d: int, window: int):
        h = ctypes.c_void_p()
        _check(lib().vsd_ssm_create(max_batch, heads, d, window, ctypes.byref(h)))
        self.handle, self.max_batch, self.heads, self.d, self.window = h, max_batch, heads, d, window

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.vsd_ssm_destroy(self.handle)

    def set_state(self, req: int, state, stream=None) -> None:
        """state: float32 device tensor [heads, d, d]."""
        _check(lib().vsd_ssm_set_state(self.handle, req, _dev(state, F32, "state", self.heads * self.d * self.d),
                                       _stream(stream)))

    def get_state(self, req: int, state, stream=None) -> None:
        _check(lib().vsd_ssm_get_state(self.handle, req, _dev(state, F32, "state", self.heads * self.d * self.d),
                                       _stream(stream)))

    def verify(self, batch: int, q, k, v, alpha, beta, out, stream=None) -> None:
        n = batch * self.heads * 17
        _check(lib().vsd_ssm_verify(self.handle, batch, _dev(q, F32, "q", n * self.d), _dev(k, F32, "k", n * self.d),
                                    _dev(v, F32, "v", n * self.d), _dev(alpha, F32, "alpha", n),
                                    _dev(beta, F32, "beta", n), _dev(out, F32, "out", n * self.d), _stream(stream)))

    def commit(self, batch: int, accepted, stream=None) -> None:
        _check(lib().vsd_ssm_commit(self.handle, batch, _dev(accepted, I32, "accepted", batch), _stream(stream)))

    def device_status(self, stream=None) -> int:
        out = ctypes.c_int32()
        _check(lib().vsd_ssm_get_device_status(self.handle, _stream(stream), ctypes.byref(out)))
        return out.value


def vsd_kv_set_step_kernel(kv: KV, mode: int) -> None:
    """How the cache's steps launch the layers and the head: STEP_LAYERED
    (one launch per GEMM / attention, the default) or STEP_PERSISTENT (one
    persistent launch)."""
    _check(lib().vsd_kv_set_step_kernel(kv.handle, mode))


def vsd_debug_wait_probe(kv: KV, limit_cycles: int, stream=None) -> None:
    """Test-only: a kernel whose bounded waits can never succeed gives up after
    limit_cycles and sets VSD_DEV_TIMEOUT in the cache's status word."""
    _check(lib().vsd_debug_wait_probe(kv.handle, ctypes.c_int64(limit_cycles), _stream(stream)))


def vsd_get_device_status(kv: KV, stream=None) -> int:
    out = ctypes.c_int32()
    _check(lib().vsd_get_device_status(kv.handle, _stream(stream), ctypes.byref(out)))
    return out.value


def vsd_verify_step(model: Model, kv: KV, batch: int, seq_lens, pending, drafts, accepted, out_tokens,
                    stream=None) -> None:
    _check(lib().vsd_verify_step(model.handle, kv.handle, batch, _dev(seq_lens, I32, "seq_lens", batch),
                                 _dev(pending, I32, "pending", batch), _dev(drafts, I32, "drafts", batch * 16),
                                 _dev(accepted, I32, "accepted", batch),
                                 _dev(out_tokens, I32, "out_tokens", batch * 17), _stream(stream)))


def vsd_verify_step_host(model: Model, kv: KV, batch: int, seq_lens, pending, drafts, accepted, out_tokens,
                         stream=None) -> None:
    """The step on host arrays (int32 numpy arrays or CPU tensors); synchronous."""
    _check(lib().vsd_verify_step_host(model.handle, kv.handle, batch, _host(seq_lens, "seq_lens", batch),
                                      _host(pending, "pending", batch), _host(drafts, "drafts", batch * 16, writable=False),
                                      _host(accepted, "accepted", batch),
                                      _host(out_tokens, "out_tokens", batch * 17), _stream(stream)))


def vsd_verify_step_debug(model: Model, kv: KV, batch: int, seq_lens, pending, drafts, accepted,
                          out_tokens, logits=None, hidden=None, stream=None) -> None:
    _check(lib().vsd_verify_step_debug(model.handle, kv.handle, batch,
                                       _dev(seq_lens, I32, "seq_lens", batch),
                                       _dev(pending, I32, "pending", batch),
                                       _dev(drafts, I32, "drafts", batch * 16),
                                       _dev(accepted, I32, "accepted", batch),
                                       _dev(out_tokens, I32, "out_tokens", batch * 17),
                                       _dev(logits, F32, "logits"), _dev(hidden, F32, "hidden"),
                                       _stream(stream)))


def vsd_verify_step_sampled(model: Model, kv: KV, batch: int, seq_lens, pending, drafts, accepted, out_tokens,
                            u_accept, u_sample, temperature: float, logits=None, stream=None) -> None:
    _check(lib().vsd_verify_step_sampled(model.handle, kv.handle, batch,
                                         _dev(seq_lens, I32, "seq_lens", batch), _dev(pending, I32, "pending", batch),
                                         _dev(drafts, I32, "drafts", batch * 16),
                                         _dev(accepted, I32, "accepted", batch),
                                         _dev(out_tokens, I32, "out_tokens", batch * 17),
                                         _dev(u_accept, F32, "u_accept", batch * 16),
                                         _dev(u_sample, F32, "u_sample", batch * 17), float(temperature),
                                         _dev(logits, F32, "logits"), _stream(stream)))


def vsd_draft_step(drafter: Model, kv: KV, batch: int, seq_lens, mask_token: int, drafts, stream=None) -> None:
    _check(lib().vsd_draft_step(drafter.handle, kv.handle, batch, _dev(seq_lens, I32, "seq_lens", batch),
                                int(mask_token), _dev(drafts, I32, "drafts", batch * 16), _stream(stream)))


def vsd_draft_step_debug(drafter: Model, kv: KV, batch: int, seq_lens, mask_token: int, drafts, anchor=None,
                         logits=None, hidden=None, stream=None) -> None:
    _check(lib().vsd_draft_step_debug(drafter.handle, kv.handle, batch, _dev(seq_lens, I32, "seq_lens", batch),
                                      int(mask_token), _dev(anchor, F32, "anchor"),
                                      _dev(drafts, I32, "drafts", batch * 16), _dev(logits, F32, "logits"),
                                      _dev(hidden, F32, "hidden"), _stream(stream)))


class LoopState:
    """Device arrays of one device-resident loop: per-request inputs and outputs, slot state."""

    def __init__(self, slots: int, req_len, req_pending, req_budget, req_anchor, out_cap: int):
        q = int(req_len.numel())
        self.slots, self.queued, self.out_cap = slots, q, out_cap
        self.req_len = req_len.to(torch.int32).cuda().contiguous()
        self.req_pending = req_pending.to(torch.int32).cuda().contiguous()
        self.req_budget = req_budget.to(torch.int32).cuda().contiguous()
        self.req_anchor = req_anchor.to(torch.float32).cuda().contiguous()
        self.slot_req = torch.full((slots,), -1, dtype=torch.int32, device="cuda")
        self.next_req = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.iter = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.req_generated = torch.zeros(q, dtype=torch.int32, device="cuda")
        self.req_admit_iter = torch.full((q,), -1, dtype=torch.int32, device="cuda")
        self.req_out = torch.full((q, out_cap), -1, dtype=torch.int32, device="cuda")


def vsd_spec_loop(target: Model, drafter: Model, kv: KV, st: LoopState, n_iters: int, mask_token: int,
                  stream=None) -> None:
    q = st.queued
    _check(lib().vsd_spec_loop(target.handle, drafter.handle, kv.handle, st.slots, q,
                               _dev(st.req_len, I32, "req_len", q), _dev(st.req_pending, I32, "req_pending", q),
                               _dev(st.req_budget, I32, "req_budget", q),
                               _dev(st.req_anchor, F32, "req_anchor"), _dev(st.slot_req, I32, "slot_req", st.slots),
                               _dev(st.next_req, I32, "next_req", 1), _dev(st.iter, I32, "iter", 1),
                               _dev(st.req_generated, I32, "req_generated", q),
                               _dev(st.req_admit_iter, I32, "req_admit_iter", q),
                               _dev(st.req_out, I32, "req_out", q * st.out_cap), st.out_cap, int(n_iters),
                               int(mask_token), _stream(stream)))


def vsd_kv_get_anchor(kv: KV, batch: int, dst, stream=None) -> None:
    _check(lib().vsd_kv_get_anchor(kv.handle, batch, _dev(dst, F32, "anchor"), _stream(stream)))


def vsd_verify_step_profiled(model: Model, kv: KV, batch: int, seq_lens, pending, drafts, accepted,
                             out_tokens, max_launches: int = 4096, stream=None):
    """Runs one step with per-launch events; returns [(kind name, ms)] in launch order."""
    kinds = (ctypes.c_int32 * max_launches)()
    ms = (ctypes.c_float * max_launches)()
    n = ctypes.c_int32()
    _check(lib().vsd_verify_step_profiled(model.handle, kv.handle, batch,
                                          _dev(seq_lens, I32, "seq_lens", batch),
                                          _dev(pending, I32, "pending", batch),
                                          _dev(drafts, I32, "drafts", batch * 16),
                                          _dev(accepted, I32, "accepted", batch),
                                          _dev(out_tokens, I32, "out_tokens", batch * 17), max_launches,
                                          ctypes.cast(kinds, ctypes.c_void_p), ctypes.cast(ms, ctypes.c_void_p),
                                          ctypes.byref(n), _stream(stream)))
    return [(KERNEL_KINDS[kinds[i]], float(ms[i])) for i in range(min(n.value, max_launches))]


def vsd_linear(weight: Weight, n: int, k: int, x, y, stream=None) -> None:
    m = x.shape[0]
    _check(lib().vsd_linear(ctypes.byref(weight), n, k, _dev(x, (torch.float16,), "x", m * k), m,
                            _dev(y, F32, "y", m * n), _stream(stream)))


def vsd_block_attention(model: Model, kv: KV, layer: int, batch: int, seq_lens, q, k_new, v_new, out,
                        stream=None) -> None:
    _check(lib().vsd_block_attention(model.handle, kv.handle, layer, batch,
                                     _dev(seq_lens, I32, "seq_lens", batch), _dev(q, B16, "q"),
                                     _dev(k_new, B16, "k_new"), _dev(v_new, B16, "v_new"),
                                     _dev(out, (torch.float16,), "out"), _stream(stream)))


def vsd_block_attention_static(model: Model, kv: KV, layer: int, batch: int, seq_lens, q, k_new, v_new, out,
                               stream=None) -> None:
    """vsd_block_attention with its scratch in the library's static device
    array: no device allocation on any call (for callers that cannot
    allocate while running).  Calls on one device share that array, so they
    must not overlap on the GPU."""
    _check(lib().vsd_block_attention_static(model.handle, kv.handle, layer, batch,
                                            _dev(seq_lens, I32, "seq_lens", batch), _dev(q, B16, "q"),
                                            _dev(k_new, B16, "k_new"), _dev(v_new, B16, "v_new"),
                                            _dev(out, (torch.float16,), "out"), _stream(stream)))


def vsd_accept_commit(model: Model, kv: KV, batch: int, logits, k_new, v_new, seq_lens, pending, drafts,
                      accepted, out_tokens, stream=None) -> None:
    _check(lib().vsd_accept_commit(model.handle, kv.handle, batch, _dev(logits, F32, "logits"),
                                   _dev(k_new, B16, "k_new"), _dev(v_new, B16, "v_new"),
                                   _dev(seq_lens, I32, "seq_lens", batch), _dev(pending, I32, "pending", batch),
                                   _dev(drafts, I32, "drafts", batch * 16), _dev(accepted, I32, "accepted", batch),
                                   _dev(out_tokens, I32, "out_tokens", batch * 17), _stream(stream)))
