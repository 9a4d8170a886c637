"""Shapes and batch recipes of the five verify-step workloads.

These are plain data: model dimensions, weight precision per matrix group,
batch size and context-length recipe.  Nothing here computes any part of the
verification step.  Both the float64 oracle and the CUDA library read these
descriptions; neither depends on the other.

Sources for the numbers:
  * block of 16 drafted tokens verified in one target pass -- HunyuanOCR-1.5
    summary (page "yeyulingfeng", section one, inference loop steps 2-4);
  * BF16 / FP8 / NVFP4 weight mix -- "The Inference Stack Behind OCRia",
    section "Reducing the data moved: workload-aware quantization";
  * GQA with shared KV heads and paged KV -- "LLM inference acceleration",
    section two (stack diagram);
  * the model sizes, batch sizes and context recipes themselves are the
    workload definitions this library is measured on (0.5B-class and
    7B-class random-init targets).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

BLOCK = 16          # drafted tokens per request per step
ROWS = BLOCK + 1    # rows per request: the pending token plus the drafts


@dataclass(frozen=True)
class ModelShape:
    name: str
    layers: int
    hidden: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    tied: bool
    attn_fmt: str   # "bf16" | "fp8"     (QKV and O projections)
    mlp_fmt: str    # "bf16" | "nvfp4"   (gate, up, down)
    eps: float = 1e-6
    init_std: float = 0.02

    @property
    def group(self) -> int:
        return self.n_q // self.n_kv

    @property
    def qkv_out(self) -> int:
        return (self.n_q + 2 * self.n_kv) * self.head_dim

    @property
    def kv_bytes_per_token(self) -> int:
        """BF16 K and V of one token over all layers."""
        return self.layers * 2 * self.n_kv * self.head_dim * 2


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    batch: int
    ctx_lo: int
    ctx_hi: int              # context length drawn uniform in [ctx_lo, ctx_hi]
    kv_source: str           # "prefill" (oracle prefill of random prompt ids) | "synthetic"
    paged: bool = False      # shuffled page table instead of the identity one
    page_size: int = 16
    steps: int = 1           # consecutive committing verify steps
    draft_means: tuple = (8.9,)  # planted-prefix mean(s); "uniform" for the tiny case
    draft_dist: str = "geometric"  # "geometric" | "uniform"
    seed: int = 0

    @property
    def rows(self) -> int:
        return ROWS * self.batch

    def max_tokens_per_req(self) -> int:
        # room for every committed row of every step plus one in-flight block
        return self.ctx_hi + self.steps * ROWS + ROWS


TINY = ModelShape("tiny-2L-h256", layers=2, hidden=256, n_q=4, n_kv=2, head_dim=64,
                  ffn=688, vocab=4096, rope_theta=1e4, tied=True,
                  attn_fmt="bf16", mlp_fmt="bf16")
HALF_B_BF16 = ModelShape("0.5B-class-bf16", layers=24, hidden=896, n_q=14, n_kv=2,
                         head_dim=64, ffn=4864, vocab=151936, rope_theta=1e4, tied=True,
                         attn_fmt="bf16", mlp_fmt="bf16")
HALF_B_MIXED = ModelShape("0.5B-class-mixed", layers=24, hidden=896, n_q=14, n_kv=2,
                          head_dim=64, ffn=4864, vocab=151936, rope_theta=1e4, tied=True,
                          attn_fmt="fp8", mlp_fmt="nvfp4")
SEVEN_B_MIXED = ModelShape("7B-class-mixed", layers=32, hidden=4096, n_q=32, n_kv=8,
                           head_dim=128, ffn=14336, vocab=32000, rope_theta=5e5, tied=False,
                           attn_fmt="fp8", mlp_fmt="nvfp4")

WORKLOADS = {
    "tiny_b1_ctx128": Workload(
        "tiny_b1_ctx128", TINY, batch=1, ctx_lo=128, ctx_hi=128, kv_source="prefill",
        draft_dist="uniform", seed=101),
    "0.5b_bf16_b1_ctx2048": Workload(
        "0.5b_bf16_b1_ctx2048", HALF_B_BF16, batch=1, ctx_lo=2048, ctx_hi=2048,
        kv_source="synthetic", seed=202),
    "0.5b_mixed_b8_ctx512-4096": Workload(
        "0.5b_mixed_b8_ctx512-4096", HALF_B_MIXED, batch=8, ctx_lo=512, ctx_hi=4096,
        kv_source="synthetic", seed=303),
    "0.5b_mixed_b32_ctx1024-8192_paged16_64steps": Workload(
        "0.5b_mixed_b32_ctx1024-8192_paged16_64steps", HALF_B_MIXED, batch=32,
        ctx_lo=1024, ctx_hi=8192, kv_source="synthetic", paged=True, steps=64,
        draft_means=(7.7, 8.6, 10.4), seed=404),
    "7b_mixed_b16_ctx4096": Workload(
        "7b_mixed_b16_ctx4096", SEVEN_B_MIXED, batch=16, ctx_lo=4096, ctx_hi=4096,
        kv_source="synthetic", seed=505),
}

# order of the workload list these correspond to
WORKLOAD_ORDER = list(WORKLOADS)


def linear_shapes(s: ModelShape) -> dict:
    """(out_features, in_features, format) of every weight matrix of one layer."""
    return {
        "wq": (s.n_q * s.head_dim, s.hidden, s.attn_fmt),
        "wk": (s.n_kv * s.head_dim, s.hidden, s.attn_fmt),
        "wv": (s.n_kv * s.head_dim, s.hidden, s.attn_fmt),
        "wo": (s.hidden, s.n_q * s.head_dim, s.attn_fmt),
        "wg": (s.ffn, s.hidden, s.mlp_fmt),
        "wu": (s.ffn, s.hidden, s.mlp_fmt),
        "wd": (s.hidden, s.ffn, s.mlp_fmt),
    }


# ------------------------------------------------------------------ drafter
DRAFTER_LAYERS = 5  # the block drafter copies the target's last five decoder layers


def drafter_shape(s: ModelShape, layers: int = DRAFTER_LAYERS) -> ModelShape:
    """The drafter: the target's layer shapes and formats, its last `layers` layers."""
    return replace(s, name=s.name + "-drafter", layers=min(layers, s.layers))


def mask_token(s: ModelShape) -> int:
    """Token id whose embedding fills the drafter's 16 block rows (the last id)."""
    return s.vocab - 1
