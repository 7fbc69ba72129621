"""Workload shapes: the five drafting workloads plus small test shapes.

Each entry fixes the drafter's architecture (hidden size, heads, layers,
vocabulary, RoPE base) and the synthetic serving scenario around it (batch,
context lengths, rounds, per-position match probability of the stand-in
target).  Mask id is the last vocabulary id; the first verified token of
every request is id 1.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class DraftConfig:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    n_layers: int
    vocab: int
    rope_theta: float
    batch: int
    ctx0: Optional[int]              # prompt length per request; None -> drawn U[ctx_lo, ctx_hi]
    rounds: int
    match_p: Optional[float]         # None -> per-request U[p_lo, p_hi]
    ctx_range: Tuple[int, int] = (512, 4096)
    p_range: Tuple[float, float] = (0.6, 0.95)
    n_fused: int = 5
    block: int = 16
    page_size: int = 64
    rms_eps: float = 1e-6
    weight_std: float = 0.02
    gain_std: float = 0.0            # RMSNorm gains = 1 + gain_std * N(0,1); 0 -> all ones
    first_token: int = 1
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def mask_id(self) -> int:
        return self.vocab - 1

    @property
    def fused_dim(self) -> int:
        return self.n_fused * self.hidden

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def with_(self, **kw) -> "DraftConfig":
        return replace(self, **kw)

    def weight_bytes(self) -> int:
        H, I, V, F = self.hidden, self.intermediate, self.vocab, self.fused_dim
        per_layer = self.qkv_rows * H + H * self.n_q_heads * self.head_dim + 2 * I * H + I * H
        return 2 * (V * H + H * F + self.n_layers * per_layer)


CONFIGS = {
    # 1: tiny drafter, batch 1
    "tiny": DraftConfig(
        name="tiny", hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, intermediate=768,
        n_layers=2, vocab=4096, rope_theta=1e6, batch=1, ctx0=128, rounds=8, match_p=0.8),
    # 2: Qwen3-8B-shaped drafter, batch 1 (the headline workload)
    "qwen3-8b": DraftConfig(
        name="qwen3-8b", hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
        intermediate=12288, n_layers=5, vocab=151936, rope_theta=1e6, batch=1, ctx0=2048,
        rounds=64, match_p=0.9),
    # 3: Llama-3.1-8B-shaped drafter, batch 1
    "llama3.1-8b": DraftConfig(
        name="llama3.1-8b", hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
        intermediate=14336, n_layers=5, vocab=128256, rope_theta=5e5, batch=1, ctx0=8192,
        rounds=64, match_p=0.85),
    # 4: batched serving with ragged contexts and ragged acceptance
    "batched-qwen3-8b": DraftConfig(
        name="batched-qwen3-8b", hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
        intermediate=12288, n_layers=5, vocab=151936, rope_theta=1e6, batch=64, ctx0=None,
        rounds=32, match_p=None, ctx_range=(512, 4096), p_range=(0.6, 0.95)),
    # 5: long-reasoning 8-layer drafter, batch 4, 32K context
    "long-8layer": DraftConfig(
        name="long-8layer", hidden=2048, n_q_heads=32, n_kv_heads=4, head_dim=128,
        intermediate=6144, n_layers=8, vocab=151936, rope_theta=1e6, batch=4, ctx0=32768,
        rounds=128, match_p=0.9),
}

# Small shapes for parity tests: several tiles per GEMM, ragged vocabulary
# tail, ragged pages, GQA group 4 and 8, head_dim 64 and 128, random gains.
# Projections at std 0.05 keep the layers' outputs larger than the tied
# embedding row, so the argmax is not dominated by the mask token's own row
# and the drafted ids are diverse.
TEST_CONFIGS = {
    "tiny-gains": CONFIGS["tiny"].with_(name="tiny-gains", gain_std=0.1, weight_std=0.05),
    "small": DraftConfig(
        name="small", hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=128, intermediate=1024,
        n_layers=2, vocab=8000, rope_theta=1e6, batch=1, ctx0=200, rounds=4, match_p=0.85,
        gain_std=0.1),
    "small-batch": DraftConfig(
        name="small-batch", hidden=512, n_q_heads=8, n_kv_heads=1, head_dim=128,
        intermediate=768, n_layers=2, vocab=5000, rope_theta=5e5, batch=3, ctx0=None,
        rounds=4, match_p=None, ctx_range=(30, 300), p_range=(0.5, 0.95), gain_std=0.1,
        weight_std=0.05),
    # Mid-size shape for detailed hardware-counter captures: the tied
    # embedding (134 MB) is larger than L2, the whole drafter stays under 1 GB.
    "mid": DraftConfig(
        name="mid", hidden=2048, n_q_heads=16, n_kv_heads=4, head_dim=128, intermediate=6144,
        n_layers=2, vocab=32768, rope_theta=1e6, batch=1, ctx0=1024, rounds=8, match_p=0.9),
    # The mid shape at batch 64 (1,024 block rows, as the batched workload):
    # the batched GEMMs' hardware counters with a device footprint of ~1 GB.
    "mid-b64": DraftConfig(
        name="mid-b64", hidden=2048, n_q_heads=16, n_kv_heads=4, head_dim=128, intermediate=6144,
        n_layers=2, vocab=32768, rope_theta=1e6, batch=64, ctx0=None, rounds=4, match_p=None,
        ctx_range=(256, 1024), p_range=(0.6, 0.95)),
    # The long-context attention (32 query / 4 KV heads x 128, 4 requests at
    # 32K) with two layers and a small vocabulary: its hardware counters with
    # a device footprint of ~1.5 GB.
    "mid-long": DraftConfig(
        name="mid-long", hidden=2048, n_q_heads=32, n_kv_heads=4, head_dim=128, intermediate=6144,
        n_layers=2, vocab=32768, rope_theta=1e6, batch=4, ctx0=32768, rounds=4, match_p=0.9),
    # Batch 16: 256 block tokens, so every GEMM of the round runs with a full
    # 256-token tile shared by a cluster of CTAs.
    "small-b16": DraftConfig(
        name="small-b16", hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=128,
        intermediate=768, n_layers=2, vocab=5000, rope_theta=5e5, batch=16, ctx0=None,
        rounds=3, match_p=None, ctx_range=(30, 200), p_range=(0.5, 0.95), gain_std=0.1,
        weight_std=0.05),
    # 16 (request, KV head) pairs over ~290 pages each: more attention splits
    # than thread-block clusters fit at once, each holding 32+ pages, so they
    # merge through global memory.
    "small-long": DraftConfig(
        name="small-long", hidden=512, n_q_heads=8, n_kv_heads=4, head_dim=128,
        intermediate=768, n_layers=2, vocab=5000, rope_theta=1e6, batch=4, ctx0=18500,
        rounds=3, match_p=0.85, gain_std=0.1, weight_std=0.05),
    # Inference at blocks smaller than the trained 16 (S-1 drafts per round).
    "tiny-b8": CONFIGS["tiny"].with_(name="tiny-b8", block=8, gain_std=0.1, weight_std=0.05),
    "small-batch-b10": DraftConfig(
        name="small-batch-b10", hidden=512, n_q_heads=8, n_kv_heads=1, head_dim=128,
        intermediate=768, n_layers=2, vocab=5000, rope_theta=5e5, batch=3, ctx0=None,
        rounds=4, match_p=None, ctx_range=(30, 300), p_range=(0.5, 0.95), gain_std=0.1,
        weight_std=0.05, block=10),
    # Batch 32: a round appends up to 512 feature rows, more than one token
    # tile, so the injection gathers the appended rows and computes only them.
    "small-b32": DraftConfig(
        name="small-b32", hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=128, intermediate=768,
        n_layers=2, vocab=5000, rope_theta=1e6, batch=32, ctx0=None, rounds=3, match_p=None,
        ctx_range=(30, 200), p_range=(0.3, 0.95), gain_std=0.1, weight_std=0.05),
    # Attention shapes beyond the workloads': one query head per KV head, and
    # head_dim 64 with 4 and 8 query heads per KV head.
    "small-g1": DraftConfig(
        name="small-g1", hidden=512, n_q_heads=4, n_kv_heads=4, head_dim=128, intermediate=768,
        n_layers=2, vocab=5000, rope_theta=1e6, batch=2, ctx0=None, rounds=3, match_p=None,
        ctx_range=(30, 300), p_range=(0.5, 0.95), gain_std=0.1, weight_std=0.05),
    "small-d64-g4": DraftConfig(
        name="small-d64-g4", hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64, intermediate=768,
        n_layers=2, vocab=5000, rope_theta=1e6, batch=2, ctx0=None, rounds=3, match_p=None,
        ctx_range=(30, 300), p_range=(0.5, 0.95), gain_std=0.1, weight_std=0.05),
    "small-d64-g8": DraftConfig(
        name="small-d64-g8", hidden=1024, n_q_heads=16, n_kv_heads=2, head_dim=64, intermediate=768,
        n_layers=2, vocab=5000, rope_theta=1e6, batch=2, ctx0=None, rounds=3, match_p=None,
        ctx_range=(30, 300), p_range=(0.5, 0.95), gain_std=0.1, weight_std=0.05),
    # Wide hidden sizes (the fusion projection 5H -> H at H = 4096 and 8192)
    # with a small vocabulary and few layers, for the static-scratch injection.
    "wide-4096": DraftConfig(
        name="wide-4096", hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, intermediate=1024,
        n_layers=2, vocab=4096, rope_theta=1e6, batch=1, ctx0=64, rounds=2, match_p=0.9),
    "wide-8192": DraftConfig(
        name="wide-8192", hidden=8192, n_q_heads=32, n_kv_heads=8, head_dim=128, intermediate=1024,
        n_layers=1, vocab=2048, rope_theta=1e6, batch=1, ctx0=64, rounds=2, match_p=0.9),
}


def get_config(name: str) -> DraftConfig:
    if name in CONFIGS:
        return CONFIGS[name]
    if name in TEST_CONFIGS:
        return TEST_CONFIGS[name]
    raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS) + sorted(TEST_CONFIGS)}")
