"""Drafter shapes and synthetic workloads.

Shapes follow the drafters the DFlash pages describe: a five-layer drafter
(eight for the larger target) generating 16-token blocks over Qwen3-8B- and
Llama-3.1-8B-sized targets ("DFlash Crea Blocchi Interi di Token...",
sections "Come funziona il drafting a blocchi" and "L'idea chiave"). The pages
give no layer widths; the widths below are those of the named target models.
Nothing here computes any part of the method.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class DrafterShape:
    hidden: int          # H, drafter hidden size
    n_heads: int         # nq, query heads
    n_kv_heads: int      # nkv, key/value heads
    head_dim: int        # d
    n_layers: int        # L, draft layers
    intermediate: int    # I, SwiGLU inner size
    vocab: int           # V
    n_taps: int          # k, tapped target layers
    target_hidden: int   # Ht, target hidden size
    rope_theta: float
    rms_eps: float = 1e-6


@dataclass(frozen=True)
class Workload:
    name: str
    shape: DrafterShape
    ctx: int                     # injected context length at start (per sequence)
    block: int                   # B, slots per draft block (slot 0 = last accepted token)
    batch: int                   # sequences drafted together
    steps: int                   # consecutive draft+verify steps
    p_plant: float = 0.8         # per-slot probability that the target agrees with the draft
    ctx_range: Optional[Tuple[int, int]] = None   # ragged ctx: uniform integer range per sequence
    p_range: Optional[Tuple[float, float]] = None  # ragged agreement: uniform per sequence
    weight_std: float = 0.02
    gain_std: float = 0.1        # RMSNorm gains are 1 + N(0, gain_std)

    def with_block(self, block: int) -> "Workload":
        base = self.name[: self.name.rfind("-B")] if "-B" in self.name else self.name
        return replace(self, block=block, name=f"{base}-B{block}")

    def kv_capacity(self) -> int:
        """Positions a sequence's cache must hold: the longest ctx plus every
        step's maximal acceptance plus one block of scratch slots."""
        hi = self.ctx_range[1] if self.ctx_range else self.ctx
        return hi + self.steps * self.block + self.block


TINY = DrafterShape(hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, n_layers=2,
                    intermediate=768, vocab=1024, n_taps=3, target_hidden=256,
                    rope_theta=1e6)

QWEN3_8B = DrafterShape(hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, n_layers=5,
                        intermediate=12288, vocab=151936, n_taps=5, target_hidden=4096,
                        rope_theta=1e6)

LLAMA31_8B = DrafterShape(hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, n_layers=8,
                          intermediate=14336, vocab=128256, n_taps=5, target_hidden=4096,
                          rope_theta=5e5)

# The five workloads: a tiny correctness step, the batch-1 Qwen3-8B-shaped step,
# its block-size sweep, batched serving with ragged contexts, and the
# long-context Llama-3.1-8B-shaped step.
W_TINY = Workload("tiny", TINY, ctx=64, block=4, batch=1, steps=3)
W_QWEN3_8B = Workload("qwen3-8b-b1-ctx2048-B16", QWEN3_8B, ctx=2048, block=16, batch=1, steps=100)
W_SWEEP = tuple(W_QWEN3_8B.with_block(b) for b in (4, 8, 12, 16))
W_BATCHED = Workload("qwen3-8b-b32-ctx512..8192-B16", QWEN3_8B, ctx=4352, block=16, batch=32,
                     steps=50, ctx_range=(512, 8192), p_range=(0.5, 0.95))
W_LLAMA = Workload("llama3.1-8b-L8-b4-ctx32768-B16", LLAMA31_8B, ctx=32768, block=16, batch=4,
                   steps=20)

WORKLOADS = {w.name: w for w in (W_TINY, W_QWEN3_8B, *W_SWEEP, W_BATCHED, W_LLAMA)}


def weight_bytes(s: DrafterShape) -> dict:
    """Bytes of each bf16 weight group (for roofline accounting)."""
    H, d = s.hidden, s.head_dim
    per_layer = 2 * (H * s.n_heads * d + 2 * H * s.n_kv_heads * d + s.n_heads * d * H
                     + 3 * H * s.intermediate + 2 * H)
    return {
        "fc": 2 * H * s.n_taps * s.target_hidden,
        "inject_kv": 2 * s.n_layers * 2 * s.n_kv_heads * d * H,
        "layers": s.n_layers * per_layer,
        "lm_head": 2 * s.vocab * H,
        "embed_row": 2 * H,
    }
