"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. Every tensor gets its own sub-seed derived from a base
seed and the tensor's name, so the draw order never matters and any single
tensor can be regenerated alone. Large draws use torch's CPU generator
(multi-threaded); values are rounded once to bf16 (round-to-nearest-even) and
both sides consume the identical rounded values.

Distributions follow the workload statement: weights N(0, 0.02), target hidden
states N(0, 1), target logits N(0, 1) plus +10 on the drafted token at each
slot with probability p. RMSNorm gains are 1 + N(0, 0.1) (a reading: the pages
do not give initialisations; a non-unit gain keeps the gain multiply visible
to the parity tests).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List

import numpy as np
import torch

from .configs import DrafterShape, Workload

_MASK64 = (1 << 64) - 1


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _fnv1a64(s: str) -> int:
    h = 0xCBF29CE484222325
    for b in s.encode():
        h = ((h ^ b) * 0x100000001B3) & _MASK64
    return h


def sub_seed(base: int, name: str) -> int:
    """63-bit seed for tensor `name` under base seed `base`."""
    return _splitmix64((base & _MASK64) ^ _fnv1a64(name)) >> 1


def _gen(base: int, name: str) -> torch.Generator:
    return torch.Generator().manual_seed(sub_seed(base, name))


def normal_bf16(shape, std: float, base: int, name: str, mean: float = 0.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=_gen(base, name), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU bf16 tensor as a numpy uint16 array (no copy of values)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass
class LayerWeights:
    wq: torch.Tensor      # [nq*d, H]
    wk: torch.Tensor      # [nkv*d, H]
    wv: torch.Tensor      # [nkv*d, H]
    wo: torch.Tensor      # [H, nq*d]
    w_gate: torch.Tensor  # [I, H]
    w_up: torch.Tensor    # [I, H]
    w_down: torch.Tensor  # [H, I]
    g_attn: torch.Tensor  # [H]
    g_mlp: torch.Tensor   # [H]


@dataclass
class Weights:
    w_fc: torch.Tensor     # [H, k*Ht]
    g_ctx: torch.Tensor    # [H]
    embed: torch.Tensor    # [V, H]
    mask_emb: torch.Tensor  # [H]
    g_final: torch.Tensor  # [H]
    lm_head: torch.Tensor  # [V, H]
    layers: List[LayerWeights]

    def tensors(self) -> Dict[str, torch.Tensor]:
        out = {"w_fc": self.w_fc, "g_ctx": self.g_ctx, "embed": self.embed,
               "mask_emb": self.mask_emb, "g_final": self.g_final, "lm_head": self.lm_head}
        for i, lw in enumerate(self.layers):
            for k, v in lw.__dict__.items():
                out[f"layers.{i}.{k}"] = v
        return out

    def to(self, device) -> "Weights":
        mv = lambda t: t.to(device, non_blocking=True)
        return Weights(mv(self.w_fc), mv(self.g_ctx), mv(self.embed), mv(self.mask_emb),
                       mv(self.g_final), mv(self.lm_head),
                       [LayerWeights(**{k: mv(v) for k, v in lw.__dict__.items()})
                        for lw in self.layers])

    def bits(self) -> Dict[str, np.ndarray]:
        """uint16 bf16 bit patterns of every CPU tensor, keyed like `tensors()`."""
        return {k: bf16_bits(v) for k, v in self.tensors().items()}


def make_weights(s: DrafterShape, seed: int, std: float = 0.02, gain_std: float = 0.1) -> Weights:
    H, d = s.hidden, s.head_dim
    g = lambda name: normal_bf16((H,), gain_std, seed, name, mean=1.0)
    w = lambda shape, name: normal_bf16(shape, std, seed, name)
    layers = []
    for l in range(s.n_layers):
        p = f"layers.{l}."
        layers.append(LayerWeights(
            wq=w((s.n_heads * d, H), p + "wq"),
            wk=w((s.n_kv_heads * d, H), p + "wk"),
            wv=w((s.n_kv_heads * d, H), p + "wv"),
            wo=w((H, s.n_heads * d), p + "wo"),
            w_gate=w((s.intermediate, H), p + "w_gate"),
            w_up=w((s.intermediate, H), p + "w_up"),
            w_down=w((H, s.intermediate), p + "w_down"),
            g_attn=g(p + "g_attn"),
            g_mlp=g(p + "g_mlp"),
        ))
    return Weights(
        w_fc=w((H, s.n_taps * s.target_hidden), "w_fc"),
        g_ctx=g("g_ctx"),
        embed=w((s.vocab, H), "embed"),
        mask_emb=w((H,), "mask_emb"),
        g_final=g("g_final"),
        lm_head=w((s.vocab, H), "lm_head"),
        layers=layers,
    )


def make_hidden(s: DrafterShape, n_pos: int, seed: int, name: str = "hidden") -> torch.Tensor:
    """Target hidden states of the k tapped layers for n_pos positions: [k, n_pos, Ht] bf16, N(0,1)."""
    return normal_bf16((s.n_taps, n_pos, s.target_hidden), 1.0, seed, name)


def make_logit_noise(batch: int, block: int, vocab: int, seed: int, name: str = "logits") -> torch.Tensor:
    """Target logits before planting: [batch, block, V] fp32, N(0,1)."""
    return torch.randn(batch, block, vocab, generator=_gen(seed, name), dtype=torch.float32)


def make_plant_mask(batch: int, block: int, p, seed: int, name: str = "plant") -> np.ndarray:
    """Bernoulli plant decisions [batch, block] (uint8). Row i < block-1 of sequence s is planted
    (target agrees with draft d_{i+1}) when the mask is 1; row block-1 never is (no draft there)."""
    u = torch.rand(batch, block, generator=_gen(seed, name), dtype=torch.float64).numpy()
    p = np.broadcast_to(np.asarray(p, dtype=np.float64).reshape(-1, 1), (batch, 1))
    m = (u < p).astype(np.uint8)
    m[:, block - 1] = 0
    return m


def plant_logits(noise: np.ndarray, drafted: np.ndarray, mask: np.ndarray, bump: float = 10.0) -> np.ndarray:
    """Synthetic target: add `bump` to logit of draft d_{i+1} at row i where mask[s, i] is set.

    noise [b, B, V] float32, drafted [b, B-1] int, mask [b, B] uint8 -> new float32 array.
    """
    out = np.array(noise, dtype=np.float32, copy=True)
    b, B, _ = out.shape
    for s in range(b):
        for i in range(B - 1):
            if mask[s, i]:
                out[s, i, int(drafted[s, i])] += np.float32(bump)
    return out


def initial_tokens(batch: int, vocab: int, seed: int) -> np.ndarray:
    g = _gen(seed, "last_token")
    return torch.randint(0, vocab, (batch,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def ragged_ctx(w: Workload, seed: int) -> np.ndarray:
    if w.ctx_range is None:
        return np.full(w.batch, w.ctx, dtype=np.int32)
    lo, hi = w.ctx_range
    g = _gen(seed, "ctx_len")
    return torch.randint(lo, hi + 1, (w.batch,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def per_seq_p(w: Workload, seed: int) -> np.ndarray:
    if w.p_range is None:
        return np.full(w.batch, w.p_plant, dtype=np.float64)
    lo, hi = w.p_range
    u = torch.rand(w.batch, generator=_gen(seed, "p_plant"), dtype=torch.float64).numpy()
    return lo + (hi - lo) * u
