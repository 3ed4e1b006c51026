"""End-to-end speculative generation with the DFlash drafter (the user-level loop the pages
show as spec_generate(input_ids, max_new_tokens, temperature, target, stop_token_ids):
7minutos.es, "Ejecutando DFlash").

Every step of the draft-and-verify path runs in the library's kernels through the C ABI;
this module only sequences the calls around the caller's target model:

  prefill   the target reads the prompt; the hidden states of its tapped layers at every
            prompt position are injected into the drafter's KV cache, and the target's own
            next token becomes slot 0 of the first block
  repeat    draft a block of B slots (slot 0 = last committed token, slots 1..B-1 drafted)
            -> the target runs once over those B tokens -> verification keeps the longest
            valid prefix plus one token of the target's own (greedy, or speculative
            sampling at temperature > 0) -> the target drops the rejected positions -> the
            hidden states of the tau kept positions are injected -> the last committed
            token becomes the next slot 0

Greedy generation is lossless: the committed tokens are exactly the target's own greedy
continuation (theaistack.guide, "DFlash").

The target is any object with three methods:
  prefill(input_ids int64 [P]) -> (tapped bf16 [k, P, Ht], logits fp32 [V] after the last token)
  forward_block(tokens int64 [B]) -> (tapped bf16 [k, B, Ht], logits fp32 [B, V]); row i
      predicts the token after tokens[i]; the B positions are appended to its cache
  truncate(length) keeps the first `length` positions of its cache
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch


@dataclass
class GenerationStats:
    steps: int = 0                       # draft-and-verify steps
    accept_lens: List[int] = field(default_factory=list)

    @property
    def mean_tau(self) -> float:
        return sum(self.accept_lens) / max(1, len(self.accept_lens))


def spec_generate(drafter, target, input_ids, max_new_tokens: int, temperature: float = 0.0,
                  stop_token_ids: Sequence[int] = (), block: Optional[int] = None,
                  generator: Optional[torch.Generator] = None, stream=None):
    """Generate up to max_new_tokens tokens after input_ids (a 1-D token sequence) with the
    drafter (a binding.Drafter bound with max_batch >= 1; sequence slot 0 is used and reset)
    and the caller's target. Generation stops after the first token in stop_token_ids.
    temperature > 0 verifies by speculative sampling with uniforms drawn from `generator`.
    Returns (new tokens as a list of ints, GenerationStats)."""
    dev = drafter.last_token.device
    B = block or drafter.cfg.max_block
    V = drafter.shape.vocab
    stops = set(int(t) for t in stop_token_ids)
    out: List[int] = []
    stats = GenerationStats()
    if max_new_tokens <= 0:
        return out, stats

    def pick(logits_row):
        if temperature > 0:
            p = torch.softmax(logits_row.double() / temperature, dim=-1)
            u = torch.rand((), generator=generator, device=logits_row.device, dtype=torch.float64)
            return int(min(int(torch.searchsorted(torch.cumsum(p, 0), u, right=True)), V - 1))
        return int(torch.argmax(logits_row))

    def emit(tokens) -> bool:
        for t in tokens:
            out.append(int(t))
            if int(t) in stops or len(out) >= max_new_tokens:
                return True
        return False

    ids = torch.as_tensor(input_ids, dtype=torch.int64, device=dev).reshape(-1)
    tapped, logits = target.prefill(ids)
    P = ids.numel()
    drafter.len.zero_()
    drafter.inject(tapped.contiguous(), P, torch.tensor([P], dtype=torch.int32, device=dev), 1, stream)
    first = pick(logits.reshape(-1))
    drafter.last_token[0] = first
    if emit([first]):
        return out, stats
    drafted = torch.zeros(1, max(B - 1, 1), dtype=torch.int32, device=dev)
    acc = torch.zeros(1, dtype=torch.int32, device=dev)
    com = torch.zeros(1, B, dtype=torch.int32, device=dev)
    n_cached = P
    while True:
        drafter.draft(1, B, drafted, stream=stream)
        block_tokens = torch.cat([drafter.last_token[:1].to(torch.int64), drafted[0, : B - 1].to(torch.int64)])
        tapped, logits = target.forward_block(block_tokens)
        logits = logits.to(torch.float32).reshape(1, B, V).contiguous()
        if temperature > 0:
            u = torch.rand(1, B, generator=generator, device=dev, dtype=torch.float32)
            drafter.verify_sampling(logits, drafted, u, temperature, 1, B, acc, com, stream)
        else:
            drafter.verify(logits, drafted, 1, B, acc, com, stream)
        tau = int(acc[0])
        stats.steps += 1
        stats.accept_lens.append(tau)
        target.truncate(n_cached + tau)   # keep slot 0 and the accepted drafts
        rows = torch.zeros(tapped.shape[0], B, tapped.shape[2], dtype=torch.bfloat16, device=dev)
        rows[:, :tau] = tapped[:, :tau]
        drafter.inject(rows, B, acc, 1, stream)
        n_cached += tau
        if emit(com[0, :tau].tolist()):
            return out, stats
