"""The generation loop's host logic on the CPU: with a stand-in drafter (a fixed draft, the
oracle's verification) and the synthetic target, speculative generation must return the
target's own greedy continuation, honour stop tokens and max_new_tokens, and keep the
target's cache and the drafter's injected length in step."""
from types import SimpleNamespace

import numpy as np
import torch

from block_diffusion_drafter_kv_gb300.generate import spec_generate
from oracle.dflash_ref import verify_greedy
from synthetic_target import TinyTarget, greedy_reference


class FakeDrafter:
    """Drafts a fixed token in every slot; verification by the oracle."""

    def __init__(self, vocab, block, token):
        self.shape = SimpleNamespace(vocab=vocab)
        self.cfg = SimpleNamespace(max_block=block)
        self.last_token = torch.zeros(1, dtype=torch.int32)
        self.len = torch.zeros(1, dtype=torch.int32)
        self.token = token

    def inject(self, hidden, rows_per_seq, n_new, batch, stream=None):
        assert hidden.dtype == torch.bfloat16 and hidden.shape[1] == rows_per_seq
        self.len[0] += int(n_new[0])

    def draft(self, batch, block, drafted, logits=None, x_trace=None, stream=None):
        drafted[0, : block - 1] = self.token

    def verify(self, logits, drafted, batch, block, acc, com, stream=None):
        r = verify_greedy(logits[0].numpy(), drafted[0, : block - 1].numpy())
        acc[0] = r.accept_len
        com[0] = -1
        com[0, : r.accept_len] = torch.as_tensor(r.committed, dtype=torch.int32)
        self.last_token[0] = r.last_token


def test_greedy_generation_equals_the_target_greedy_continuation():
    t = TinyTarget(1024, 256, seed=3, bias_token=77, bias=4.8, device="cpu")
    ids = torch.randint(0, 1024, (24,), generator=torch.Generator().manual_seed(1))
    ref = greedy_reference(t, ids, 120)
    d = FakeDrafter(1024, 8, 77)
    out, stats = spec_generate(d, t, ids, 120)
    assert out == ref
    assert stats.mean_tau > 1.0 and min(stats.accept_lens) == 1
    # the drafter holds the prompt plus every kept position; the target's cache the same
    assert int(d.len[0]) == t.n == 24 + sum(stats.accept_lens)


def test_stop_token_and_max_new_tokens():
    t = TinyTarget(1024, 256, seed=3, bias_token=77, bias=4.8, device="cpu")
    ids = torch.randint(0, 1024, (24,), generator=torch.Generator().manual_seed(1))
    ref = greedy_reference(t, ids, 60)
    stop = ref[10]
    first = ref.index(stop)
    out, _ = spec_generate(FakeDrafter(1024, 8, 77), t, ids, 60, stop_token_ids=[stop])
    assert out == ref[: first + 1]
    out, _ = spec_generate(FakeDrafter(1024, 8, 77), t, ids, 7)
    assert out == ref[:7]
    assert spec_generate(FakeDrafter(1024, 8, 77), t, ids, 0)[0] == []
