"""End-to-end speculative generation through the library (spec_generate: prefill
injection, block drafts, the target's block pass, verification, rollback and incremental
injection) with the synthetic float64 target. Greedy generation must reproduce the target's
own greedy decoding token for token, over a few hundred tokens, with blocks accepted
beyond the bonus token.

The drafter has random weights, so on its own it would almost never agree with the
target. Its output projections (attention output and SwiGLU down) are set to zero, which
leaves every masked slot's state at the mask embedding, so it drafts one fixed token c;
the target's LM head carries a bias toward c, so its greedy output has runs of c that the
drafts match, and other tokens that they do not."""
import numpy as np
import pytest
import torch

from synth import W_TINY
from synth import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    from block_diffusion_drafter_kv_gb300 import binding as B
    from block_diffusion_drafter_kv_gb300.build import build
    from oracle.dflash_ref import bf16_to_float, rms_norm
    from synthetic_target import TinyTarget
    build()
    s = W_TINY.shape
    w = I.make_weights(s, 21)
    for lw in w.layers:
        lw.wo.zero_()
        lw.w_down.zero_()
    bits = w.bits()
    h = rms_norm(bf16_to_float(bits["mask_emb"]), bf16_to_float(bits["g_final"]), s.rms_eps)
    z = bf16_to_float(bits["lm_head"]) @ h
    c = int(np.argmax(z))
    assert np.sort(z)[-1] - np.sort(z)[-2] > 1e-2   # the fixed draft is not a near-tie
    dr = B.Drafter(s, w.to("cuda"), max_block=16, max_batch=1, kv_capacity=2048)
    t = TinyTarget(s.vocab, s.target_hidden, seed=3, bias_token=c, bias=4.8, device="cuda")
    return dr, t, c


@pytest.mark.parametrize("block", [16, 6])
def test_greedy_generation_is_lossless(setup, block):
    from block_diffusion_drafter_kv_gb300.generate import spec_generate
    from synthetic_target import greedy_reference
    dr, t, c = setup
    ids = torch.randint(0, W_TINY.shape.vocab, (40,), generator=torch.Generator().manual_seed(block))
    ref = greedy_reference(t, ids, 300)
    out, stats = spec_generate(dr, t, ids, 300, block=block)
    torch.cuda.synchronize()
    assert dr.device_error() == 0
    assert out == ref
    assert stats.mean_tau > 1.0, stats.accept_lens
    assert min(stats.accept_lens) < block      # some drafts were rejected
    assert int(dr.len[0]) == 40 + sum(stats.accept_lens)


def test_stop_tokens(setup):
    from block_diffusion_drafter_kv_gb300.generate import spec_generate
    from synthetic_target import greedy_reference
    dr, t, c = setup
    ids = torch.randint(0, W_TINY.shape.vocab, (40,), generator=torch.Generator().manual_seed(9))
    ref = greedy_reference(t, ids, 120)
    stop = next(x for x in ref[5:] if x != c)
    out, _ = spec_generate(dr, t, ids, 120, stop_token_ids=[stop])
    assert out == ref[: ref.index(stop) + 1]


def test_sampling_generation_runs_and_commits_valid_tokens(setup):
    """At temperature 0.7 the loop verifies by speculative sampling; the output is a valid
    token sequence of the requested length (its distribution is pinned on the oracle)."""
    from block_diffusion_drafter_kv_gb300.generate import spec_generate
    dr, t, c = setup
    ids = torch.randint(0, W_TINY.shape.vocab, (40,), generator=torch.Generator().manual_seed(4))
    out, stats = spec_generate(dr, t, ids, 200, temperature=0.7,
                               generator=torch.Generator(device="cuda").manual_seed(0))
    torch.cuda.synchronize()
    assert dr.device_error() == 0
    assert len(out) == 200 and all(0 <= x < W_TINY.shape.vocab for x in out)
    assert 1 <= min(stats.accept_lens) and max(stats.accept_lens) <= 16
