"""Pins of the fused target-side verification oracle (the target's final norm, LM head and
argmax from its last hidden states, then the longest-prefix rule): brute force against the
naive scalar loops, planted agreement, a mismatch at slot 0, and the scale invariance that
the final RMSNorm gives."""
import numpy as np
import pytest

import oracle.dflash_ref as R
from oracle.naive import naive_verify_from_hidden
from synth import inputs as I

EPS = 1e-6


def _bits(x):
    import torch
    return I.bf16_bits(torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16))


def _target(seed, B=4, Ht=64, V=96):
    rng = np.random.default_rng(seed)
    h = _bits(rng.standard_normal((B, Ht)))
    g = _bits(1.0 + 0.1 * rng.standard_normal(Ht))
    W = _bits(0.05 * rng.standard_normal((V, Ht)))
    return h, g, W


@pytest.mark.parametrize("seed,B", [(0, 4), (1, 1), (2, 7), (3, 16)])
def test_matches_naive_scalar_loops(seed, B):
    h, g, W = _target(seed, B=B)
    rng = np.random.default_rng(100 + seed)
    z = R.target_logits_from_hidden(h, g, W, EPS)
    gt = np.argmax(z, axis=-1)
    for trial in range(4):
        d = rng.integers(0, W.shape[0], size=B - 1)
        run = int(rng.integers(0, B))
        d[:run] = gt[:run]                      # agree on a random leading run
        r, _ = R.verify_greedy_from_hidden(h, g, W, d, EPS)
        tau, com, g_naive = naive_verify_from_hidden(h, g, W, d, EPS)
        assert list(r.target_argmax) == g_naive
        assert r.accept_len == tau and list(r.committed) == list(com)


def test_planted_agreement_and_slot0_mismatch():
    """A head whose row t_i points along the normed hidden state of position i makes t_i
    that position's argmax: drafting t_1..t_{B-1} accepts all B; changing the first draft
    accepts only the bonus token."""
    B, Ht, V = 5, 64, 96
    h, g, W = _target(7, B=B, Ht=Ht, V=V)
    a = R.rms_norm(R.bf16_to_float(h), R.bf16_to_float(g), EPS)
    Wf = R.bf16_to_float(W)
    t = [11, 23, 37, 52, 90]
    for i in range(B):
        Wf[t[i]] = 4.0 * a[i] / np.linalg.norm(a[i])
    W2 = _bits(Wf)
    r, z = R.verify_greedy_from_hidden(h, g, W2, np.array(t[:B - 1]), EPS)
    assert list(r.target_argmax) == t
    assert r.accept_len == B and list(r.committed) == t and r.last_token == t[-1]
    d = np.array(t[:B - 1]); d[0] = (d[0] + 1) % V
    r, _ = R.verify_greedy_from_hidden(h, g, W2, d, EPS)
    assert r.accept_len == 1 and list(r.committed) == [t[0]] and r.last_token == t[0]


def test_final_norm_makes_logits_scale_invariant():
    """Scaling every hidden state by 4 (exact in bf16) leaves RMSNorm(h), hence the logits,
    unchanged up to the epsilon."""
    h, g, W = _target(9, B=6)
    z1 = R.target_logits_from_hidden(h, g, W, EPS)
    h4 = _bits(4.0 * R.bf16_to_float(h))
    z4 = R.target_logits_from_hidden(h4, g, W, EPS)
    assert np.allclose(z1, z4, rtol=1e-5, atol=1e-7)
