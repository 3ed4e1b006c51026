"""Pins of the oracle's building blocks against closed forms and library routines
(the routines are called here, in the tests, never inside the oracle)."""
import math

import numpy as np
import pytest
import torch

from oracle import dflash_ref as R
from oracle.naive import _rope_complex


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_closed_form():
    # x = [3, 4]: mean square 12.5, so x / sqrt(12.5) = [3, 4] * sqrt(2) / 5
    out = R.rms_norm(np.array([[3.0, 4.0]]), np.array([1.0, 1.0]), 0.0)
    assert np.allclose(out, [[3 * math.sqrt(2) / 5, 4 * math.sqrt(2) / 5]], rtol=0, atol=1e-15)
    # a constant vector normalises to the gain (times its sign)
    g = np.array([0.5, 2.0, -1.0, 3.0])
    out = R.rms_norm(np.full((1, 4), -7.0), g, 0.0)
    assert np.allclose(out, -g[None], atol=1e-15)


def test_rmsnorm_eps_and_scale():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 64))
    g = 1 + 0.1 * rng.standard_normal(64)
    # scale invariance without eps
    assert np.allclose(R.rms_norm(5.0 * x, g, 0.0), R.rms_norm(x, g, 0.0), atol=1e-13)
    # eps enters under the square root of the mean square
    eps = 0.25
    ms = (x * x).mean(axis=1, keepdims=True)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(g), eps).numpy()
    assert np.allclose(R.rms_norm(x, g, eps), ref, atol=1e-12)
    assert np.allclose(R.rms_norm(x, g, eps), x * g / np.sqrt(ms + eps), atol=1e-13)


# ---------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(2).standard_normal((1, 3, 64))
    assert np.array_equal(R.apply_rope(x, np.array([0]), 1e6), x)


def test_rope_first_pair_closed_form():
    # d = 2: the single pair rotates by the position itself (inv_freq_0 = 1)
    for p in (1, 2, 5, 1000):
        out = R.apply_rope(np.array([[[1.0, 0.0]]]), np.array([p]), 1e6)
        assert np.allclose(out[0, 0], [math.cos(p), math.sin(p)], atol=1e-12)
        out = R.apply_rope(np.array([[[0.0, 1.0]]]), np.array([p]), 1e6)
        assert np.allclose(out[0, 0], [-math.sin(p), math.cos(p)], atol=1e-12)


@pytest.mark.parametrize("d,theta", [(64, 1e6), (128, 5e5), (8, 10000.0)])
def test_rope_matches_complex_rotation(d, theta):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((5, 2, d))
    pos = np.array([0, 1, 17, 2048, 32767])
    out = R.apply_rope(x, pos, theta)
    for n in range(5):
        for h in range(2):
            assert np.allclose(out[n, h], _rope_complex(x[n, h], int(pos[n]), theta), atol=1e-9)


def test_rope_relative_and_norm():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((1, 1, 128)), rng.standard_normal((1, 1, 128))
    a = np.sum(R.apply_rope(q, [100], 1e6) * R.apply_rope(k, [37], 1e6))
    b = np.sum(R.apply_rope(q, [1100], 1e6) * R.apply_rope(k, [1037], 1e6))
    assert abs(a - b) < 1e-9
    r = R.apply_rope(q, [12345], 1e6)
    pairs = lambda v: v[..., :64] ** 2 + v[..., 64:] ** 2
    assert np.allclose(pairs(r), pairs(q), atol=1e-12)


# ---------------------------------------------------------------- attention

def test_attention_mha_matches_sdpa():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((5, 3, 16))
    k = rng.standard_normal((9, 3, 16))
    v = rng.standard_normal((9, 3, 16))
    out = R.gqa_attention(q, k, v)
    t = lambda a: torch.from_numpy(a).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v))[0].permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, atol=1e-12)


def test_attention_gqa_head_mapping_matches_sdpa():
    """Query head h reads kv head h // (nq/nkv): contiguous groups of query heads."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 8, 16))
    k = rng.standard_normal((7, 2, 16))
    v = rng.standard_normal((7, 2, 16))
    out = R.gqa_attention(q, k, v)
    t = lambda a: torch.from_numpy(a).permute(1, 0, 2)[None]
    kk = t(k).repeat_interleave(4, dim=1)
    vv = t(v).repeat_interleave(4, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), kk, vv)[0].permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((3, 2, 8))
    v = rng.standard_normal((1, 1, 8))
    # a single key: every query returns its value
    assert np.allclose(R.gqa_attention(q, rng.standard_normal((1, 1, 8)), v), np.broadcast_to(v, (3, 2, 8)))
    # identical keys: uniform weights, the mean of the values
    k = np.repeat(rng.standard_normal((1, 1, 8)), 6, axis=0)
    vs = rng.standard_normal((6, 1, 8))
    assert np.allclose(R.gqa_attention(q, k, vs), np.broadcast_to(vs.mean(axis=0), (3, 2, 8)))


def test_attention_is_bidirectional():
    """Changing the last key changes the first query's output (no causal mask)."""
    rng = np.random.default_rng(8)
    q, k, v = (rng.standard_normal((4, 1, 8)) for _ in range(3))
    a = R.gqa_attention(q, k, v)
    k2 = k.copy()
    k2[-1] += 3.0
    b = R.gqa_attention(q, k2, v)
    assert not np.allclose(a[0], b[0])


# ---------------------------------------------------------------- SwiGLU pieces

def test_silu_closed_forms():
    x = np.linspace(-20, 20, 401)
    s = R.silu(x)
    assert R.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(s - R.silu(-x), x, atol=1e-12)          # silu(x) - silu(-x) = x
    assert np.allclose(s, torch.nn.functional.silu(torch.from_numpy(x)).numpy(), atol=1e-14)


def test_bf16_widening_exact():
    t = torch.tensor([1.0, -2.5, 3.140625, 1e-3, 65504.0]).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(R.bf16_to_float(bits), t.double().numpy())
