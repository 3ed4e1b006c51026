"""Pins of the sampling-mode verification oracle: hand-worked golden cases, the
speculative-sampling guarantee that committed tokens follow the target's own distribution
(checked by Monte Carlo), and the low-temperature limit, where it must equal greedy
verification."""
import numpy as np
import pytest

import oracle.dflash_ref as R
from golden_io import load_sampling_cases


@pytest.mark.parametrize("case", load_sampling_cases(), ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    r = R.verify_sampling(case["logits"], np.array(case["drafted"]), case["T"], np.array(case["uniforms"]))
    assert r.accept_len == case["tau"]
    assert list(r.committed) == case["committed"]
    assert r.last_token == case["last"]


def test_committed_tokens_follow_the_target_distribution():
    """With u and w uniform, the first committed token is distributed as p_0, and given that
    the first draft was accepted, the second is distributed as p_1: the output of
    verification has the target's own sampling distribution (40 000 draws, 5 sigma)."""
    rng = np.random.default_rng(0)
    B, V, T = 3, 6, 0.8
    z = rng.standard_normal((B, V)) * 1.5
    d = np.array([2, 4])
    p = R.softmax(z / T, axis=-1)
    n = 40_000
    first = np.zeros(V)
    second = np.zeros(V)
    n_acc = 0
    us = rng.random((n, B))
    for k in range(n):
        r = R.verify_sampling(z, d, T, us[k])
        first[r.committed[0]] += 1
        if r.accept_len >= 2:
            n_acc += 1
            second[r.committed[1]] += 1
    for v in range(V):
        sd = np.sqrt(p[0, v] * (1 - p[0, v]) / n)
        assert abs(first[v] / n - p[0, v]) < 5 * sd + 1e-9, (v, first[v] / n, p[0, v])
    assert abs(n_acc / n - p[0, d[0]]) < 5 * np.sqrt(p[0, d[0]] * (1 - p[0, d[0]]) / n)
    for v in range(V):
        sd = np.sqrt(p[1, v] * (1 - p[1, v]) / n_acc)
        assert abs(second[v] / n_acc - p[1, v]) < 5 * sd + 1e-9, (v, second[v] / n_acc, p[1, v])


def test_low_temperature_equals_greedy():
    rng = np.random.default_rng(1)
    for trial in range(20):
        B, V = 5, 50
        z = rng.standard_normal((B, V))
        g = np.argmax(z, axis=-1)
        d = rng.integers(0, V, size=B - 1)
        run = int(rng.integers(0, B))
        d[:run] = g[:run]
        r = R.verify_sampling(z, d, 1e-4, rng.random(B))
        gr = R.verify_greedy(z, d)
        assert r.accept_len == gr.accept_len and list(r.committed) == list(gr.committed)
