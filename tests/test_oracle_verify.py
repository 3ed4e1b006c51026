"""Pins of the oracle's greedy verification (exact: integer results)."""
import itertools

import numpy as np
import pytest

from oracle.dflash_ref import verify_greedy
from oracle.naive import naive_verify
from golden_io import load_verify_cases


@pytest.mark.parametrize("case", load_verify_cases(), ids=lambda c: c["name"])
def test_hand_worked_cases(case):
    r = verify_greedy(case["logits"], np.array(case["drafted"], dtype=np.int64))
    assert r.accept_len == case["tau"]
    assert list(r.committed) == case["committed"]
    assert r.last_token == case["last"]
    tau, comm = naive_verify(case["logits"], case["drafted"])
    assert (tau, list(comm)) == (case["tau"], case["committed"])


def _logits_with_argmax(g, V, rng):
    T = rng.standard_normal((len(g), V)).astype(np.float32)
    for i, t in enumerate(g):
        T[i, t] = T[i].max() + 1.0 + rng.random()
    return T


@pytest.mark.parametrize("B", [2, 3, 4, 5])
def test_all_agreement_masks(B):
    """Every pattern of agreeing/disagreeing slots: tau-1 is the index of the first
    disagreement (or B-1), committed tokens are the target's argmax rows."""
    rng = np.random.default_rng(B)
    V = 11
    for mask in itertools.product([0, 1], repeat=B - 1):
        g = rng.integers(0, V, size=B)
        T = _logits_with_argmax(g, V, rng)
        d = np.array([g[i] if mask[i] else (g[i] + 1 + rng.integers(0, V - 1)) % V
                      for i in range(B - 1)])
        first_bad = next((i for i in range(B - 1) if not mask[i]), B - 1)
        r = verify_greedy(T, d)
        assert r.accept_len == first_bad + 1
        assert list(r.committed) == list(g[: first_bad + 1])
        assert r.last_token == g[first_bad]
        assert (r.accept_len, list(r.committed)) == tuple((lambda t: (t[0], list(t[1])))(naive_verify(T, d)))


def test_full_agreement_gives_B_and_slot0_mismatch_gives_one():
    rng = np.random.default_rng(0)
    for B in (1, 4, 16):
        g = rng.integers(0, 50, size=B)
        T = _logits_with_argmax(g, 50, rng)
        assert verify_greedy(T, g[:-1]).accept_len == B
        if B > 1:
            d = g[:-1].copy()
            d[0] = (d[0] + 1) % 50
            r = verify_greedy(T, d)
            assert r.accept_len == 1 and list(r.committed) == [g[0]]


def test_lossless_committed_equal_target_greedy():
    """Whatever the drafts, every committed token is the target's own greedy token."""
    rng = np.random.default_rng(7)
    for _ in range(200):
        B = int(rng.integers(1, 17))
        T = rng.standard_normal((B, 37)).astype(np.float32)
        d = rng.integers(0, 37, size=B - 1)
        r = verify_greedy(T, d)
        assert 1 <= r.accept_len <= B
        assert np.array_equal(r.committed, np.argmax(T, axis=1)[: r.accept_len])
