"""Sampling-mode verification (dflash_verify_sampling) against the oracle: the hand-worked
golden cases, and random cases at temperatures below, at and above 1, with the tiny and the
Qwen3-8B-sized vocabulary. Outcomes must be equal; a sequence in which some uniform lies
within 1e-5 of the probability (or cumulative probability) it is compared with is not
compared, since fp32 and fp64 may decide it differently."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle.dflash_ref as R
from golden_io import load_sampling_cases
from synth import TINY
from synth import inputs as I

pytestmark = pytest.mark.gpu
MARGIN = 1e-5


def _drafter(shape, max_batch=4):
    from block_diffusion_drafter_kv_gb300 import binding as B
    from block_diffusion_drafter_kv_gb300.build import build
    build()
    return B.Drafter(shape, I.make_weights(shape, 13).to("cuda"), max_block=16, max_batch=max_batch, kv_capacity=64)


def _run(dr, T, d, u, temp, batch, B):
    acc = torch.full((batch,), -9, dtype=torch.int32, device="cuda")
    com = torch.full((batch, B), -9, dtype=torch.int32, device="cuda")
    dd = torch.as_tensor(np.asarray(d, np.int32).reshape(batch, max(B - 1, 1)), device="cuda")
    dr.verify_sampling(torch.as_tensor(T, device="cuda"), dd if B > 1 else None,
                       torch.as_tensor(np.asarray(u, np.float32), device="cuda"), temp, batch, B, acc, com)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), com.cpu().numpy(), dr.last_token[:batch].cpu().numpy()


@pytest.fixture(scope="module")
def tiny():
    return _drafter(TINY)


@pytest.mark.parametrize("case", load_sampling_cases(), ids=lambda c: c["name"])
def test_hand_worked_cases_on_gpu(tiny, case):
    V = TINY.vocab
    T = np.full((1, case["B"], V), -1.0e4, dtype=np.float32)   # padding logits carry no mass
    T[0, :, : case["V"]] = case["logits"]
    acc, com, last = _run(tiny, T, [case["drafted"]], [case["uniforms"]], case["T"], 1, case["B"])
    assert acc[0] == case["tau"]
    assert list(com[0, : case["tau"]]) == case["committed"] and (com[0, case["tau"]:] == -1).all()
    assert last[0] == case["last"]


def _near_boundary(z, d, temp, u):
    """True when a decision of the oracle's rule lies within MARGIN of its threshold."""
    p = R.softmax(np.asarray(z, np.float64) / temp, axis=-1)
    B = p.shape[0]
    j = 0
    while j < B - 1:
        if abs(u[j] - p[j, d[j]]) < MARGIN:
            return True
        if not u[j] < p[j, d[j]]:
            break
        j += 1
    r = p[j].copy()
    if j < B - 1:
        r[d[j]] = 0.0
    cdf = np.cumsum(r / r.sum())
    return bool(np.min(np.abs(cdf - u[B - 1])) < MARGIN)


def _random_cases(dr, shape, batch, B, temp, seed, trials):
    rng = np.random.default_rng(seed)
    V = shape.vocab
    compared = 0
    for t in range(trials):
        T = (2.0 * rng.standard_normal((batch, B, V))).astype(np.float32)
        d = rng.integers(0, V, size=(batch, max(B - 1, 1))).astype(np.int32)
        for s in range(batch):   # plant likely drafts on a random leading run
            run = int(rng.integers(0, B))
            for i in range(min(run, B - 1)):
                T[s, i, d[s, i]] += 8.0
        u = rng.random((batch, B)).astype(np.float32)
        acc, com, last = _run(dr, T, d, u, temp, batch, B)
        for s in range(batch):
            if _near_boundary(T[s], d[s], temp, u[s].astype(np.float64)):
                continue
            compared += 1
            r = R.verify_sampling(T[s], d[s, : B - 1], temp, u[s].astype(np.float64))
            assert acc[s] == r.accept_len, (t, s)
            assert list(com[s, : r.accept_len]) == list(r.committed) and (com[s, r.accept_len:] == -1).all()
            assert last[s] == r.last_token
    return compared


@pytest.mark.parametrize("batch,B,temp", [(1, 16, 1.0), (3, 4, 0.6), (4, 7, 1.7), (2, 1, 1.0)])
def test_random_cases_match_oracle_tiny(tiny, batch, B, temp):
    assert _random_cases(tiny, TINY, batch, B, temp, seed=batch * 100 + B, trials=6) >= 3


def test_random_cases_match_oracle_qwen3_8b_vocabulary():
    s = replace(TINY, vocab=151936)
    dr = _drafter(s, 2)
    assert _random_cases(dr, s, 2, 16, 0.8, seed=5, trials=3) >= 3
