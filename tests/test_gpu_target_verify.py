"""Fused target-side verification (dflash_verify_greedy_hidden) against the oracle: the
target's final RMSNorm, LM head and argmax of every block position computed from its last
hidden states, then the longest-prefix acceptance. Acceptance and committed tokens must be
bit-exact; a sequence in which some position's two largest oracle logits lie within 1e-2
(where fp32 and fp64 may legitimately pick different tokens) is not compared."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle.dflash_ref as R
from synth import TINY
from synth import inputs as I

pytestmark = pytest.mark.gpu
GAP_EXEMPT = 1e-2


def _drafter(shape, max_batch):
    from block_diffusion_drafter_kv_gb300 import binding as B
    from block_diffusion_drafter_kv_gb300.build import build
    build()
    return B.Drafter(shape, I.make_weights(shape, 11).to("cuda"), max_block=16, max_batch=max_batch, kv_capacity=64)


def _target(shape, seed, std=0.02, device="cuda"):
    g = torch.Generator(device=device).manual_seed(seed)
    Ht, V = shape.target_hidden, shape.vocab
    gain = (1.0 + 0.1 * torch.randn(Ht, generator=g, device=device)).to(torch.bfloat16)
    lm = (std * torch.randn(V, Ht, generator=g, device=device)).to(torch.bfloat16)
    return gain, lm


def _bits(t):
    return I.bf16_bits(t.cpu())


def _run(dr, hid, gain, lm, drafted, batch, B):
    acc = torch.full((batch,), -9, dtype=torch.int32, device="cuda")
    com = torch.full((batch, B), -9, dtype=torch.int32, device="cuda")
    dr.verify_hidden(hid, gain, lm, drafted if B > 1 else None, batch, B, acc, com)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), com.cpu().numpy(), dr.last_token[:batch].cpu().numpy()


def _check(shape, dr, gain, lm, batch, B, seed, trials):
    rng = np.random.default_rng(seed)
    gb, lb = _bits(gain), _bits(lm)
    compared = 0
    for t in range(trials):
        g = torch.Generator(device="cuda").manual_seed(seed * 100 + t)
        hid = torch.randn(batch * B, shape.target_hidden, generator=g, device="cuda").to(torch.bfloat16)
        hb = _bits(hid).reshape(batch, B, shape.target_hidden)
        zs = [R.target_logits_from_hidden(hb[s], gb, lb, shape.rms_eps) for s in range(batch)]
        d = np.zeros((batch, max(B - 1, 1)), dtype=np.int32)
        for s in range(batch):
            gt = np.argmax(zs[s], axis=-1)
            d[s, : B - 1] = rng.integers(0, shape.vocab, size=B - 1)
            run = int(rng.integers(0, B))
            d[s, :run] = gt[:run]
        acc, com, last = _run(dr, hid, gain, lm, torch.as_tensor(d, device="cuda"), batch, B)
        for s in range(batch):
            p = np.partition(zs[s], -2, axis=-1)
            if float((p[:, -1] - p[:, -2]).min()) < GAP_EXEMPT:
                continue
            compared += 1
            r, _ = R.verify_greedy_from_hidden(hb[s], gb, lb, d[s, : B - 1], shape.rms_eps)
            assert acc[s] == r.accept_len, (t, s)
            assert list(com[s, : r.accept_len]) == list(r.committed) and (com[s, r.accept_len:] == -1).all()
            assert last[s] == r.last_token
    return compared


@pytest.mark.parametrize("batch,B", [(1, 4), (3, 16), (4, 1), (2, 7)])
def test_fused_verify_matches_oracle_tiny(batch, B):
    dr = _drafter(TINY, 4)
    gain, lm = _target(TINY, 5, std=0.2)   # logits spread so that near-ties are rare
    assert _check(TINY, dr, gain, lm, batch, B, seed=batch * 10 + B, trials=8) >= 3


def test_fused_verify_planted_agreement():
    """An LM head whose row t_i points along position i's normed hidden state: drafting
    t_1.. accepts the whole block; a wrong first draft accepts only the bonus token."""
    s = TINY
    dr = _drafter(s, 4)
    gain, lm = _target(s, 6)
    B = 5
    hid = torch.randn(B, s.target_hidden, generator=torch.Generator(device="cuda").manual_seed(3),
                      device="cuda").to(torch.bfloat16)
    a = R.rms_norm(R.bf16_to_float(_bits(hid)), R.bf16_to_float(_bits(gain)), s.rms_eps)
    lmf = lm.float().cpu().numpy()
    t = [17, 201, 333, 512, 1000]
    for i in range(B):
        lmf[t[i]] = 4.0 * a[i] / np.linalg.norm(a[i])
    lm2 = torch.as_tensor(lmf).to(torch.bfloat16).cuda()
    acc, com, last = _run(dr, hid, gain, lm2, torch.as_tensor([t[:B - 1]], dtype=torch.int32, device="cuda"), 1, B)
    assert acc[0] == B and list(com[0]) == t and last[0] == t[-1]
    wrong = [t[0] + 1] + t[1:B - 1]
    acc, com, last = _run(dr, hid, gain, lm2, torch.as_tensor([wrong], dtype=torch.int32, device="cuda"), 1, B)
    assert acc[0] == 1 and com[0, 0] == t[0] and (com[0, 1:] == -1).all() and last[0] == t[0]


def test_fused_verify_matches_oracle_qwen3_8b_target_size():
    """A Qwen3-8B-sized target head (Ht 4096, V 151 936, 1.24 GB bf16), two sequences of
    B = 16: every row's argmax over the full vocabulary in many weight-streaming tiles."""
    s = replace(TINY, vocab=151936, target_hidden=4096)
    dr = _drafter(s, 2)
    gain, lm = _target(s, 7)
    assert _check(s, dr, gain, lm, 2, 16, seed=77, trials=3) >= 1


def test_fused_verify_rejects_bad_arguments():
    from block_diffusion_drafter_kv_gb300 import binding as BND
    dr = _drafter(TINY, 4)
    gain, lm = _target(TINY, 5)
    hid = torch.zeros(4 * 16 + 8, TINY.target_hidden, dtype=torch.bfloat16, device="cuda")
    d = torch.zeros(4, 15, dtype=torch.int32, device="cuda")
    acc = torch.zeros(5, dtype=torch.int32, device="cuda")
    com = torch.zeros(5, 16, dtype=torch.int32, device="cuda")
    with pytest.raises(BND.DFlashError) as ei:   # misaligned hidden states
        dr.verify_hidden(hid.view(-1)[1:].view(-1)[: 4 * TINY.target_hidden].view(4, -1), gain, lm, d, 1, 4, acc, com)
    assert ei.value.status == BND.DFLASH_E_INVAL
    with pytest.raises(BND.DFlashError) as ei:   # batch beyond the handle's maximum
        dr.verify_hidden(hid, gain, lm, d, 5, 4, acc, com)
    assert ei.value.status == -3
