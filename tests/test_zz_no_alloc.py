"""The allocation-free greedy verification entry point (dflash_verify_greedy_noalloc).

It is for callers that cannot allocate device memory at all, for example code running
inside another engine's decode loop on a memory pool that forbids new allocations, and
so cannot hand the library a workspace. Its result must equal that of the regular entry
point (dflash_verify_greedy, which uses the workspace bound to a handle), exactly,
call after call even though every call reuses the same fixed scratch array.

This file sorts last so that a run stopping at its first failure has run everything else.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def drafter():
    from block_diffusion_drafter_kv_gb300 import binding as B
    from block_diffusion_drafter_kv_gb300.build import build
    from synth import TINY
    from synth import inputs as I
    build()
    w = I.make_weights(TINY, 3).to("cuda")
    return B.Drafter(TINY, w, max_block=16, max_batch=8, kv_capacity=64)


def _inputs(rng, batch, block, vocab):
    T = rng.standard_normal((batch, block, vocab)).astype(np.float32)
    d = rng.integers(0, vocab, size=(batch, block - 1)).astype(np.int32)
    g = np.argmax(T, axis=-1)
    for s in range(batch):           # make each sequence agree on a random leading run
        run = int(rng.integers(0, block))
        d[s, :run] = g[s, :run]
    T[0, 0, 3] = T[0, 0, 11] = T[0, 0].max() + 1.0   # an exact tie: the lower index wins
    return torch.as_tensor(T, device="cuda"), torch.as_tensor(d, device="cuda")


@pytest.mark.parametrize("batch,block", [(5, 16), (1, 4), (8, 7)])
def test_noalloc_matches_regular_entry_on_consecutive_calls(drafter, batch, block):
    from block_diffusion_drafter_kv_gb300 import binding as B
    rng = np.random.default_rng(batch * 31 + block)
    vocab = drafter.shape.vocab
    for _ in range(2):               # two calls in a row on the shared scratch array
        T, d = _inputs(rng, batch, block, vocab)
        acc_a = torch.full((batch,), -9, dtype=torch.int32, device="cuda")
        com_a = torch.full((batch, block), -9, dtype=torch.int32, device="cuda")
        last_a = torch.full((batch,), -9, dtype=torch.int32, device="cuda")
        B.verify_greedy_noalloc(T, d, batch, block, acc_a, com_a, last_a)
        acc_b = torch.full((batch,), -9, dtype=torch.int32, device="cuda")
        com_b = torch.full((batch, block), -9, dtype=torch.int32, device="cuda")
        drafter.verify(T, d, batch, block, acc_b, com_b)
        torch.cuda.synchronize()
        assert torch.equal(acc_a, acc_b)
        assert torch.equal(com_a, com_b)
        assert torch.equal(last_a, drafter.last_token[:batch])
        assert int(acc_a.min()) >= 1


@pytest.fixture(scope="module")
def wide_vocab():
    """A drafter handle whose vocabulary is the Qwen3-8B-sized one (151 936 logits per row),
    so the regular entry point and the allocation-free one both split a row into many
    chunks; max_batch 64 covers the fixed array's largest batch."""
    from dataclasses import replace
    from block_diffusion_drafter_kv_gb300 import binding as B
    from block_diffusion_drafter_kv_gb300.build import build
    from synth import TINY
    from synth import inputs as I
    build()
    s = replace(TINY, vocab=151936)
    return B.Drafter(s, I.make_weights(s, 5).to("cuda"), max_block=16, max_batch=64, kv_capacity=64)


@pytest.mark.parametrize("batch,block", [(32, 16), (64, 16), (3, 5)])
def test_noalloc_multi_chunk_rows_match_oracle_and_regular_entry(wide_vocab, batch, block):
    """At V = 151 936 each row is reduced in several chunks (up to 32) through the fixed
    array's layout; batch 64 with B = 16 fills the array to its stated limit. Two calls in
    a row must both equal the oracle's greedy verification and the regular entry point."""
    from block_diffusion_drafter_kv_gb300 import binding as B
    from oracle.dflash_ref import verify_greedy
    vocab = wide_vocab.shape.vocab
    rng = np.random.default_rng(batch * 7 + block)
    for call in range(2):
        T, d = _inputs(rng, batch, block, vocab)
        T[batch - 1, block - 1, vocab - 1] = T[batch - 1, block - 1].max() + 2.0   # the last logit wins a row
        acc = torch.full((batch,), -9, dtype=torch.int32, device="cuda")
        com = torch.full((batch, block), -9, dtype=torch.int32, device="cuda")
        last = torch.full((batch,), -9, dtype=torch.int32, device="cuda")
        B.verify_greedy_noalloc(T, d, batch, block, acc, com, last)
        acc_b = torch.full((batch,), -9, dtype=torch.int32, device="cuda")
        com_b = torch.full((batch, block), -9, dtype=torch.int32, device="cuda")
        wide_vocab.verify(T, d, batch, block, acc_b, com_b)
        torch.cuda.synchronize()
        assert torch.equal(acc, acc_b) and torch.equal(com, com_b)
        assert torch.equal(last, wide_vocab.last_token[:batch])
        Tn, dn = T.cpu().numpy(), d.cpu().numpy()
        a, c, l = acc.cpu().numpy(), com.cpu().numpy(), last.cpu().numpy()
        for q in range(batch):
            r = verify_greedy(Tn[q], dn[q])
            assert a[q] == r.accept_len, (call, q)
            assert list(c[q, : r.accept_len]) == list(r.committed) and (c[q, r.accept_len:] == -1).all()
            assert l[q] == r.last_token


def test_noalloc_rejects_sizes_beyond_its_array():
    from block_diffusion_drafter_kv_gb300 import binding as B
    L = B.lib()
    T = torch.zeros(1, 16, 64, device="cuda")
    i32 = torch.zeros(1024, dtype=torch.int32, device="cuda")
    p = i32.data_ptr()
    assert L.dflash_verify_greedy_noalloc(T.data_ptr(), p, 65, 16, 64, p, p, p, None) == -3
    assert L.dflash_verify_greedy_noalloc(T.data_ptr(), p, 1, 17, 64, p, p, p, None) == -3
