"""Pins of the oracle's injection and draft forward on the tiny drafter:
associativity of injection, row independence, and brute-force agreement with the
naive per-slot recomputation over consecutive steps."""
import numpy as np
import pytest

from oracle.dflash_ref import Oracle
from oracle.naive import naive_draft, naive_context_kv
from synth import W_TINY
from synth import inputs as I

SEED = 1234


@pytest.fixture(scope="module")
def tiny():
    s = W_TINY.shape
    w = I.make_weights(s, SEED)
    bits = w.bits()
    hid = I.bf16_bits(I.make_hidden(s, 160, SEED))
    return s, bits, hid


def test_injection_is_associative(tiny):
    """Two incremental injections equal one injection over the same positions
    (the injected projections persist across drafting iterations). The BLAS library
    may pick a different kernel for a different row count, so equality holds up to
    fp64 rounding order."""
    s, bits, hid = tiny
    o = Oracle(s, bits)
    a = o.new_sequence(128)
    o.inject(a, hid[:, :64])
    o.inject(a, hid[:, 64:71])
    b = o.new_sequence(128)
    o.inject(b, hid[:, :71])
    assert a.length == b.length == 71
    for l in range(s.n_layers):
        assert np.allclose(a.k_cache[l][:71], b.k_cache[l][:71], rtol=1e-12, atol=1e-13)
        assert np.allclose(a.v_cache[l][:71], b.v_cache[l][:71], rtol=1e-12, atol=1e-13)
        # and the positions after 71 were never touched
        assert not a.k_cache[l][71:].any() and not b.k_cache[l][71:].any()


def test_injection_row_independent(tiny):
    s, bits, hid = tiny
    o = Oracle(s, bits)
    batch = o.context_feature(hid[:, 10:20])
    for r in (0, 3, 9):
        assert np.allclose(o.context_feature(hid[:, 10 + r:11 + r])[0], batch[r], rtol=0, atol=1e-13)


def test_injection_matches_naive(tiny):
    s, bits, hid = tiny
    o = Oracle(s, bits)
    st = o.new_sequence(64)
    o.inject(st, hid[:, :40])
    K, V = naive_context_kv(s, bits, hid[:, :40])
    for l in range(s.n_layers):
        assert np.allclose(st.k_cache[l][:40], K[l], atol=1e-10)
        assert np.allclose(st.v_cache[l][:40], V[l], atol=1e-10)


def test_draft_steps_match_naive_recomputation(tiny):
    """Three draft+verify steps: the block oracle (persistent cache, vectorised) equals the
    naive per-slot recomputation from the full hidden-state history at every step."""
    s, bits, hid = tiny
    w = W_TINY
    o = Oracle(s, bits)
    last = int(I.initial_tokens(1, s.vocab, SEED)[0])
    st = o.new_sequence(w.kv_capacity(), last)
    o.inject(st, hid[:, : w.ctx])
    for step in range(w.steps):
        r = o.draft(st, w.block)
        nd, nl, ntr = naive_draft(s, bits, hid[:, : st.length], st.last_token, w.block)
        assert np.array_equal(r.drafted, nd)
        assert np.allclose(r.logits, nl, rtol=1e-9, atol=1e-10)
        assert np.allclose(r.x_trace, ntr, rtol=1e-9, atol=1e-10)
        noise = I.make_logit_noise(1, w.block, s.vocab, SEED, f"logits.{step}").numpy()
        mask = I.make_plant_mask(1, w.block, w.p_plant, SEED, f"plant.{step}")
        T = I.plant_logits(noise, r.drafted[None], mask)[0]
        v = o.verify(st, T, r.drafted)
        # lossless: what is committed is exactly the target's greedy continuation
        assert np.array_equal(v.committed, np.argmax(T, axis=1)[: v.accept_len])
        # planted slots agree: tau is at least the leading run of planted rows plus one
        run = next((i for i in range(w.block - 1) if not mask[0, i]), w.block - 1)
        assert v.accept_len >= run + 1
        o.inject(st, hid[:, st.length: st.length + v.accept_len])


def test_block_of_one_with_no_context_returns_value_path(tiny):
    """N = 0 and B = 1: attention over the single block key returns its value, so each
    layer's attention output is v itself."""
    s, bits, hid = tiny
    o = Oracle(s, bits)
    st = o.new_sequence(4, last_token=5)
    r = o.draft(st, 1)
    assert r.drafted.shape == (0,) and r.x_trace.shape == (s.n_layers + 1, 1, s.hidden)
    nd, nl, ntr = naive_draft(s, bits, hid[:, :0], 5, 1)
    assert np.allclose(r.x_trace, ntr, atol=1e-10)


def test_fp32_mode_close_to_fp64(tiny):
    s, bits, hid = tiny
    r = {}
    for dt in (np.float64, np.float32):
        o = Oracle(s, bits, dtype=dt)
        st = o.new_sequence(80, 3)
        o.inject(st, hid[:, :64])
        r[dt] = o.draft(st, 4)
    a, b = r[np.float64], r[np.float32]
    assert np.max(np.abs(a.logits - b.logits)) < 1e-4 * np.std(a.logits) * 100


def _uncached(s, bits):
    """The oracle as the full-size workloads run it: weights widened per use (no cache, the
    branch taken once the widened weights exceed the cache limit) and the LM head in row
    chunks, here of an odd size (7) that divides no dimension of the tiny drafter."""
    o = Oracle(s, bits, cache_limit_bytes=0, lm_chunk=7)
    assert o._cache is None
    return o


def test_uncached_chunked_oracle_matches_naive(tiny):
    """The uncached, chunked branch against the naive per-slot recomputation, over three
    draft+verify steps with incremental injection (as the cached branch is pinned above)."""
    s, bits, hid = tiny
    w = W_TINY
    o = _uncached(s, bits)
    last = int(I.initial_tokens(1, s.vocab, SEED + 1)[0])
    st = o.new_sequence(w.kv_capacity(), last)
    o.inject(st, hid[:, : w.ctx])
    K, V = naive_context_kv(s, bits, hid[:, : w.ctx])
    for l in range(s.n_layers):
        assert np.allclose(st.k_cache[l][: w.ctx], K[l], atol=1e-10)
        assert np.allclose(st.v_cache[l][: w.ctx], V[l], atol=1e-10)
    for step in range(w.steps):
        r = o.draft(st, w.block)
        nd, nl, ntr = naive_draft(s, bits, hid[:, : st.length], st.last_token, w.block)
        assert np.array_equal(r.drafted, nd)
        assert np.allclose(r.logits, nl, rtol=1e-9, atol=1e-10)
        assert np.allclose(r.x_trace, ntr, rtol=1e-9, atol=1e-10)
        noise = I.make_logit_noise(1, w.block, s.vocab, SEED + 1, f"logits.{step}").numpy()
        mask = I.make_plant_mask(1, w.block, w.p_plant, SEED + 1, f"plant.{step}")
        v = o.verify(st, I.plant_logits(noise, r.drafted[None], mask)[0], r.drafted)
        o.inject(st, hid[:, st.length: st.length + v.accept_len])


def test_uncached_chunked_oracle_equals_cached(tiny):
    """Both branches compute the same step: inject, draft and verify agree to fp64 rounding
    over three steps (the chunked LM head computes each logit as one whole dot product)."""
    s, bits, hid = tiny
    w = W_TINY
    a, b = Oracle(s, bits), _uncached(s, bits)
    assert a._cache is not None
    last = int(I.initial_tokens(1, s.vocab, SEED + 2)[0])
    sa, sb = a.new_sequence(w.kv_capacity(), last), b.new_sequence(w.kv_capacity(), last)
    a.inject(sa, hid[:, : w.ctx])
    b.inject(sb, hid[:, : w.ctx])
    for step in range(w.steps):
        ra, rb = a.draft(sa, w.block), b.draft(sb, w.block)
        assert np.array_equal(ra.drafted, rb.drafted)
        assert np.allclose(ra.logits, rb.logits, rtol=1e-12, atol=1e-13)
        assert np.allclose(ra.x_trace, rb.x_trace, rtol=1e-12, atol=1e-13)
        noise = I.make_logit_noise(1, w.block, s.vocab, SEED + 2, f"logits.{step}").numpy()
        mask = I.make_plant_mask(1, w.block, w.p_plant, SEED + 2, f"plant.{step}")
        T = I.plant_logits(noise, ra.drafted[None], mask)[0]
        va, vb = a.verify(sa, T, ra.drafted), b.verify(sb, T, rb.drafted)
        assert va.accept_len == vb.accept_len and np.array_equal(va.committed, vb.committed)
        a.inject(sa, hid[:, sa.length: sa.length + va.accept_len])
        b.inject(sb, hid[:, sb.length: sb.length + vb.accept_len])
        for l in range(s.n_layers):
            assert np.allclose(sa.k_cache[l][: sa.length], sb.k_cache[l][: sb.length], rtol=1e-12, atol=1e-13)
            assert np.allclose(sa.v_cache[l][: sa.length], sb.v_cache[l][: sb.length], rtol=1e-12, atol=1e-13)
