"""Parity of the CUDA path with the oracle through the C ABI: greedy verification
(bit-exact), KV injection (tolerance and bit-exact persistence) and the full
inject -> draft -> verify step loop on the tiny drafter."""
import numpy as np
import pytest
import torch

from oracle.dflash_ref import verify_greedy
from synth import W_TINY
from synth import inputs as I

pytestmark = pytest.mark.gpu

SEED = 2024


@pytest.fixture(scope="module")
def tiny():
    from gpu_util import Setup
    return Setup(W_TINY, seed=SEED, max_batch=4, kv_capacity=256)


# ------------------------------------------------------------------ verification

def _verify_gpu(setup, T, d, batch, B):
    dev = "cuda"
    acc = torch.full((batch,), -7, dtype=torch.int32, device=dev)
    com = torch.full((batch, B), -7, dtype=torch.int32, device=dev)
    dd = torch.as_tensor(np.asarray(d, dtype=np.int32).reshape(batch, max(B - 1, 0)), device=dev)
    setup.drafter.verify(torch.as_tensor(T, device=dev), dd if B > 1 else None, batch, B, acc, com)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), com.cpu().numpy(), setup.drafter.last_token[:batch].cpu().numpy()


@pytest.mark.parametrize("batch,B", [(1, 4), (1, 16), (3, 16), (4, 1), (2, 7)])
def test_verify_bit_exact(tiny, batch, B):
    V = tiny.s.vocab
    rng = np.random.default_rng(batch * 100 + B)
    for trial in range(6):
        T = rng.standard_normal((batch, B, V)).astype(np.float32)
        d = rng.integers(0, V, size=(batch, max(B - 1, 0)))
        for s in range(batch):      # plant agreement on a random prefix of each sequence
            k = int(rng.integers(0, B))
            for i in range(min(k, B - 1)):
                T[s, i, d[s, i]] = 10.0
        if trial == 0:               # exact ties inside a row: lowest index must win
            T[0, 0, 5] = T[0, 0, 9] = 50.0
        acc, com, last = _verify_gpu(tiny, T, d, batch, B)
        for s in range(batch):
            r = verify_greedy(T[s], d[s])
            assert acc[s] == r.accept_len
            assert list(com[s, : r.accept_len]) == list(r.committed)
            assert (com[s, r.accept_len:] == -1).all()
            assert last[s] == r.last_token


def test_verify_full_agreement_and_slot0_mismatch(tiny):
    V, B = tiny.s.vocab, 4
    rng = np.random.default_rng(1)
    T = rng.standard_normal((2, B, V)).astype(np.float32)
    g = np.argmax(T, axis=-1)
    d = np.stack([g[0, :-1], g[1, :-1]])
    d[1, 0] = (d[1, 0] + 1) % V
    acc, com, last = _verify_gpu(tiny, T, d, 2, B)
    assert acc[0] == B and list(com[0]) == list(g[0]) and last[0] == g[0, -1]
    assert acc[1] == 1 and com[1, 0] == g[1, 0] and last[1] == g[1, 0]


# ------------------------------------------------------------------ injection

def test_inject_matches_oracle_and_persists_bit_exact(tiny):
    s = tiny.s
    hid = I.make_hidden(s, 96, SEED, "inject")
    bits = I.bf16_bits(hid)
    d = tiny.drafter
    # sequence 0: 37 rows at once; sequence 1: 20 rows then 17 rows (two injections)
    d.len.zero_()
    h0 = torch.zeros(s.n_taps, 2 * 37, s.target_hidden, dtype=torch.bfloat16)
    h0[:, :37] = hid[:, :37]
    h0[:, 37:57] = hid[:, :20]
    tiny.gpu_inject(h0, [37, 20], rows_per_seq=37, batch=2)
    h1 = torch.zeros(s.n_taps, 2 * 17, s.target_hidden, dtype=torch.bfloat16)
    h1[:, 17:34] = hid[:, 20:37]
    tiny.gpu_inject(h1, [0, 17], rows_per_seq=17, batch=2)
    torch.cuda.synchronize()
    assert d.len[:2].tolist() == [37, 37]
    assert d.device_error() == 0
    # bit-exact persistence: one injection == two incremental injections
    assert torch.equal(d.k_cache[:, 0, :37], d.k_cache[:, 1, :37])
    assert torch.equal(d.v_cache[:, 0, :37], d.v_cache[:, 1, :37])
    # untouched positions stay zero
    assert not d.k_cache[:, 1, 37:64].any()
    # K and V are stored as fp16, and every injected value is finite
    assert d.k_cache.dtype == torch.float16 and d.v_cache.dtype == torch.float16
    assert bool(torch.isfinite(d.k_cache[:, :2, :37]).all()) and bool(torch.isfinite(d.v_cache[:, :2, :37]).all())
    # tolerance against the oracle
    st = tiny.oracle.new_sequence(64)
    tiny.oracle.inject(st, bits[:, :37])
    from gpu_util import max_rel, LAYER_RTOL
    k, v = tiny.gpu_cache(0, 37)
    for l in range(s.n_layers):
        assert max_rel(k[l], st.k_cache[l][:37]) <= LAYER_RTOL
        assert max_rel(v[l], st.v_cache[l][:37]) <= LAYER_RTOL


def test_inject_capacity_overflow_is_flagged(tiny):
    s = tiny.s
    d = tiny.drafter
    d.len[:1] = tiny.cap - 3
    h = torch.zeros(s.n_taps, 8, s.target_hidden, dtype=torch.bfloat16)
    tiny.gpu_inject(h, [8], rows_per_seq=8, batch=1)
    torch.cuda.synchronize()
    assert d.device_error() & 2
    assert int(d.len[0]) == tiny.cap
    d.len.zero_()


# ------------------------------------------------------------------ full step loop

@pytest.mark.parametrize("B", [4, 1, 16, 8, 12])
def test_step_loop_matches_oracle(tiny, B):
    """Prefill injection, then 3 steps of draft -> (synthetic target) -> verify -> inject,
    compared with the oracle at every stage. Verification is fed the oracle's drafts so a
    legitimately different draft (top-2 gap < 1e-2) cannot desynchronise the two sides."""
    _step_loop(tiny, B)


@pytest.mark.parametrize("B", [16, 4])
def test_step_loop_with_one_key_group(tiny, B):
    """The same loop with one warp per query head in the attention kernel (instead of two
    taking alternate key tiles)."""
    from block_diffusion_drafter_kv_gb300 import binding as BND
    d = tiny.drafter
    d.set_option(BND.OPT_ATTN_KEY_GROUPS, 1)
    try:
        _step_loop(tiny, B)
    finally:
        d.set_option(BND.OPT_ATTN_KEY_GROUPS, 2)


@pytest.mark.parametrize("B", [16, 4])
def test_step_loop_with_flat_attention(tiny, B):
    """The same loop with the flat key-split attention kernel (every pair's key tiles in one
    list over one CTA per SM). The tiny cache has fewer tiles than there are CTAs, so every
    pair of more than one tile is cut between CTAs and merged by the last to arrive."""
    from block_diffusion_drafter_kv_gb300 import binding as BND
    d = tiny.drafter
    d.set_option(BND.OPT_ATTN_MODE, 2)
    try:
        _step_loop(tiny, B)
    finally:
        d.set_option(BND.OPT_ATTN_MODE, 0)


def _step_loop(tiny, B):
    from gpu_util import check_draft, max_rel, LAYER_RTOL
    s, w = tiny.s, W_TINY
    d = tiny.drafter
    d.len.zero_()
    d.k_cache.zero_()
    d.v_cache.zero_()
    hid = I.make_hidden(s, 160, SEED, f"steps.{B}")
    bits = I.bf16_bits(hid)
    last = int(I.initial_tokens(1, s.vocab, SEED)[0])
    st = tiny.oracle.new_sequence(tiny.cap, last)
    tiny.oracle.inject(st, bits[:, : w.ctx])
    tiny.gpu_inject(hid[:, : w.ctx].contiguous(), [w.ctx], rows_per_seq=w.ctx, batch=1)
    d.last_token[0] = last
    for step in range(w.steps):
        N = st.length
        assert int(d.len[0]) == N
        k, v = tiny.gpu_cache(0, N)
        for l in range(s.n_layers):
            assert max_rel(k[l], st.k_cache[l][:N]) <= LAYER_RTOL
            assert max_rel(v[l], st.v_cache[l][:N]) <= LAYER_RTOL
        drafted = torch.full((1, max(B - 1, 1)), -1, dtype=torch.int32, device="cuda")
        logits = torch.full((1, max(B - 1, 1), s.vocab), float("nan"), device="cuda")
        trace = torch.full((s.n_layers + 1, B, s.hidden), float("nan"), device="cuda")
        d.draft(1, B, drafted, logits, trace)
        torch.cuda.synchronize()
        assert d.device_error() == 0
        ores = tiny.oracle.draft(st, B)
        check_draft(ores, drafted[0, : B - 1].cpu().numpy(), logits[0, : B - 1].cpu().numpy(),
                    trace.cpu().numpy())
        noise = I.make_logit_noise(1, B, s.vocab, SEED, f"logits.{B}.{step}").numpy()
        mask = I.make_plant_mask(1, B, w.p_plant, SEED, f"plant.{B}.{step}")
        T = I.plant_logits(noise, ores.drafted[None], mask)
        acc, com, lastg = _verify_gpu(tiny, T, ores.drafted[None], 1, B)
        r = tiny.oracle.verify(st, T[0], ores.drafted)
        assert acc[0] == r.accept_len and list(com[0, : r.accept_len]) == list(r.committed)
        assert lastg[0] == r.last_token == st.last_token
        tau = r.accept_len
        rows = torch.zeros(s.n_taps, 16, s.target_hidden, dtype=torch.bfloat16)
        rows[:, :tau] = hid[:, N:N + tau]
        tiny.gpu_inject(rows, [tau], rows_per_seq=16, batch=1)
        tiny.oracle.inject(st, bits[:, N:N + tau])
    torch.cuda.synchronize()
    assert int(d.len[0]) == st.length


def test_draft_rejects_misaligned_output_buffers(tiny):
    """logits and x_trace are written 16 bytes at a time: a buffer that is not 16-byte
    aligned is refused before any launch, and the handle stays usable."""
    from block_diffusion_drafter_kv_gb300 import binding as BND
    s, d = tiny.s, tiny.drafter
    B = 4
    drafted = torch.zeros(1, B - 1, dtype=torch.int32, device="cuda")
    flat = torch.zeros((B - 1) * s.vocab + 1, device="cuda")
    with pytest.raises(BND.DFlashError) as ei:
        d.draft(1, B, drafted, flat[1:].view(1, B - 1, s.vocab))
    assert ei.value.status == BND.DFLASH_E_INVAL
    trace = torch.zeros((s.n_layers + 1) * B * s.hidden + 1, device="cuda")
    with pytest.raises(BND.DFlashError) as ei:
        d.draft(1, B, drafted, None, trace[1:])
    assert ei.value.status == BND.DFLASH_E_INVAL
    d.device_error()  # clear what earlier tests left
    d.len.zero_()
    d.last_token.zero_()
    d.draft(1, B, drafted, flat[: (B - 1) * s.vocab].view(1, B - 1, s.vocab))
    torch.cuda.synchronize()
    assert d.device_error() == 0
    assert bool(torch.isfinite(flat[: (B - 1) * s.vocab]).all())


def test_verify_rejects_misaligned_logits(tiny):
    """Target logits are read 16 bytes at a time: a pointer that is not 16-byte aligned is
    refused before any launch (for every vocabulary size), and the handle stays usable."""
    from block_diffusion_drafter_kv_gb300 import binding as BND
    s, d = tiny.s, tiny.drafter
    B = 4
    flat = torch.zeros(B * s.vocab + 4, device="cuda")
    drafted = torch.zeros(1, B - 1, dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    com = torch.zeros(1, B, dtype=torch.int32, device="cuda")
    for off in (1, 2, 3):
        with pytest.raises(BND.DFlashError) as ei:
            d.verify(flat[off: off + B * s.vocab].view(1, B, s.vocab), drafted, 1, B, acc, com)
        assert ei.value.status == BND.DFLASH_E_INVAL
    d.verify(flat[4: 4 + B * s.vocab].view(1, B, s.vocab), drafted, 1, B, acc, com)
    torch.cuda.synchronize()
    assert 1 <= int(acc[0]) <= B


def test_options_round_trip(tiny):
    from block_diffusion_drafter_kv_gb300 import binding as BND
    d = tiny.drafter
    assert d.get_option(BND.OPT_WAIT_LIMIT_NS) == 2_000_000_000
    assert d.get_option(BND.OPT_CHAIN_MAX) == 8
    assert d.get_option(BND.OPT_ATTN_MODE) == 0
    for opt, bad in ((BND.OPT_WAIT_LIMIT_NS, 10), (BND.OPT_CHAIN_MAX, 9), (BND.OPT_GEMV_VARIANT, 6),
                     (BND.OPT_ATTN_SPLIT, 17), (BND.OPT_ATTN_MODE, 4), (BND.OPT_ATTN_MODE, -1), (99, 1)):
        with pytest.raises(BND.DFlashError):
            d.set_option(opt, bad)
    d.set_option(BND.OPT_CHAIN_MAX, 3)
    assert d.get_option(BND.OPT_CHAIN_MAX) == 3
    d.set_option(BND.OPT_CHAIN_MAX, 8)


def test_bounded_wait_unwinds_and_the_handle_recovers(tiny):
    """A chained projection kernel whose grid barrier can never be met (the self-test
    entry) gives up after the handle's 1 ms wait limit: the call returns, the timeout bit
    is set, and once it is read and cleared the same handle runs a full step loop that
    matches the oracle (tensor memory was released and the counters were reset)."""
    from block_diffusion_drafter_kv_gb300 import binding as BND
    d = tiny.drafter
    d.device_error()
    d.set_option(BND.OPT_WAIT_LIMIT_NS, 1_000_000)
    try:
        d.selftest_timeout()
        torch.cuda.synchronize()
        flags = d.device_error(clear=True)
        assert flags & BND.DEV_TIMEOUT
    finally:
        d.set_option(BND.OPT_WAIT_LIMIT_NS, 2_000_000_000)
    assert d.device_error() == 0
    _step_loop(tiny, 4)
