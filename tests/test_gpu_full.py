"""Parity at the full Qwen3-8B-shaped drafter size (H=4096, 32/8 heads, head_dim 128, 5 layers,
SwiGLU 12288, vocab 151936, k=5 taps), batch 1, context 2048, B=16: the launch configuration
the benchmark times. The oracle runs the whole step here (float64, weights widened per use),
so every output is compared, not a sample: the injected KV cache, every layer's residual
stream, the block's logits, the drafted tokens, and verification bit-exact; then one
incremental injection of the accepted rows and a second draft on the grown cache."""
import numpy as np
import pytest
import torch

from synth import W_QWEN3_8B
from synth import inputs as I

pytestmark = pytest.mark.gpu

SEED = 77


@pytest.fixture(scope="module")
def full():
    from gpu_util import Setup
    w = W_QWEN3_8B
    return Setup(w, seed=SEED, max_batch=1, kv_capacity=w.ctx + 64)


def _draft(full, B):
    s = full.s
    d = full.drafter
    drafted = torch.full((1, B - 1), -1, dtype=torch.int32, device="cuda")
    logits = torch.full((1, B - 1, s.vocab), float("nan"), device="cuda")
    trace = torch.full((s.n_layers + 1, B, s.hidden), float("nan"), device="cuda")
    d.draft(1, B, drafted, logits, trace)
    torch.cuda.synchronize()
    assert d.device_error() == 0
    return drafted[0].cpu().numpy(), logits[0].cpu().numpy(), trace.cpu().numpy()


class _Prefilled:
    pass


@pytest.fixture(scope="module")
def prefilled(full):
    """The 2048-position context injected on both sides (checked element by element), and
    the slot-0 token set: the state every block size below drafts from."""
    from gpu_util import max_rel, LAYER_RTOL
    w, s, d = W_QWEN3_8B, full.s, full.drafter
    P = _Prefilled()
    P.hid = I.make_hidden(s, w.ctx + w.block, SEED, "full")
    P.bits = I.bf16_bits(P.hid)
    last = int(I.initial_tokens(1, s.vocab, SEED)[0])
    d.len.zero_()
    d.k_cache.zero_()
    d.v_cache.zero_()
    full.gpu_inject(P.hid[:, : w.ctx].contiguous(), [w.ctx], rows_per_seq=w.ctx, batch=1)
    d.last_token[0] = last
    P.st = full.oracle.new_sequence(full.cap, last)
    full.oracle.inject(P.st, P.bits[:, : w.ctx])
    torch.cuda.synchronize()
    assert int(d.len[0]) == w.ctx and d.device_error() == 0

    def check_cache(n0, n1):
        k, v = full.gpu_cache(0, n1)
        for l in range(s.n_layers):
            assert max_rel(k[l][n0:n1], P.st.k_cache[l][n0:n1]) <= LAYER_RTOL, f"K layer {l}"
            assert max_rel(v[l][n0:n1], P.st.v_cache[l][n0:n1]) <= LAYER_RTOL, f"V layer {l}"

    check_cache(0, w.ctx)
    P.check_cache = check_cache
    return P


@pytest.mark.parametrize("B", [4, 8, 12])
def test_full_size_block_sweep_draft_matches_oracle(full, prefilled, B):
    """The block-size sweep (B = 4, 8, 12 beside the 16 below) on the same injected context:
    every layer's residual, the logits and the drafted tokens against the oracle."""
    from gpu_util import check_draft
    assert int(full.drafter.len[0]) == prefilled.st.length == W_QWEN3_8B.ctx
    g_dr, g_lo, g_tr = _draft(full, B)
    check_draft(full.oracle.draft(prefilled.st, B), g_dr, g_lo, g_tr)


@pytest.mark.parametrize("mode,B", [(2, 16), (2, 4), (3, 16)])
def test_full_size_flat_attention_matches_oracle(full, prefilled, mode, B):
    """The flat key-split attention kernels (the default for many or long sequences) on the
    single-sequence context: 33 key tiles per KV head cut over every SM, so each head is
    merged from several CTAs' parts. Mode 2 takes the tcgen05 kernel (head dim 128, groups
    of 4 query heads; at B = 4 most of its 64 query rows are unused slots), mode 3 the
    mma.sync one. Every layer's residual, the logits and the drafts against the oracle."""
    from gpu_util import check_draft
    from block_diffusion_drafter_kv_gb300 import binding as BND
    d = full.drafter
    d.set_option(BND.OPT_ATTN_MODE, mode)
    try:
        g_dr, g_lo, g_tr = _draft(full, B)
    finally:
        d.set_option(BND.OPT_ATTN_MODE, 0)
    check_draft(full.oracle.draft(prefilled.st, B), g_dr, g_lo, g_tr)


def test_full_size_step_matches_oracle(full, prefilled):
    from gpu_util import check_draft
    w, s, d = W_QWEN3_8B, full.s, full.drafter
    B = w.block
    st, hid, bits, check_cache = prefilled.st, prefilled.hid, prefilled.bits, prefilled.check_cache

    # first draft on the injected context
    g_dr, g_lo, g_tr = _draft(full, B)
    ores = full.oracle.draft(st, B)
    check_draft(ores, g_dr, g_lo, g_tr)

    # verification of the oracle's drafts against planted target logits: bit-exact
    noise = I.make_logit_noise(1, B, s.vocab, SEED, "full.logits").numpy()
    mask = I.make_plant_mask(1, B, w.p_plant, SEED, "full.plant")
    T = I.plant_logits(noise, ores.drafted[None], mask)
    acc = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    com = torch.full((1, B), -7, dtype=torch.int32, device="cuda")
    dd = torch.as_tensor(ores.drafted[None].astype(np.int32), device="cuda")
    d.verify(torch.as_tensor(T, device="cuda"), dd, 1, B, acc, com)
    torch.cuda.synchronize()
    r = full.oracle.verify(st, T[0], ores.drafted)
    assert int(acc[0]) == r.accept_len
    assert list(com[0, : r.accept_len].cpu().numpy()) == list(r.committed)
    assert int(d.last_token[0]) == r.last_token

    # incremental injection of the accepted rows, then a second draft on the grown cache
    tau = r.accept_len
    rows = torch.zeros(s.n_taps, 16, s.target_hidden, dtype=torch.bfloat16)
    rows[:, :tau] = hid[:, w.ctx: w.ctx + tau]
    full.gpu_inject(rows, [tau], rows_per_seq=16, batch=1)
    full.oracle.inject(st, bits[:, w.ctx: w.ctx + tau])
    torch.cuda.synchronize()
    assert int(d.len[0]) == st.length == w.ctx + tau
    check_cache(w.ctx, w.ctx + tau)
    g_dr, g_lo, g_tr = _draft(full, B)
    ores = full.oracle.draft(st, B)
    check_draft(ores, g_dr, g_lo, g_tr)


# ------------------------------------------------------------------ batched and long-context configs
# Sequences are independent in every step of the path (projections act row by row,
# attention within a sequence, verification per sequence), so at these sizes the oracle
# checks sampled sequences of a full-size GPU run. Sequences the oracle does not check get
# N(0,1) hidden states drawn on the device.

def _run_sampled(w, seed, sampled, oracle_dtype=np.float64, chunk=4096, attn_mode=0):
    from gpu_util import Setup, check_draft, max_rel, LAYER_RTOL
    from oracle.dflash_ref import Oracle
    from block_diffusion_drafter_kv_gb300 import binding as BND
    s, B, batch = w.shape, w.block, w.batch
    ctx = I.ragged_ctx(w, seed)
    sampled = list(sampled(ctx))
    cap = int(ctx.max()) + 64
    S = Setup(w, seed=seed, max_batch=batch, kv_capacity=cap)
    d = S.drafter
    d.set_option(BND.OPT_ATTN_MODE, attn_mode)
    rps = int(ctx.max())
    hid = torch.empty(s.n_taps, batch * rps, s.target_hidden, dtype=torch.bfloat16, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed)
    hid.normal_(generator=g)
    host = {}
    for q in sampled:
        h = I.make_hidden(s, int(ctx[q]) + B, seed, f"seq{q}")
        host[q] = h
        hid[:, q * rps: q * rps + int(ctx[q])] = h[:, : int(ctx[q])].cuda()
    last = I.initial_tokens(batch, s.vocab, seed)
    d.len.zero_()
    d.inject(hid, rps, torch.as_tensor(ctx, dtype=torch.int32, device="cuda"), batch)
    d.last_token[:batch] = torch.as_tensor(last, device="cuda")
    torch.cuda.synchronize()
    assert d.len[:batch].cpu().tolist() == ctx.tolist() and d.device_error() == 0
    del hid
    o = Oracle(s, S.bits, dtype=oracle_dtype)
    states = {}
    for q in sampled:
        st = o.new_sequence(cap, int(last[q]))
        bits = I.bf16_bits(host[q][:, : int(ctx[q])])
        for r0 in range(0, int(ctx[q]), chunk):
            o.inject(st, bits[:, r0: r0 + chunk])
        states[q] = st
        k, v = S.gpu_cache(q, int(ctx[q]))
        for l in range(s.n_layers):
            assert max_rel(k[l], st.k_cache[l][: st.length]) <= LAYER_RTOL, f"seq {q} K layer {l}"
            assert max_rel(v[l], st.v_cache[l][: st.length]) <= LAYER_RTOL, f"seq {q} V layer {l}"
    drafted = torch.full((batch, B - 1), -1, dtype=torch.int32, device="cuda")
    logits = torch.full((batch, B - 1, s.vocab), float("nan"), device="cuda")
    trace = torch.full((s.n_layers + 1, batch * B, s.hidden), float("nan"), device="cuda")
    d.draft(batch, B, drafted, logits, trace)
    torch.cuda.synchronize()
    assert d.device_error() == 0
    dr = drafted.cpu().numpy()
    ores = {}
    for q in sampled:
        ores[q] = o.draft(states[q], B)
        check_draft(ores[q], dr[q], logits[q].cpu().numpy(), trace[:, q * B:(q + 1) * B].cpu().numpy())
        dr[q] = ores[q].drafted
    # verification of the whole batch; the sampled sequences against the oracle, bit-exact
    noise = I.make_logit_noise(batch, B, s.vocab, seed, "full.logits").numpy()
    mask = I.make_plant_mask(batch, B, I.per_seq_p(w, seed), seed, "full.plant")
    T = I.plant_logits(noise, dr, mask)
    acc = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    com = torch.full((batch, B), -7, dtype=torch.int32, device="cuda")
    d.verify(torch.as_tensor(T, device="cuda"), torch.as_tensor(dr, device="cuda"), batch, B, acc, com)
    torch.cuda.synchronize()
    for q in sampled:
        r = o.verify(states[q], T[q], dr[q])
        assert int(acc[q]) == r.accept_len
        assert list(com[q, : r.accept_len].cpu().numpy()) == list(r.committed)
        assert int(d.last_token[q]) == r.last_token


@pytest.mark.parametrize("attn_mode", [0, 2])
def test_batched_ragged_sampled_sequences_match_oracle(attn_mode):
    """Batch 32, context lengths uniform in [512, 8192], B = 16, per-sequence agreement
    rates. Sampled by index: one sequence in each group of eight (the rows of one 128-row
    projection pass, and of one 256-row pass in pairs of groups), plus the sequence with
    the longest context (the most key tiles per attention CTA). Attention by the default
    choice for this batch (the mma.sync flat split) and by the tcgen05 flat kernel."""
    from synth import W_BATCHED
    _run_sampled(W_BATCHED, 31, lambda ctx: sorted({3, 12, 21, 30, int(np.argmax(ctx))}), attn_mode=attn_mode)


def test_long_context_llama_shaped_sequence_matches_oracle():
    """Llama-3.1-8B-shaped drafter (8 layers, SwiGLU 14336, vocab 128256, theta 5e5), batch 4
    at context 32768, B = 16: sequence 0 against the oracle in fp32."""
    from synth import W_LLAMA
    _run_sampled(W_LLAMA, 41, lambda ctx: [0], oracle_dtype=np.float32)
