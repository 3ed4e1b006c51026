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


def test_full_size_step_matches_oracle(full):
    from gpu_util import check_draft, max_rel, LAYER_RTOL
    w, s, d = W_QWEN3_8B, full.s, full.drafter
    B = w.block
    hid = I.make_hidden(s, w.ctx + B, SEED, "full")
    bits = I.bf16_bits(hid)
    last = int(I.initial_tokens(1, s.vocab, SEED)[0])
    d.len.zero_()
    d.k_cache.zero_()
    d.v_cache.zero_()
    full.gpu_inject(hid[:, : w.ctx].contiguous(), [w.ctx], rows_per_seq=w.ctx, batch=1)
    d.last_token[0] = last
    st = full.oracle.new_sequence(full.cap, last)
    full.oracle.inject(st, bits[:, : w.ctx])
    torch.cuda.synchronize()
    assert int(d.len[0]) == w.ctx and d.device_error() == 0

    def check_cache(n0, n1):
        k, v = full.gpu_cache(0, n1)
        for l in range(s.n_layers):
            assert max_rel(k[l][n0:n1], st.k_cache[l][n0:n1]) <= LAYER_RTOL, f"K layer {l}"
            assert max_rel(v[l][n0:n1], st.v_cache[l][n0:n1]) <= LAYER_RTOL, f"V layer {l}"

    check_cache(0, w.ctx)

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
