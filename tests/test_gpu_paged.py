"""The paged KV cache (dflash_bind_state_paged): a drafter whose K/V live in a shared pool
of 64-position pages, reached through a page table, must compute exactly what a drafter with
a sequence-major cache computes, for ragged sequences whose pages are scattered through the
pool: the same cache contents, drafts, logits, per-layer residuals and verification, call
after call. An out-of-range page id is flagged, not followed."""
import numpy as np
import pytest
import torch

from synth import W_TINY
from synth import inputs as I
from synth.configs import DrafterShape

pytestmark = pytest.mark.gpu
SEED = 55
BATCH, CAP, PPS = 3, 256, 4      # pages_per_seq * 64 = kv_capacity
# head dim 128, 4 query heads per KV head, 2 KV heads: the shape of the tensor-core flat
# attention kernel, at a size the tests run in seconds
TINY128 = DrafterShape(hidden=512, n_heads=8, n_kv_heads=2, head_dim=128, n_layers=2,
                       intermediate=1536, vocab=1024, n_taps=3, target_hidden=512, rope_theta=1e6)


@pytest.fixture(scope="module", params=[(W_TINY.shape, 0), (TINY128, 2), (TINY128, 3)],
                ids=["tiny-auto", "d128-flat-tensor-core", "d128-flat-mma-sync"])
def pair(request):
    """Two drafters of one shape and attention mode (DFLASH_OPT_ATTN_MODE): a sequence-major
    cache and a paged one. Mode 2 takes the tcgen05 flat kernel, which reads the cache in
    32-position steps (two per page); mode 3 the mma.sync flat kernel."""
    from block_diffusion_drafter_kv_gb300 import binding as B
    from block_diffusion_drafter_kv_gb300.build import build
    build()
    s, mode = request.param
    w = I.make_weights(s, SEED).to("cuda")
    flat = B.Drafter(s, w, max_block=16, max_batch=BATCH, kv_capacity=CAP)
    n_pages = BATCH * PPS + 5
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(SEED))[: BATCH * PPS]
    pt = perm.view(BATCH, PPS).to(torch.int32).cuda()
    paged = B.Drafter(s, w, max_block=16, max_batch=BATCH, kv_capacity=CAP, n_pages=n_pages, page_table=pt)
    for d in (flat, paged):
        d.set_option(B.OPT_ATTN_MODE, mode)
    return flat, paged, pt, s


def _gather(paged, pt, seq, upto):
    rows = torch.cat([pt[seq, p].long() * 64 + torch.arange(64, device="cuda") for p in range(PPS)])[:upto]
    return paged.k_cache[:, rows], paged.v_cache[:, rows]


def _step(d, s, batch, B, noise, drafted_in=None):
    drafted = torch.full((batch, B - 1), -1, dtype=torch.int32, device="cuda")
    logits = torch.full((batch, B - 1, s.vocab), float("nan"), device="cuda")
    trace = torch.full((s.n_layers + 1, batch * B, s.hidden), float("nan"), device="cuda")
    d.draft(batch, B, drafted, logits, trace)
    acc = torch.zeros(batch, dtype=torch.int32, device="cuda")
    com = torch.zeros(batch, B, dtype=torch.int32, device="cuda")
    d.verify(noise, drafted if drafted_in is None else drafted_in, batch, B, acc, com)
    torch.cuda.synchronize()
    return drafted, logits, trace, acc, com


def test_paged_cache_is_bit_identical_to_sequence_major(pair):
    flat, paged, pt, s = pair
    ctx = [70, 130, 37]          # ragged: 2, 3 and 1 pages
    rps = max(ctx)
    hid = I.make_hidden(s, BATCH * rps, SEED, "paged").cuda()
    nn = torch.tensor(ctx, dtype=torch.int32, device="cuda")
    last = torch.as_tensor(I.initial_tokens(BATCH, s.vocab, SEED), device="cuda")
    for d in (flat, paged):
        d.len.zero_()
        d.inject(hid, rps, nn, BATCH)
        d.last_token[:BATCH] = last
    torch.cuda.synchronize()
    assert flat.device_error() == 0 and paged.device_error() == 0
    for q in range(BATCH):
        k, v = _gather(paged, pt, q, ctx[q])
        assert torch.equal(k, flat.k_cache[:, q, : ctx[q]]) and torch.equal(v, flat.v_cache[:, q, : ctx[q]])
    B = 16
    for step in range(3):
        noise = I.make_logit_noise(BATCH, B, s.vocab, SEED, f"paged.{step}").cuda()
        a = _step(flat, s, BATCH, B, noise)
        b = _step(paged, s, BATCH, B, noise, drafted_in=a[0])
        for x, y in zip(a, b):
            assert torch.equal(x, y)
        assert torch.equal(flat.last_token[:BATCH], paged.last_token[:BATCH])
        rows = I.make_hidden(s, BATCH * B, SEED, f"paged.rows.{step}").cuda()
        for d in (flat, paged):
            d.inject(rows, B, a[3], BATCH)
        torch.cuda.synchronize()
        assert torch.equal(flat.len[:BATCH], paged.len[:BATCH])
    for q in range(BATCH):
        n = int(flat.len[q])
        k, v = _gather(paged, pt, q, n)
        assert torch.equal(k, flat.k_cache[:, q, :n]) and torch.equal(v, flat.v_cache[:, q, :n])
    assert flat.device_error() == 0 and paged.device_error() == 0


def test_out_of_range_page_is_flagged(pair):
    flat, paged, pt, s = pair
    saved = pt.clone()
    paged.len[:BATCH] = torch.tensor([60, 0, 0], dtype=torch.int32, device="cuda")
    pt[0, 1] = 10_000                     # the page that positions 64..127 of sequence 0 map to
    rows = torch.zeros(s.n_taps, 8, s.target_hidden, dtype=torch.bfloat16, device="cuda")
    paged.inject(rows, 8, torch.tensor([8, 0, 0], dtype=torch.int32, device="cuda"), BATCH)
    torch.cuda.synchronize()
    from block_diffusion_drafter_kv_gb300 import binding as BND
    assert paged.device_error() & BND.DEV_CAPACITY
    pt.copy_(saved)
    paged.len.zero_()


def test_wide_injection_passes_match_oracle_and_persist_bit_exact():
    """128-row injection passes (the prefill setting, DFLASH_OPT_INJECT_PASS_ROWS): the K/V of
    200 positions match the oracle, and injecting them in two calls (120 + 80 rows) gives
    bit-identical K/V to one call at the same width. (Different widths may differ in the
    last bits, which is why the width is fixed per handle.)"""
    from block_diffusion_drafter_kv_gb300 import binding as B
    from block_diffusion_drafter_kv_gb300.build import build
    from gpu_util import LAYER_RTOL, max_rel, to_np64
    from oracle.dflash_ref import Oracle
    build()
    s = W_TINY.shape
    w = I.make_weights(s, SEED)
    wc = w.to("cuda")
    one = B.Drafter(s, wc, max_block=16, max_batch=1, kv_capacity=CAP)
    two = B.Drafter(s, wc, max_block=16, max_batch=1, kv_capacity=CAP)
    for d in (one, two):
        d.set_option(B.OPT_INJECT_PASS_ROWS, 128)
    hid = I.make_hidden(s, 200, SEED, "widths")
    one.inject(hid.cuda(), 200, torch.tensor([200], dtype=torch.int32, device="cuda"), 1)
    two.inject(hid[:, :120].contiguous().cuda(), 120, torch.tensor([120], dtype=torch.int32, device="cuda"), 1)
    two.inject(hid[:, 120:].contiguous().cuda(), 80, torch.tensor([80], dtype=torch.int32, device="cuda"), 1)
    torch.cuda.synchronize()
    assert int(one.len[0]) == int(two.len[0]) == 200
    assert torch.equal(one.k_cache[:, 0, :200], two.k_cache[:, 0, :200])
    assert torch.equal(one.v_cache[:, 0, :200], two.v_cache[:, 0, :200])
    o = Oracle(s, w.bits())
    st = o.new_sequence(CAP)
    o.inject(st, I.bf16_bits(hid))
    k, v = to_np64(one.k_cache[:, 0, :200]), to_np64(one.v_cache[:, 0, :200])
    for l in range(s.n_layers):
        assert max_rel(k[l], st.k_cache[l][:200]) <= LAYER_RTOL
        assert max_rel(v[l], st.v_cache[l][:200]) <= LAYER_RTOL
