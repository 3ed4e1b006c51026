"""Mutation checks of the oracle pins: each plausible mistake, planted in the oracle on
the CPU, must make at least one pin fail. This shows the pins constrain every part of
the oracle rather than restating it."""
import numpy as np
import pytest

import oracle.dflash_ref as R
import test_oracle_math as M
import test_oracle_model as MM
import test_oracle_sampling as SV
import test_oracle_target_verify as TV
import test_oracle_verify as V
from golden_io import load_sampling_cases, load_verify_cases


def _rope_wrong_sign(x, pos, theta):
    d = x.shape[-1]; h = d // 2
    ang = np.outer(np.asarray(pos, dtype=np.float64), R.rope_inv_freq(d, theta))
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1)


def _rope_interleaved(x, pos, theta):
    d = x.shape[-1]
    ang = np.outer(np.asarray(pos, dtype=np.float64), R.rope_inv_freq(d, theta))
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x1 * c - x2 * s
    out[..., 1::2] = x2 * c + x1 * s
    return out


def _rope_freq_exponent_d(x, pos, theta):   # theta^(-j/d) instead of theta^(-2j/d)
    d = x.shape[-1]; h = d // 2
    j = np.arange(h)
    ang = np.outer(np.asarray(pos, dtype=np.float64), theta ** (-j / d))
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def _rms_no_gain(x, g, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def _rms_eps_outside(x, g, eps):
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * g


def _gqa_modulo(q, keys, vals):
    B, nq, d = q.shape
    nkv = keys.shape[1]
    out = np.empty_like(q)
    for h in range(nq):
        g = h % nkv
        s = (q[:, h, :] @ keys[:, g, :].T) / np.sqrt(d)
        out[:, h, :] = R.softmax(s) @ vals[:, g, :]
    return out


def _causal(q, keys, vals):
    B, nq, d = q.shape
    S, nkv = keys.shape[0], keys.shape[1]
    out = np.empty_like(q)
    N = S - B
    for h in range(nq):
        g = h // (nq // nkv)
        s = (q[:, h, :] @ keys[:, g, :].T) / np.sqrt(d)
        for i in range(B):
            s[i, N + i + 1:] = -np.inf
        out[:, h, :] = R.softmax(s) @ vals[:, g, :]
    return out


def _no_scale(q, keys, vals):
    B, nq, d = q.shape
    nkv = keys.shape[1]
    out = np.empty_like(q)
    for h in range(nq):
        g = h // (nq // nkv)
        out[:, h, :] = R.softmax(q[:, h, :] @ keys[:, g, :].T) @ vals[:, g, :]
    return out


def _silu_wrong(x):
    return x / (1.0 + np.exp(x))


def _verify_off_by_one(T, d):
    r = _orig_verify(T, d)
    t = max(1, r.accept_len - 1) if r.accept_len == len(T) else r.accept_len
    return R.VerifyResult(t, r.committed[:t], int(r.committed[t - 1]), r.target_argmax)


def _verify_highest_tie(T, d):
    g = T.shape[1] - 1 - np.argmax(np.asarray(T)[:, ::-1], axis=-1)
    j = 0
    while j < len(g) - 1 and int(d[j]) == int(g[j]):
        j += 1
    return R.VerifyResult(j + 1, g[: j + 1], int(g[j]), g)


def _verify_skip_mismatch(T, d):   # counts all matching slots instead of the leading run
    g = np.argmax(T, axis=-1)
    j = int(sum(int(d[i]) == int(g[i]) for i in range(len(g) - 1)))
    return R.VerifyResult(j + 1, g[: j + 1], int(g[j]), g)


_orig_verify = R.verify_greedy
_orig_ctx = R.Oracle.context_feature
_orig_draft = R.Oracle.draft


def _ctx_taps_reversed(self, hidden_bits):
    return _orig_ctx(self, np.ascontiguousarray(hidden_bits[::-1]))


def _ctx_no_norm(self, hidden_bits):
    hid = R.bf16_to_float(hidden_bits, self.dtype)
    X = np.concatenate([hid[j] for j in range(hid.shape[0])], axis=-1)
    return (X @ self.W("w_fc").T) * self.W("g_ctx")


def _lm_chunk_short(self, h):   # each chunk one LM-head row short of its bound
    V = self.s.vocab
    if self._cache is not None:
        return h @ self.W("lm_head").T
    out = np.zeros((h.shape[0], V), dtype=self.dtype)
    bits = self.bits["lm_head"]
    for v0 in range(0, V, self.lm_chunk):
        v1 = min(V, v0 + self.lm_chunk - 1)
        out[:, v0:v1] = h @ R.bf16_to_float(bits[v0:v1], self.dtype).T
    return out


def _embed_row_next(self, tok):   # the uncached lookup widens the row after the token's
    if self._cache is not None:
        return self.W("embed")[tok]
    return R.bf16_to_float(self.bits["embed"][(tok + 1) % self.s.vocab], self.dtype)


def _target_no_final_norm(hidden_bits, gain_bits, lm_bits, eps, dtype=np.float64, chunk=16384):
    h = R.bf16_to_float(hidden_bits, dtype) * R.bf16_to_float(gain_bits, dtype)
    return h @ R.bf16_to_float(lm_bits, dtype).T


def _target_no_gain(hidden_bits, gain_bits, lm_bits, eps, dtype=np.float64, chunk=16384):
    h = R.bf16_to_float(hidden_bits, dtype)
    h = h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)
    return h @ R.bf16_to_float(lm_bits, dtype).T


_orig_sampling = R.verify_sampling


def _sampling_keeps_draft(target_logits, drafted, temperature, uniforms):
    # the residual keeps the rejected draft's probability
    p = R.softmax(np.asarray(target_logits, np.float64) / temperature, axis=-1)
    B = p.shape[0]
    j = 0
    while j < B - 1 and float(uniforms[j]) < p[j, int(drafted[j])]:
        j += 1
    tok = int(np.searchsorted(np.cumsum(p[j]), float(uniforms[B - 1]), side="right"))
    return R.SampleResult(j + 1, np.array([int(t) for t in drafted[:j]] + [tok]), tok, j)


def _sampling_no_temperature(target_logits, drafted, temperature, uniforms):
    return _orig_sampling(target_logits, drafted, 1.0, uniforms)


def _sampling_bonus_prev_row(target_logits, drafted, temperature, uniforms):
    r = _orig_sampling(target_logits, drafted, temperature, uniforms)
    B = np.asarray(target_logits).shape[0]
    if r.accept_len < B:
        return r
    p = R.softmax(np.asarray(target_logits, np.float64)[B - 2] / temperature)
    tok = int(np.searchsorted(np.cumsum(p), float(uniforms[B - 1]), side="right"))
    return R.SampleResult(B, np.array(list(r.committed[:-1]) + [tok]), tok, B - 1)


MUTATIONS = {
    "rope_sign": ("apply_rope", _rope_wrong_sign),
    "rope_interleaved_pairs": ("apply_rope", _rope_interleaved),
    "rope_freq_exponent": ("apply_rope", _rope_freq_exponent_d),
    "rms_no_gain": ("rms_norm", _rms_no_gain),
    "rms_eps_outside_sqrt": ("rms_norm", _rms_eps_outside),
    "gqa_modulo_mapping": ("gqa_attention", _gqa_modulo),
    "causal_mask": ("gqa_attention", _causal),
    "no_softmax_scale": ("gqa_attention", _no_scale),
    "silu_sign": ("silu", _silu_wrong),
    "verify_off_by_one": ("verify_greedy", _verify_off_by_one),
    "verify_tie_highest": ("verify_greedy", _verify_highest_tie),
    "verify_skips_mismatch": ("verify_greedy", _verify_skip_mismatch),
    "fc_taps_reversed": ("Oracle.context_feature", _ctx_taps_reversed),
    "fc_missing_rmsnorm": ("Oracle.context_feature", _ctx_no_norm),
    "lm_chunk_bound_short": ("Oracle._lm_head", _lm_chunk_short),
    "uncached_embed_wrong_row": ("Oracle._embed_row", _embed_row_next),
    "target_no_final_norm": ("target_logits_from_hidden", _target_no_final_norm),
    "target_no_gain": ("target_logits_from_hidden", _target_no_gain),
    "sampling_residual_keeps_draft": ("verify_sampling", _sampling_keeps_draft),
    "sampling_ignores_temperature": ("verify_sampling", _sampling_no_temperature),
    "sampling_bonus_previous_row": ("verify_sampling", _sampling_bonus_prev_row),
}


def _all_pins(tiny):
    """Run every pin; return the names of those that fail."""
    failed = []
    checks = {
        "rms_closed": M.test_rmsnorm_closed_form,
        "rms_eps": M.test_rmsnorm_eps_and_scale,
        "rope_first_pair": M.test_rope_first_pair_closed_form,
        "rope_complex": lambda: M.test_rope_matches_complex_rotation(64, 1e6),
        "attn_mha": M.test_attention_mha_matches_sdpa,
        "attn_gqa": M.test_attention_gqa_head_mapping_matches_sdpa,
        "attn_bidir": M.test_attention_is_bidirectional,
        "silu": M.test_silu_closed_forms,
        "verify_golden": lambda: [V.test_hand_worked_cases(c) for c in load_verify_cases()],
        "verify_masks": lambda: V.test_all_agreement_masks(4),
        "verify_lossless": V.test_lossless_committed_equal_target_greedy,
        "inject_naive": lambda: MM.test_injection_matches_naive(tiny),
        "draft_naive": lambda: MM.test_draft_steps_match_naive_recomputation(tiny),
        "uncached_naive": lambda: MM.test_uncached_chunked_oracle_matches_naive(tiny),
        "uncached_equals_cached": lambda: MM.test_uncached_chunked_oracle_equals_cached(tiny),
        "target_naive": lambda: [TV.test_matches_naive_scalar_loops(sd, b) for sd, b in ((0, 4), (2, 7))],
        "target_planted": TV.test_planted_agreement_and_slot0_mismatch,
        "target_scale": TV.test_final_norm_makes_logits_scale_invariant,
        "sampling_golden": lambda: [SV.test_hand_worked_cases(c) for c in load_sampling_cases()],
        "sampling_distribution": SV.test_committed_tokens_follow_the_target_distribution,
        "sampling_low_temperature": SV.test_low_temperature_equals_greedy,
    }
    for name, fn in checks.items():
        try:
            fn()
        except Exception:
            failed.append(name)
    return failed


@pytest.fixture(scope="module")
def tiny():
    return _make_tiny()


def _make_tiny():
    from synth import W_TINY
    from synth import inputs as I
    s = W_TINY.shape
    return s, I.make_weights(s, MM.SEED).bits(), I.bf16_bits(I.make_hidden(s, 160, MM.SEED))


def test_unmutated_oracle_passes_every_pin(tiny):
    assert _all_pins(tiny) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tiny, monkeypatch):
    target, fn = MUTATIONS[name]
    if target.startswith("Oracle."):
        monkeypatch.setattr(R.Oracle, target.split(".", 1)[1], fn)
    else:
        monkeypatch.setattr(R, target, fn)
        for mod in (M, V):                       # modules that imported the name directly
            if hasattr(mod, target):
                monkeypatch.setattr(mod, target, fn)
    failed = _all_pins(tiny)
    assert failed, f"mutation {name} survived every pin"
