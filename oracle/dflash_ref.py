"""Reference (oracle) implementation of one DFlash draft-and-verify step.

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the CPU-baseline
leg of the benchmark, never by the library.

Plain NumPy, computing in float64 unless another dtype is asked for. Weights and
target hidden states arrive as bf16 bit patterns (uint16) and are widened exactly.
One sequence at a time, every step in the order the pages give it:

  inject  — hidden states from several target layers are fused into one compact
            target-context feature, which is injected into the Key and Value
            projections of every draft layer; those projections sit in the draft
            KV cache and persist across drafting iterations
            (theaistack.guide, "L'idea chiave: Il target sa meglio";
             7minutos.es, "La idea de que 'el objetivo sabe más'";
             jansverre.net, "Hva gjør DFlash annerledes enn vanlig spekulativ dekoding?").
  draft   — a whole masked token block is denoised in one forward pass
            (jansverre.net, same section; theaistack.guide, "Come funziona il drafting
             a blocchi"); attention inside the block is bidirectional.
  verify  — the target checks the block in parallel and keeps the longest valid
            prefix (bpdata.com, introduction and "Hogyan működik a DFlash
            spekulatív dekódolás?"), which keeps the output lossless
            (theaistack.guide, "DFlash").

Readings where the pages are silent (each listed in the design notes):
  * fusion: X = concat of the k tapped layers along features in tap order,
    F = X·Wfcᵀ, c = RMSNorm(F)·g_ctx; K_l = RoPE(c·Wk_lᵀ), V_l = c·Wv_lᵀ using each
    draft layer's own Wk/Wv.
  * block: slot 0 is the last accepted token (embedding row), slots 1..B-1 hold a
    learned mask embedding; slot i sits at position N+i where N is the number of
    injected positions.
  * pre-norm layers (RMSNorm, eps 1e-6) with residual adds, SwiGLU MLP, a final
    RMSNorm before the LM head; rotate-half RoPE, inv_freq_j = theta^(-2j/d).
  * LM head on slots 1..B-1 only; argmax ties go to the lowest index.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np


# ----------------------------------------------------------------------------- helpers

def bf16_to_float(bits: np.ndarray, dtype=np.float64) -> np.ndarray:
    """Widen bf16 bit patterns to `dtype` exactly (bf16 is the top half of an fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(dtype)


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope_inv_freq(d: int, theta: float, dtype=np.float64) -> np.ndarray:
    j = np.arange(d // 2, dtype=np.float64)
    return (theta ** (-(2.0 * j) / d)).astype(dtype)


def apply_rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE. x [n, heads, d], pos [n] absolute positions.

    Pair (j, j + d/2) is rotated by angle pos * theta^(-2j/d):
      out[j]       = x[j] cos - x[j+d/2] sin
      out[j + d/2] = x[j+d/2] cos + x[j] sin
    """
    d = x.shape[-1]
    h = d // 2
    ang = np.outer(np.asarray(pos, dtype=np.float64), rope_inv_freq(d, theta)).astype(x.dtype)
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def gqa_attention(q: np.ndarray, keys: np.ndarray, vals: np.ndarray) -> np.ndarray:
    """Bidirectional (unmasked) attention of every query over every key.

    q [B, nq, d]; keys, vals [S, nkv, d]; query head h reads kv head h // (nq/nkv).
    Returns [B, nq, d].
    """
    B, nq, d = q.shape
    nkv = keys.shape[1]
    group = nq // nkv
    out = np.empty_like(q)
    scale = 1.0 / np.sqrt(d)
    for h in range(nq):
        g = h // group
        s = (q[:, h, :] @ keys[:, g, :].T) * scale      # [B, S]
        out[:, h, :] = softmax(s, axis=-1) @ vals[:, g, :]
    return out


def argmax_lowest(z: np.ndarray, axis: int = -1) -> np.ndarray:
    """Index of the maximum; the first (lowest) index wins ties."""
    return np.argmax(z, axis=axis)


# ----------------------------------------------------------------------------- verify

@dataclass
class VerifyResult:
    accept_len: int            # tau in [1, B]: accepted drafts plus the bonus token
    committed: np.ndarray      # [tau] target-greedy tokens g_0..g_{tau-1}
    last_token: int            # g_{tau-1}, the next block's slot 0
    target_argmax: np.ndarray  # [B]


def verify_greedy(target_logits: np.ndarray, drafted: np.ndarray) -> VerifyResult:
    """Greedy verification: keep the longest prefix of drafts matching the target's argmax.

    target_logits [B, V] (row i = the target's prediction after slot i), drafted [B-1]
    (drafted[i] = d_{i+1}, the draft at slot i+1). j = number of leading i with
    d_{i+1} == g_i; tau = j + 1; committed = g_0..g_j; the bonus g_j becomes slot 0.
    """
    g = argmax_lowest(np.asarray(target_logits, dtype=np.float64), axis=-1)
    B = g.shape[0]
    j = 0
    while j < B - 1 and int(drafted[j]) == int(g[j]):
        j += 1
    return VerifyResult(j + 1, g[: j + 1].astype(np.int64), int(g[j]), g.astype(np.int64))


# ----------------------------------------------------------------------------- fused target verify

def target_logits_from_hidden(hidden_bits: np.ndarray, gain_bits: np.ndarray, lm_bits: np.ndarray,
                              eps: float, dtype=np.float64, chunk: int = 16384) -> np.ndarray:
    """The target's logits of B block positions from its last hidden states: the target's
    own final RMSNorm (gain g, the drafter's eps) and LM head, z = RMSNorm(h)·g · W_lmᵀ.
    hidden [B, Ht], gain [Ht], lm [V, Ht] as bf16 bit patterns; returns [B, V]. The LM head
    rows are widened `chunk` at a time; each logit is one whole dot product."""
    h = rms_norm(bf16_to_float(hidden_bits, dtype), bf16_to_float(gain_bits, dtype), eps)
    V = lm_bits.shape[0]
    z = np.empty((h.shape[0], V), dtype=dtype)
    for v0 in range(0, V, chunk):
        z[:, v0:v0 + chunk] = h @ bf16_to_float(lm_bits[v0:v0 + chunk], dtype).T
    return z


def verify_greedy_from_hidden(hidden_bits: np.ndarray, gain_bits: np.ndarray, lm_bits: np.ndarray,
                              drafted: np.ndarray, eps: float):
    """Greedy verification starting from the target's last hidden states instead of its
    logits (the target checks the drafted block in one parallel pass and keeps the longest
    valid prefix: bpdata.com, introduction). The target's argmax g_i of each position comes
    from its final norm and LM head (target_logits_from_hidden); the accept rule is
    verify_greedy's. Returns (VerifyResult, logits [B, V])."""
    z = target_logits_from_hidden(hidden_bits, gain_bits, lm_bits, eps)
    return verify_greedy(z, drafted), z


# ----------------------------------------------------------------------------- sampling verify

@dataclass
class SampleResult:
    accept_len: int            # tau in [1, B]: accepted drafts plus the sampled token
    committed: np.ndarray      # [tau] d_1..d_{tau-1}, then the sampled token
    last_token: int            # committed[-1], the next block's slot 0
    stop_row: int              # the row the last token was sampled from (tau - 1)


def verify_sampling(target_logits: np.ndarray, drafted: np.ndarray, temperature: float,
                    uniforms: np.ndarray) -> SampleResult:
    """Verification when the target samples at a temperature (7minutos.es, "Casos de uso con
    ejemplos": the method is also measured under sampling, at about 3.9x). The pages state no
    accept rule; the reading taken here is the standard speculative-sampling rule for a
    drafter whose proposal is its own argmax (a point mass q_i at d_{i+1}), which keeps the
    committed tokens distributed exactly as the target's own samples:

      p_i = softmax(target_logits[i] / temperature)
      for i = 0..B-2: accept d_{i+1} if uniforms[i] < p_i(d_{i+1}) (= min(1, p_i / q_i));
                      else stop at row i
      at the stop row j the last token is sampled with uniforms[B-1] by inverse CDF (the
      first index whose cumulative probability exceeds it) from
        p_j without d_{j+1}, renormalised (the residual max(0, p_j - q_j)),  j < B-1
        p_{B-1} itself (every draft accepted: the bonus token),             j = B-1

    target_logits [B, V]; drafted [B-1]; uniforms [B] in [0, 1)."""
    z = np.asarray(target_logits, dtype=np.float64) / float(temperature)
    p = softmax(z, axis=-1)
    B = p.shape[0]
    j = 0
    while j < B - 1 and float(uniforms[j]) < p[j, int(drafted[j])]:
        j += 1
    r = p[j].copy()
    if j < B - 1:
        r[int(drafted[j])] = 0.0
    r /= r.sum()
    tok = int(np.searchsorted(np.cumsum(r), float(uniforms[B - 1]), side="right"))
    tok = min(tok, int(np.flatnonzero(r > 0)[-1]))
    committed = np.array([int(t) for t in drafted[:j]] + [tok], dtype=np.int64)
    return SampleResult(j + 1, committed, tok, j)


# ----------------------------------------------------------------------------- model

@dataclass
class SeqState:
    """Persistent per-sequence drafter state: injected K (post-RoPE) and V per layer."""
    k_cache: List[np.ndarray]  # L x [cap, nkv, d]
    v_cache: List[np.ndarray]
    length: int = 0            # N, injected positions
    last_token: int = 0


@dataclass
class DraftResult:
    drafted: np.ndarray        # [B-1] int64, d_1..d_{B-1}
    logits: np.ndarray         # [B-1, V]
    x_trace: np.ndarray        # [L+1, B, H]: block input, then residual after each layer
    top2_gap: np.ndarray       # [B-1] gap between the two largest logits


class Oracle:
    """The step for one drafter. `weights` maps tensor names to bf16 bit arrays:
    w_fc, g_ctx, embed, mask_emb, g_final, lm_head, layers.{l}.{wq,wk,wv,wo,w_gate,w_up,
    w_down,g_attn,g_mlp}."""

    def __init__(self, shape, weights: Dict[str, np.ndarray], dtype=np.float64,
                 cache_limit_bytes: int = 3 << 30, lm_chunk: int = 16384):
        self.s = shape
        self.bits = weights
        self.dtype = dtype
        self.lm_chunk = lm_chunk
        total = sum(v.size for v in weights.values()) * np.dtype(dtype).itemsize
        self._cache: Optional[Dict[str, np.ndarray]] = {} if total <= cache_limit_bytes else None

    def W(self, name: str) -> np.ndarray:
        if self._cache is not None:
            if name not in self._cache:
                self._cache[name] = bf16_to_float(self.bits[name], self.dtype)
            return self._cache[name]
        return bf16_to_float(self.bits[name], self.dtype)

    def L(self, l: int, name: str) -> np.ndarray:
        return self.W(f"layers.{l}.{name}")

    def new_sequence(self, capacity: int, last_token: int = 0) -> SeqState:
        s = self.s
        mk = lambda: np.zeros((capacity, s.n_kv_heads, s.head_dim), dtype=self.dtype)
        return SeqState([mk() for _ in range(s.n_layers)], [mk() for _ in range(s.n_layers)],
                        0, int(last_token))

    # -- KV injection -------------------------------------------------------------
    def context_feature(self, hidden_bits: np.ndarray) -> np.ndarray:
        """c = RMSNorm(concat_j hidden[j] · Wfcᵀ) · g_ctx for hidden [k, n, Ht]; returns [n, H]."""
        hid = bf16_to_float(hidden_bits, self.dtype)
        k, n, Ht = hid.shape
        X = np.concatenate([hid[j] for j in range(k)], axis=-1)      # [n, k*Ht], tap order
        F = X @ self.W("w_fc").T                                        # [n, H]
        return rms_norm(F, self.W("g_ctx"), self.s.rms_eps)

    def inject(self, st: SeqState, hidden_bits: np.ndarray) -> np.ndarray:
        """Append the injected K/V of n new positions (hidden [k, n, Ht]) at N..N+n-1; N += n.
        Returns c [n, H]."""
        s = self.s
        n = hidden_bits.shape[1]
        if st.length + n > st.k_cache[0].shape[0]:
            raise ValueError("KV capacity exceeded")
        if n == 0:
            return np.zeros((0, s.hidden), dtype=self.dtype)
        c = self.context_feature(hidden_bits)
        pos = np.arange(st.length, st.length + n)
        for l in range(s.n_layers):
            kc = (c @ self.L(l, "wk").T).reshape(n, s.n_kv_heads, s.head_dim)
            vc = (c @ self.L(l, "wv").T).reshape(n, s.n_kv_heads, s.head_dim)
            st.k_cache[l][st.length:st.length + n] = apply_rope(kc, pos, s.rope_theta)
            st.v_cache[l][st.length:st.length + n] = vc
        st.length += n
        return c

    # -- block draft --------------------------------------------------------------
    def draft(self, st: SeqState, B: int) -> DraftResult:
        s = self.s
        H, nq, nkv, d = s.hidden, s.n_heads, s.n_kv_heads, s.head_dim
        N = st.length
        x = np.empty((B, H), dtype=self.dtype)
        x[0] = self._embed_row(st.last_token)
        x[1:] = self.W("mask_emb")
        trace = [x.copy()]
        pos = np.arange(N, N + B)
        for l in range(s.n_layers):
            a = rms_norm(x, self.L(l, "g_attn"), s.rms_eps)
            q = (a @ self.L(l, "wq").T).reshape(B, nq, d)
            k = (a @ self.L(l, "wk").T).reshape(B, nkv, d)
            v = (a @ self.L(l, "wv").T).reshape(B, nkv, d)
            q = apply_rope(q, pos, s.rope_theta)
            k = apply_rope(k, pos, s.rope_theta)
            keys = np.concatenate([st.k_cache[l][:N], k], axis=0)       # injected ctx ++ block
            vals = np.concatenate([st.v_cache[l][:N], v], axis=0)
            o = gqa_attention(q, keys, vals).reshape(B, nq * d)
            x = x + o @ self.L(l, "wo").T
            a2 = rms_norm(x, self.L(l, "g_mlp"), s.rms_eps)
            act = silu(a2 @ self.L(l, "w_gate").T) * (a2 @ self.L(l, "w_up").T)
            x = x + act @ self.L(l, "w_down").T
            trace.append(x.copy())
        hfin = rms_norm(x[1:], self.W("g_final"), s.rms_eps)            # slots 1..B-1
        logits = self._lm_head(hfin)
        drafted = argmax_lowest(logits, axis=-1)
        if B > 1:
            part = np.partition(logits, -2, axis=-1)
            gap = part[:, -1] - part[:, -2]
        else:                                                            # no drafted slots
            gap = np.zeros(0, dtype=self.dtype)
        return DraftResult(drafted.astype(np.int64), logits, np.stack(trace), gap)

    def _embed_row(self, tok: int) -> np.ndarray:
        """Row `tok` of the token embedding E (slot 0 of the block). Without the widened-weight
        cache only that one row of E is widened."""
        if self._cache is not None:
            return self.W("embed")[tok]
        return bf16_to_float(self.bits["embed"][tok], self.dtype)

    def _lm_head(self, h: np.ndarray) -> np.ndarray:
        V = self.s.vocab
        if self._cache is not None:
            return h @ self.W("lm_head").T
        out = np.empty((h.shape[0], V), dtype=self.dtype)
        bits = self.bits["lm_head"]
        for v0 in range(0, V, self.lm_chunk):           # rows of the LM head, each dot product whole
            v1 = min(V, v0 + self.lm_chunk)
            out[:, v0:v1] = h @ bf16_to_float(bits[v0:v1], self.dtype).T
        return out

    # -- one step -----------------------------------------------------------------
    def verify(self, st: SeqState, target_logits: np.ndarray, drafted: np.ndarray) -> VerifyResult:
        r = verify_greedy(target_logits, drafted)
        st.last_token = r.last_token
        return r
