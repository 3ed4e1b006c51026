"""Naive per-slot recomputation of the DFlash draft for tiny shapes — TEST INFRASTRUCTURE ONLY.

A second, independent statement of the same draft forward, written to pin
`dflash_ref` by brute force (it is far too slow for real shapes):

  * no persistent cache: every call rebuilds the injected K/V of all N context
    positions from the full history of target hidden states, position by position;
  * every projection is a loop of per-output dot products, every norm and every
    softmax a Python loop over scalars;
  * RoPE is written as a complex rotation: (x_j + i x_{j+d/2}) * exp(i * pos * w_j),
    the textbook complex form of rotary embeddings, not the rotate-half formula;
  * verify takes the largest tau whose whole prefix agrees, trying every tau.

It follows the same readings as `dflash_ref` (see that module's header) and shares
no code with it.
"""
from __future__ import annotations

import cmath
import math
from typing import Dict, List, Sequence

import numpy as np


def _f(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _matvec(Wm: np.ndarray, v: np.ndarray) -> np.ndarray:
    return np.array([float(np.dot(Wm[r], v)) for r in range(Wm.shape[0])])


def _rmsnorm(v: Sequence[float], g: np.ndarray, eps: float) -> np.ndarray:
    acc = 0.0
    for t in v:
        acc += t * t
    inv = 1.0 / math.sqrt(acc / len(v) + eps)
    return np.array([v[i] * inv * g[i] for i in range(len(v))])


def _rope_complex(vec: np.ndarray, pos: int, theta: float) -> np.ndarray:
    d = len(vec)
    h = d // 2
    out = np.empty(d)
    for j in range(h):
        w = theta ** (-2.0 * j / d)
        z = complex(vec[j], vec[j + h]) * cmath.exp(1j * pos * w)
        out[j], out[j + h] = z.real, z.imag
    return out


def _silu(t: float) -> float:
    return t / (1.0 + math.exp(-t))


def naive_context_kv(shape, W: Dict[str, np.ndarray], hist_bits: np.ndarray):
    """Injected K (post-RoPE) and V for every context position from scratch.
    hist_bits [k, N, Ht]. Returns K, V as lists over layers of [N][nkv][d]."""
    s = shape
    hid = _f(hist_bits)
    Wfc, gctx = _f(W["w_fc"]), _f(W["g_ctx"])
    N = hid.shape[1]
    K = [np.zeros((N, s.n_kv_heads, s.head_dim)) for _ in range(s.n_layers)]
    V = [np.zeros((N, s.n_kv_heads, s.head_dim)) for _ in range(s.n_layers)]
    for p in range(N):
        xcat = np.concatenate([hid[j, p] for j in range(s.n_taps)])
        c = _rmsnorm(_matvec(Wfc, xcat), gctx, s.rms_eps)
        for l in range(s.n_layers):
            kv = _matvec(_f(W[f"layers.{l}.wk"]), c)
            vv = _matvec(_f(W[f"layers.{l}.wv"]), c)
            for h in range(s.n_kv_heads):
                seg = slice(h * s.head_dim, (h + 1) * s.head_dim)
                K[l][p, h] = _rope_complex(kv[seg], p, s.rope_theta)
                V[l][p, h] = vv[seg]
    return K, V


def naive_draft(shape, W: Dict[str, np.ndarray], hist_bits: np.ndarray, last_token: int, B: int):
    """Draft tokens d_1..d_{B-1} and their logits, recomputed per slot from the history.
    Returns (drafted [B-1], logits [B-1][V], residual trace [L+1][B][H])."""
    s = shape
    d, nq, nkv = s.head_dim, s.n_heads, s.n_kv_heads
    Kc, Vc = naive_context_kv(s, W, hist_bits)
    N = hist_bits.shape[1]
    E = W["embed"]
    xs: List[np.ndarray] = [_f(E[last_token])] + [_f(W["mask_emb"]) for _ in range(B - 1)]
    trace = [np.stack(xs)]
    for l in range(s.n_layers):
        P = lambda n: _f(W[f"layers.{l}.{n}"])
        Wq, Wk, Wv, Wo = P("wq"), P("wk"), P("wv"), P("wo")
        Wg, Wu, Wd = P("w_gate"), P("w_up"), P("w_down")
        ga, gm = P("g_attn"), P("g_mlp")
        qs, ks, vs = [], [], []
        for i in range(B):
            a = _rmsnorm(xs[i], ga, s.rms_eps)
            q, k, v = _matvec(Wq, a), _matvec(Wk, a), _matvec(Wv, a)
            qs.append([_rope_complex(q[h * d:(h + 1) * d], N + i, s.rope_theta) for h in range(nq)])
            ks.append([_rope_complex(k[h * d:(h + 1) * d], N + i, s.rope_theta) for h in range(nkv)])
            vs.append([v[h * d:(h + 1) * d] for h in range(nkv)])
        new_xs = []
        for i in range(B):
            o = np.zeros(nq * d)
            for h in range(nq):
                g = h * nkv // nq
                keys = [Kc[l][p, g] for p in range(N)] + [ks[j][g] for j in range(B)]
                vals = [Vc[l][p, g] for p in range(N)] + [vs[j][g] for j in range(B)]
                sc = [float(np.dot(qs[i][h], kk)) / math.sqrt(d) for kk in keys]
                mx = max(sc)
                ex = [math.exp(t - mx) for t in sc]
                tot = sum(ex)
                acc = np.zeros(d)
                for wgt, vv in zip(ex, vals):
                    acc = acc + (wgt / tot) * vv
                o[h * d:(h + 1) * d] = acc
            x = xs[i] + _matvec(Wo, o)
            a2 = _rmsnorm(x, gm, s.rms_eps)
            gate, up = _matvec(Wg, a2), _matvec(Wu, a2)
            act = np.array([_silu(gate[r]) * up[r] for r in range(len(gate))])
            new_xs.append(x + _matvec(Wd, act))
        xs = new_xs
        trace.append(np.stack(xs))
    gf = _f(W["g_final"])
    Wlm = _f(W["lm_head"])
    logits, drafted = [], []
    for i in range(1, B):
        z = _matvec(Wlm, _rmsnorm(xs[i], gf, s.rms_eps))
        best = 0
        for vtok in range(1, len(z)):
            if z[vtok] > z[best]:
                best = vtok
        logits.append(z)
        drafted.append(best)
    lg = np.stack(logits) if logits else np.zeros((0, Wlm.shape[0]))
    return np.array(drafted, dtype=np.int64), lg, np.stack(trace)


def naive_verify(target_logits: np.ndarray, drafted: Sequence[int]):
    """Largest tau in 1..B such that d_i equals the target's argmax g_{i-1} for all 1 <= i < tau.
    Returns (tau, committed g_0..g_{tau-1})."""
    T = np.asarray(target_logits, dtype=np.float64)
    B = T.shape[0]
    g = []
    for i in range(B):
        best = 0
        for v in range(1, T.shape[1]):
            if T[i, v] > T[i, best]:
                best = v
        g.append(best)
    tau = 1
    for cand in range(1, B + 1):
        if all(int(drafted[i - 1]) == g[i - 1] for i in range(1, cand)):
            tau = cand
    return tau, g[:tau]


def naive_verify_from_hidden(hidden_bits: np.ndarray, gain_bits: np.ndarray, lm_bits: np.ndarray,
                             drafted: Sequence[int], eps: float):
    """The target's greedy tokens from its last hidden states with scalar loops (norm, one
    dot product per vocabulary row, a running argmax that keeps the first maximum), then
    the try-every-tau acceptance. Returns (tau, committed, g)."""
    g_w = _f(gain_bits)
    W = _f(lm_bits)
    g = []
    for row in _f(hidden_bits):
        a = _rmsnorm(list(row), g_w, eps)
        best, arg = -math.inf, -1
        for v in range(W.shape[0]):
            z = float(np.dot(W[v], a))
            if z > best:
                best, arg = z, v
        g.append(arg)
    B = len(g)
    tau = 1
    for t in range(B, 0, -1):
        if all(int(drafted[i]) == g[i] for i in range(t - 1)):
            tau = t
            break
    return tau, g[:tau], g
