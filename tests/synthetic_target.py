"""A small synthetic autoregressive target for end-to-end tests: a pre-norm causal
transformer (RoPE, SwiGLU, final RMSNorm, LM head) with seeded random weights, computed in
float64 with an incremental KV cache. It exposes the target interface of the generation
loop (prefill, forward_block, truncate) and returns the hidden states after its tapped
layers. Its LM head may carry a bias toward one token, so that its greedy output contains
runs of that token. Test infrastructure only: it stands in for the trained target model
the pages use, which is not available here."""
from __future__ import annotations

import math

import torch


class TinyTarget:
    def __init__(self, vocab, hidden, n_layers=4, taps=(1, 2, 3), n_heads=4, head_dim=64, inter=512,
                 theta=1e6, eps=1e-6, seed=0, bias_token=None, bias=0.0, max_len=2048, device="cuda"):
        g = torch.Generator(device="cpu").manual_seed(seed)
        f64 = dict(dtype=torch.float64)
        r = lambda *s: (0.02 * torch.randn(*s, generator=g, **f64)).to(device)
        self.V, self.H, self.L, self.taps = vocab, hidden, n_layers, tuple(taps)
        self.nh, self.hd, self.theta, self.eps = n_heads, head_dim, theta, eps
        self.E = (torch.randn(vocab, hidden, generator=g, **f64)).to(device)
        self.layers = [dict(wq=r(n_heads * head_dim, hidden), wk=r(n_heads * head_dim, hidden),
                            wv=r(n_heads * head_dim, hidden), wo=r(hidden, n_heads * head_dim),
                            wg=r(inter, hidden), wu=r(inter, hidden), wd=r(hidden, inter),
                            g1=torch.ones(hidden, device=device, **f64), g2=torch.ones(hidden, device=device, **f64))
                       for _ in range(n_layers)]
        self.gf = torch.ones(hidden, device=device, **f64)
        self.lm = r(vocab, hidden) * 5.0
        self.bias = torch.zeros(vocab, device=device, **f64)
        if bias_token is not None:
            self.bias[bias_token] = bias
        self.k = torch.zeros(n_layers, max_len, n_heads, head_dim, device=device, **f64)
        self.v = torch.zeros_like(self.k)
        self.n = 0
        self.device = device

    def _rms(self, x, gain):
        return x / torch.sqrt((x * x).mean(-1, keepdim=True) + self.eps) * gain

    def _rope(self, x, pos):
        d = x.shape[-1]
        h = d // 2
        inv = self.theta ** (-2.0 * torch.arange(h, device=x.device, dtype=torch.float64) / d)
        ang = pos[:, None].to(torch.float64) * inv[None, :]
        c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
        x1, x2 = x[..., :h], x[..., h:]
        return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)

    def _forward(self, tokens):
        n, p0 = tokens.numel(), self.n
        pos = torch.arange(p0, p0 + n, device=self.device)
        x = self.E[tokens]
        tapped = []
        for li, W in enumerate(self.layers):
            a = self._rms(x, W["g1"])
            q = self._rope((a @ W["wq"].T).view(n, self.nh, self.hd), pos)
            k = self._rope((a @ W["wk"].T).view(n, self.nh, self.hd), pos)
            self.k[li, p0:p0 + n] = k
            self.v[li, p0:p0 + n] = (a @ W["wv"].T).view(n, self.nh, self.hd)
            K, Vv = self.k[li, : p0 + n], self.v[li, : p0 + n]
            s = torch.einsum("nhd,mhd->hnm", q, K) / math.sqrt(self.hd)
            causal = torch.arange(p0 + n, device=self.device)[None, :] > pos[:, None]
            s = s.masked_fill(causal[None], float("-inf"))
            o = torch.einsum("hnm,mhd->nhd", torch.softmax(s, dim=-1), Vv).reshape(n, -1)
            x = x + o @ W["wo"].T
            a2 = self._rms(x, W["g2"])
            x = x + (torch.nn.functional.silu(a2 @ W["wg"].T) * (a2 @ W["wu"].T)) @ W["wd"].T
            if li + 1 in self.taps:
                tapped.append(x)
        self.n = p0 + n
        logits = self._rms(x, self.gf) @ self.lm.T + self.bias
        return torch.stack(tapped).to(torch.bfloat16), logits.to(torch.float32)

    def prefill(self, input_ids):
        self.n = 0
        tapped, logits = self._forward(input_ids.to(self.device))
        return tapped, logits[-1]

    def forward_block(self, tokens):
        return self._forward(tokens.to(self.device))

    def truncate(self, length):
        self.n = length


def greedy_reference(target, input_ids, n_new, stop_token_ids=()):
    """Plain autoregressive greedy decoding of the target, one token at a time."""
    _, logits = target.prefill(input_ids)
    out = [int(torch.argmax(logits))]
    while len(out) < n_new and out[-1] not in stop_token_ids:
        _, logits = target.forward_block(torch.tensor([out[-1]], device=target.device))
        out.append(int(torch.argmax(logits[-1])))
    return out
