"""A small synthetic target model that drives speculative rounds in tests.

The pages run the draft against a real target (Qwen 3.5, Laguna); no target
checkpoint exists here, so a random-init 2-layer decoder stands in for it:
hidden 256, 4 heads of 64 (MHA), SwiGLU 512, vocabulary 32, causal, RoPE with
theta 1e6, its own seed.  It produces what a DFlash draft consumes: five
hidden taps per position (embedding output, then the residual stream after
each attention and each MLP of its two layers) and raw next-token logits.

Every position is computed on its own (one row at a time against the cached
K/V of earlier rows), so a multi-row verify forward gives exactly the same
logits and taps as token-by-token decoding.  This is the block-versus-chain
exactness that the Laguna PR's probe measures on real kernels; here it holds
by construction, which makes greedy speculative output comparable token for
token with plain greedy decoding.

This is an input generator for tests; it is not part of the draft round.
"""
from __future__ import annotations

import numpy as np

from . import normal

__all__ = ["SyntheticTarget"]


class SyntheticTarget:
    def __init__(self, seed: int = 1, hidden: int = 256, n_heads: int = 4,
                 head_dim: int = 64, intermediate: int = 512, vocab: int = 32,
                 n_layers: int = 2, theta: float = 1e6, eps: float = 1e-6,
                 logit_scale: float = 8.0):
        self.H, self.nh, self.d, self.I, self.V = hidden, n_heads, head_dim, intermediate, vocab
        self.L, self.theta, self.eps = n_layers, theta, eps
        f64 = lambda name, shape, std=0.02, mean=0.0: normal(seed, "target." + name, shape, std=std, mean=mean).astype(np.float64)
        self.E = f64("embed", (vocab, hidden), std=1.0)
        # a wider unembedding makes greedy choices well separated
        self.U = f64("unembed", (vocab, hidden), std=0.02 * logit_scale)
        self.nf = f64("final_norm", (hidden,), mean=1.0)
        self.layers = []
        for l in range(n_layers):
            p = f"layers.{l}."
            self.layers.append(dict(
                n1=f64(p + "n1", (hidden,), mean=1.0),
                wq=f64(p + "wq", (n_heads * head_dim, hidden)),
                wk=f64(p + "wk", (n_heads * head_dim, hidden)),
                wv=f64(p + "wv", (n_heads * head_dim, hidden)),
                wo=f64(p + "wo", (hidden, n_heads * head_dim)),
                n2=f64(p + "n2", (hidden,), mean=1.0),
                wg=f64(p + "wg", (intermediate, hidden)),
                wu=f64(p + "wu", (intermediate, hidden)),
                wd=f64(p + "wd", (hidden, intermediate)),
            ))
        self.k_cache = [[] for _ in range(n_layers)]  # per layer: list of [nh, d]
        self.v_cache = [[] for _ in range(n_layers)]

    @property
    def n_taps(self) -> int:
        return 2 * self.L + 1

    @property
    def length(self) -> int:
        return len(self.k_cache[0])

    def _norm(self, x, g):
        return x / np.sqrt(np.mean(x * x) + self.eps) * g

    def _rope(self, x, pos):
        half = self.d // 2
        inv = self.theta ** (-np.arange(half, dtype=np.float64) * 2.0 / self.d)
        ang = pos * inv
        c, s = np.cos(ang), np.sin(ang)
        a, b = x[..., :half], x[..., half:]
        return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)

    def _step(self, token: int, pos: int):
        """One position: returns (fp32 logits [V], fp32 taps [5*H]) and caches K/V."""
        x = self.E[token].copy()
        taps = [x.copy()]
        for l, w in enumerate(self.layers):
            y = self._norm(x, w["n1"])
            q = self._rope((w["wq"] @ y).reshape(self.nh, self.d), pos)
            k = self._rope((w["wk"] @ y).reshape(self.nh, self.d), pos)
            v = (w["wv"] @ y).reshape(self.nh, self.d)
            self.k_cache[l].append(k)
            self.v_cache[l].append(v)
            K = np.stack(self.k_cache[l])  # [pos+1, nh, d]
            Vv = np.stack(self.v_cache[l])
            o = np.empty((self.nh, self.d))
            for h in range(self.nh):
                s = K[:, h, :] @ q[h] / np.sqrt(self.d)
                p = np.exp(s - s.max())
                p /= p.sum()
                o[h] = p @ Vv[:, h, :]
            x = x + w["wo"] @ o.reshape(-1)
            taps.append(x.copy())
            y = self._norm(x, w["n2"])
            g = w["wg"] @ y
            x = x + w["wd"] @ (g / (1.0 + np.exp(-g)) * (w["wu"] @ y))
            taps.append(x.copy())
        logits = self.U @ self._norm(x, self.nf)
        return logits.astype(np.float32), np.concatenate(taps).astype(np.float32)

    def forward(self, tokens, start: int):
        """Rows for tokens at positions start.. (K/V appended): logits [n,V], taps [n,5H]."""
        if start != self.length:
            raise ValueError(f"target forward at {start} but cache holds {self.length}")
        outs = [self._step(int(t), start + i) for i, t in enumerate(tokens)]
        return np.stack([o[0] for o in outs]), np.stack([o[1] for o in outs])

    def trim(self, length: int):
        """Roll the cache back to `length` rows (rejected verify rows)."""
        for l in range(self.L):
            del self.k_cache[l][length:]
            del self.v_cache[l][length:]

    def reset(self):
        self.trim(0)

    def greedy_decode(self, prompt, n_new: int):
        """Plain greedy decoding: the reference a speculative run must equal."""
        self.reset()
        logits, _ = self.forward(prompt, 0)
        out = []
        tok = int(np.argmax(logits[-1]))
        pos = len(prompt)
        while len(out) < n_new:
            out.append(tok)
            logits, _ = self.forward([tok], pos)
            pos += 1
            tok = int(np.argmax(logits[-1]))
        self.reset()
        return out
