"""CPU oracle for the target's side of a speculative round.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link this module: it is used by tests/ (and may be used by the smoke check
and bench.py's CPU legs), and by nothing else.  It shares no code with the
CUDA library.

Two things are here, in float64 numpy:

  * ``OracleTarget``: the verify forward of a small dense target with tap
    capture and rollback trim.  The mlxcel Laguna PR ("add the Laguna DFlash
    drafter": summary, the temporal-context and review commits) runs the
    target's verify forward over [current, d_1..d_n], captures five hidden
    states of every row for the drafter and trims the target caches back to
    the accepted rows afterwards.  No target checkpoint exists here, so the
    target is a random-init decoder: RMSNorm, rotate-half RoPE, causal
    multi-head attention over its cache, SwiGLU MLP, final norm and
    unembedding.  The taps are the embedding output and the residual stream
    after each attention and each MLP (2 L + 1 of them).  Every position is
    computed on its own against the cached K/V of earlier positions, so a
    multi-row forward equals token-by-token decoding by construction.

  * ``exactness_rows`` / ``exactness_summary``: the PR's block-versus-chain
    probe (the real-checkpoint probe commit and the report commits): per row,
    the number of logit bytes that differ between a multi-row verify block and
    single-token decode, and the top-2 logits of both arms; the gate allows
    the pairing when no byte differs at the first verify position.  Logits are
    fp32 here and bytes are counted over their fp32 encodings.

Pins (tests/test_oracle_target.py): the forward against an independent torch
float64 build of the same decoder (torch's RMSNorm and scaled-dot-product
attention with a causal mask), RoPE at position 0 is the identity, a single
position attends only to itself (attention output = v); the probe against
IEEE-754 byte counts worked by hand and a brute-force sort for the top two.
"""
from __future__ import annotations

import numpy as np

__all__ = ["OracleTarget", "exactness_rows", "exactness_summary"]


class OracleTarget:
    def __init__(self, weights: dict, shape):
        self.w, self.shape = weights, shape
        self.H, self.nh, self.d = shape.hidden, shape.n_heads, shape.head_dim
        self.V, self.L = shape.vocab, shape.n_layers
        self.theta, self.eps = shape.rope_theta, shape.rms_eps
        self.k_cache = [[] for _ in range(self.L)]  # per layer: one [nh, d] per position
        self.v_cache = [[] for _ in range(self.L)]

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
        """One position: (logits [V], taps [(2L+1) H]) as fp32; caches its K/V."""
        x = self.w["embed"][token].copy()
        taps = [x.copy()]
        for l, w in enumerate(self.w["layers"]):
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
        logits = self.w["unembed"] @ self._norm(x, self.w["final_norm"])
        return logits.astype(np.float32), np.concatenate(taps).astype(np.float32)

    def forward(self, tokens, start: int):
        """Rows for tokens at positions start.. (K/V appended): logits [n,V], taps [n,(2L+1)H]."""
        if start != self.length:
            raise ValueError(f"target forward at {start} but cache holds {self.length}")
        outs = [self._step(int(t), start + i) for i, t in enumerate(tokens)]
        return np.stack([o[0] for o in outs]), np.stack([o[1] for o in outs])

    def trim(self, length: int):
        """Roll the cache back to `length` rows (rejected verify rows)."""
        if not 0 <= length <= self.length:
            raise ValueError("trim length outside [0, cached]")
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


def _top2(row):
    """The two best entries by value (descending), then id (ascending); NaN never chosen."""
    ids = [i for i in range(len(row)) if not np.isnan(row[i])]
    ids.sort(key=lambda i: (-float(row[i]), i))
    best = ids[:2] + [None] * (2 - len(ids[:2]))
    return best


def exactness_rows(block, chain):
    """Per row of two fp32 logit arrays [rows, V]: differing bytes of the
    fp32 encodings, and both arms' top two (ids and values)."""
    block = np.ascontiguousarray(block, dtype=np.float32)
    chain = np.ascontiguousarray(chain, dtype=np.float32)
    assert block.shape == chain.shape and block.ndim == 2
    out = []
    for b, c in zip(block, chain):
        diff = int(np.count_nonzero(b.view(np.uint8) != c.view(np.uint8)))
        tb, tc = _top2(b), _top2(c)
        out.append(dict(differing_bytes=diff, block_top=tb, chain_top=tc,
                        block_val=[None if i is None else float(b[i]) for i in tb],
                        chain_val=[None if i is None else float(c[i]) for i in tc]))
    return out


def exactness_summary(rows):
    """The gate: it allows the pairing when no logit byte differs at the
    first verify position; disagreements counts rows whose argmax differs."""
    return dict(rows=len(rows), differing_bytes=sum(r["differing_bytes"] for r in rows),
                first_row_differing_bytes=rows[0]["differing_bytes"],
                disagreements=sum(r["block_top"][0] != r["chain_top"][0] for r in rows),
                allows=int(rows[0]["differing_bytes"] == 0))
