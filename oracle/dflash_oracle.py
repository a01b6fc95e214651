"""CPU oracle for the DFlash block-diffusion draft round.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link this module: it is used by tests/, by the smoke check in
__graft_entry__.py and by bench.py's cpu_baseline / reference legs, and by
nothing else.  It shares no code with the CUDA library.

What it computes, step by step, in float64 with plain numpy (one row at a
time, so every row's arithmetic is independent of how many rows share a
call):

  * committed / takePending / commitBlock / flush / propose / selectBlock:
    the drafter session state machine of ollama's ``mlxrunner/dflash.go``
    (gitea mirror; functions of the same names);
  * the context path aux_hidden_norms -> fc -> hidden_norm, then each
    layer's input_layernorm before a K/V-only projection (mlxcel PR #1771
    "add the Laguna DFlash drafter": summary and "Where the landed code and
    the issue text disagree");
  * the block forward over [anchor, mask x n] with the anchor row dropped
    before the unembedding ("Ollama DFlash block-diffusion draft model in
    mlxrunner", Facts; dflash.go propose/selectBlock);
  * sampling from one batched distribution (dflash.go selectBlock), done as
    Gumbel-max with a counter-based generator so that the CUDA side can draw
    the same token;
  * speculative verification: accepted prefix plus a bonus token, exact
    with respect to the target because it uses the actual proposal
    probabilities (dflash.go propose comment; DFlash2 commit note), as in
    Leviathan, Kalman & Matias (2023) and Chen et al. (2023).

Readings where the pages are silent:
  R1 norm gains are inputs (random 1 + N(0, 0.02) in tests);
  R3 eps = 1e-6;  R4 one RMSNorm per tap over that tap's slice;
  R5 per-head RMSNorm on q and k;  R6 rotate-half RoPE on pairs (j, j+d/2);
  R7 a query at position p sees a key at r iff p - r < W;
  R8 fused qkv rows are ordered q | k | v;  R9 one sigmoid gate per query
  head from g_proj;  R10 bidirectional attention inside the block unless the
  config says causal;  R11 block K/V never persist (rewound before any write);
  R13 full-vocabulary distributions unless the session sets a truncation;
  R24 truncation = top-k, softmax, top-p, min-p, each keeping a prefix of
  the (value desc, id asc) order, for draft and target rows alike;  R15 if the
  residual max(0, p - q) sums to zero, the bonus is drawn from p;
  R25 penalties are the sampler's repetition, presence and frequency
  penalties over a token history the caller supplies: an id seen c > 0
  times has a positive logit divided by the repetition penalty and a
  non-positive one multiplied by it, then loses the presence penalty once
  and the frequency penalty c times;  R26 every draft row sees the same
  committed history (no row of the block counts toward another's
  penalties), while target row r of verify sees that history plus the draft
  tokens d_1..d_r before it, the history classic decoding would have had;
  R27 (DFlash2) each layer's block-local dynamic convolution follows the
  attention residual: x = RMSNorm(h; conv_norm), per row i and channel group
  g (one group per query head) kernel weights softmax_j((W_dc x_i)[g, j])
  over conv_taps taps, and h_i += sum_j w_ij * x_{i-j} over the block's own
  rows (rows before the anchor count as zero);  R28 (DFlash2) the selector's
  candidates at position i are the sel_candidates largest logits of row i
  (value desc, id asc), scored l_i(c) + <A[prev], B[c]> with prev the token
  chosen at i - 1 (the anchor for i = 1) and A, B the [V, sel_rank] selector
  tables; the draw is Gumbel-max over the candidates at the request
  temperature only, and q_i = softmax(score / T) over them;  R29 (DFlash2)
  a proposal always drafts min(7, B_s - 1) tokens (dflash2Depth).

Storage rounding: for bf16 configs the values that the CUDA path stores in
bf16 are rounded to the nearest bf16 here too (u, c, the layer inputs fed to
matrix products, q, the cache K/V, the attention output, the residual h after
each add, the SwiGLU product, the final-norm output); fp32 configs round the
same points to fp32.  Everything between two storage points stays float64.

Parity pins: see tests/test_oracle_*.py.  Parity is unpinned only for the
architecture readings above (they are choices, not facts of the pages) and
for proposal probabilities of trained weights (none exist here).
"""
from __future__ import annotations

import numpy as np

PENDING_FLUSH_TOKENS = 256   # dflash.go: dflashPendingFlushTokens
DFLASH2_DEPTH = 7            # dflash.go: dflash2Depth, a DFlash2 session's fixed draft length


class ContextGap(Exception):
    """A committed run starts past the buffered frontier (dflash.go committed)."""


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def round_bf16(x) -> np.ndarray:
    """Nearest bf16 value (ties to even) of float64 input, returned as float64.

    bf16 keeps 8 significant bits, so 45 of float64's 53 are dropped.  Values
    are assumed to lie in bf16's normal range (true for every tensor here).
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    b = x.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    b = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    return b.view(np.float64)


def storage_round(dtype: str):
    if dtype == "bf16":
        return round_bf16
    if dtype == "f32":
        return lambda x: np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# Counter-based random numbers: Philox4x32-10
# Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
# SC'11.  Each round multiplies words 0 and 2 by two constants, keeps the
# 64-bit products' halves, and xors the high halves with words 1/3 and the
# key; the key is bumped by two Weyl constants between rounds.
# ---------------------------------------------------------------------------

_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = np.uint64(0x9E3779B9)
_PHILOX_W1 = np.uint64(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32 with 10 rounds; all arguments uint32-valued arrays."""
    c0, c1, c2, c3 = (np.asarray(v, dtype=np.uint64) & _MASK32 for v in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & _MASK32
    k1 = np.asarray(k1, dtype=np.uint64) & _MASK32
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(c0, c1, c2, c3, k0, k1)
    k0 = k0.copy(); k1 = k1.copy()
    for r in range(10):
        if r > 0:
            k0 = (k0 + _PHILOX_W0) & _MASK32
            k1 = (k1 + _PHILOX_W1) & _MASK32
        p0 = _PHILOX_M0 * c0          # < 2^64: no overflow in uint64
        p1 = _PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def random_u32(seed: int, rnd: int, stream: int, seq: int, row: int, v):
    """The random word for index v: word v mod 4 of Philox4x32-10 at counter
    (floor(v / 4), row | stream<<16, seq, round), key (low 32 bits of seed,
    high 32 bits of seed).  Each Philox output block of four words thus
    covers four consecutive indices."""
    seed = int(seed) & (2**64 - 1)
    u64 = lambda a: np.asarray(a, dtype=np.uint64)
    v = u64(v)
    ctr1 = (u64(row) & np.uint64(0xFFFF)) | ((u64(stream) & np.uint64(0xFFFF)) << np.uint64(16))
    words = philox4x32_10(v >> np.uint64(2), ctr1, u64(seq), u64(rnd), seed & 0xFFFFFFFF, seed >> 32)
    w = np.broadcast_to((v & np.uint64(3)).astype(np.int64), np.broadcast(*words).shape)
    return np.choose(w, words)


def uniform_open(x_u32) -> np.ndarray:
    """u = ((x >> 9) + 0.5) * 2^-23, strictly inside (0, 1) and exact in fp32."""
    x = np.asarray(x_u32, dtype=np.uint64) >> np.uint64(9)
    return (x.astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel(seed, rnd, stream, seq, row, v) -> np.ndarray:
    u = uniform_open(random_u32(seed, rnd, stream, seq, row, v))
    return -np.log(-np.log(u))


STREAM_DRAFT = 0    # Gumbel noise of the draft's token choice
STREAM_ACCEPT = 1   # acceptance uniforms of the verify
STREAM_BONUS = 2    # Gumbel noise of the bonus / residual draw


# ---------------------------------------------------------------------------
# Elementary steps
# ---------------------------------------------------------------------------

def rmsnorm(x, g, eps):
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope(x, pos, theta):
    """Rotate-half RoPE: pairs (j, j + d/2) turned by pos * theta^(-2j/d).

    x: [..., d]; pos: scalar or array broadcasting against x[..., 0].
    """
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def linear(w, x):
    """Rows of x times w^T, one matrix-vector product per row."""
    x = np.atleast_2d(x)
    return np.stack([w @ row for row in x]) if len(x) else np.zeros((0, w.shape[0]))


def silu(x):
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def logsumexp(s):
    m = np.max(s)
    return m + np.log(np.sum(np.exp(s - m)))


def softmax(s):
    e = np.exp(s - np.max(s))
    return e / np.sum(e)


# ---------------------------------------------------------------------------
# The draft model
# ---------------------------------------------------------------------------

class _Float64View:
    """Weights as given (exact storage values in any float array type), read
    as float64 when used; vectors are converted once, matrices per use so
    that a large draft never needs a full float64 copy."""

    def __init__(self, weights):
        self.src = dict(weights)
        self.small = {}

    def __getitem__(self, name):
        a = self.src[name]
        if a.ndim == 2 and a.size > (1 << 22):
            return np.asarray(a, dtype=np.float64)
        if name not in self.small:
            self.small[name] = np.asarray(a, dtype=np.float64)
        return self.small[name]

    def __contains__(self, name):
        return name in self.src

    def rows(self, name, idx):
        """Selected rows only (embedding lookup)."""
        return np.asarray(self.src[name][np.asarray(idx, dtype=np.int64)], dtype=np.float64)


class OracleDraft:
    """Draft weights in float64 plus the forward steps of the round.

    ``cfg`` needs the attributes of synthetic.DraftConfig; ``weights`` maps
    the tensor names of synthetic.weight_shapes to arrays holding exact
    storage values.
    """

    def __init__(self, cfg, weights):
        self.cfg = cfg
        self.w = _Float64View(weights)
        self.st = storage_round(cfg.dtype)
        self.group = cfg.n_q_heads // cfg.n_kv_heads

    # -- context path (Laguna PR: aux_hidden_norms + fc + hidden_norm, then
    #    each layer's input_layernorm before a K/V-only projection) ---------
    def context_hidden(self, feats):
        """c = hidden_norm(fc([aux_norm_k(f_k)]_k)) for rows of target features."""
        c = self.cfg
        f = np.asarray(feats, dtype=np.float64).reshape(-1, c.n_taps, c.target_hidden)
        u = self.st(rmsnorm(f, self.w["aux_norms"], c.rms_eps)).reshape(len(f), -1)
        return self.st(rmsnorm(linear(self.w["w_fc"], u), self.w["hidden_norm"], c.rms_eps))

    def context_layer_kv(self, l, hid, slots):
        """Layer l's K, V [rows, Hkv, d] of context rows (hidden `hid`) at slots:
        input_layernorm, the K/V rows of the fused projection, k norm, RoPE."""
        c = self.cfg
        p = f"layers.{l}."
        qd = c.n_q_heads * c.head_dim
        kd = c.n_kv_heads * c.head_dim
        x = self.st(rmsnorm(hid, self.w[p + "in_norm"], c.rms_eps))
        wkv = self.w[p + "w_qkv"][qd:qd + 2 * kd]       # K/V rows only
        kv = linear(wkv, x)
        k = kv[:, :kd].reshape(-1, c.n_kv_heads, c.head_dim)
        v = kv[:, kd:].reshape(-1, c.n_kv_heads, c.head_dim)
        slots = np.asarray(slots, dtype=np.float64)
        k = rope(rmsnorm(k, self.w[p + "k_norm"], c.rms_eps), slots[:, None], c.rope_theta)
        return self.st(k), self.st(v)

    def context_kv(self, feats, slots):
        """Per-layer K, V [rows, Hkv, d] of context rows at absolute slots."""
        hid = self.context_hidden(feats)
        Ks, Vs = [], []
        for l in range(self.cfg.n_layers):
            k, v = self.context_layer_kv(l, hid, slots)
            Ks.append(k)
            Vs.append(v)
        return Ks, Vs

    # -- block forward -----------------------------------------------------
    def visible(self, qpos, kpos, q_row, k_row):
        """Key visibility for one query: window limit (R7) and the in-block mask."""
        c = self.cfg
        ok = np.ones(np.shape(kpos), dtype=bool)
        if c.window:
            ok &= (qpos - np.asarray(kpos)) < c.window
        if k_row is not None and c.causal_block:
            ok &= np.asarray(k_row) <= q_row
        return ok

    def attention(self, q, k, v, pos, ck, cv, cpos):
        """softmax(q.k / sqrt(d)) . v for every block row and query head.

        Keys are the visible context rows followed by the visible block rows;
        query head hq reads KV head hq // (Hq / Hkv) (grouped-query attention).
        q [nb, Hq, d]; k, v [nb, Hkv, d]; ck, cv [N, Hkv, d]; pos [nb]; cpos [N].
        """
        c = self.cfg
        nb = len(q)
        scale = 1.0 / np.sqrt(c.head_dim)
        o = np.zeros((nb, c.n_q_heads, c.head_dim))
        for i in range(nb):
            cvis = self.visible(pos[i], cpos, i, None)
            bvis = self.visible(pos[i], pos, i, np.arange(nb))
            for hq in range(c.n_q_heads):
                hk = hq // self.group
                keys = np.concatenate([ck[cvis, hk, :], k[bvis, hk, :]])
                vals = np.concatenate([cv[cvis, hk, :], v[bvis, hk, :]])
                o[i, hq] = softmax((keys @ q[i, hq]) * scale) @ vals
        return o

    def dynamic_conv(self, l, h):
        """DFlash2's block-local dynamic convolution of layer l over the block
        rows h [nb, H] (R27); returns h plus the convolution."""
        c, st = self.cfg, self.st
        nb, H = h.shape
        G, kap = c.n_q_heads, c.conv_taps
        x = st(rmsnorm(h, self.w[f"layers.{l}.conv_norm"], c.rms_eps))
        a = linear(self.w[f"layers.{l}.w_dc"], x).reshape(nb, G, kap)
        wk = np.exp(a - a.max(axis=-1, keepdims=True))
        wk /= wk.sum(axis=-1, keepdims=True)
        gw = H // G
        out = np.zeros_like(h)
        for i in range(nb):
            for j in range(min(kap, i + 1)):
                out[i] += np.repeat(wk[i, :, j], gw) * x[i - j]
        return st(h + out)

    def block_layer(self, l, h, pos, ck, cv, cpos):
        """One draft layer over the block rows h [nb, H] at positions pos,
        against context K/V ck, cv [N, Hkv, d] at positions cpos."""
        c, w, st = self.cfg, self.w, self.st
        nb = len(h)
        qd = c.n_q_heads * c.head_dim
        kd = c.n_kv_heads * c.head_dim
        p = f"layers.{l}."
        x = st(rmsnorm(h, w[p + "in_norm"], c.rms_eps))
        qkv = linear(w[p + "w_qkv"], x)
        q = qkv[:, :qd].reshape(nb, c.n_q_heads, c.head_dim)
        k = qkv[:, qd:qd + kd].reshape(nb, c.n_kv_heads, c.head_dim)
        v = qkv[:, qd + kd:].reshape(nb, c.n_kv_heads, c.head_dim)
        q = st(rope(rmsnorm(q, w[p + "q_norm"], c.rms_eps), pos[:, None], c.rope_theta))
        k = st(rope(rmsnorm(k, w[p + "k_norm"], c.rms_eps), pos[:, None], c.rope_theta))
        v = st(v)
        gate = sigmoid(linear(w[p + "w_g"], x)) if c.gated_attention else None
        o = self.attention(q, k, v, pos, ck, cv, cpos)
        if gate is not None:
            o = o * gate[:, :, None]
        o = st(o.reshape(nb, qd))
        h = st(h + linear(w[p + "w_o"], o))
        if c.variant == "dflash2":
            h = self.dynamic_conv(l, h)
        y = st(rmsnorm(h, w[p + "post_norm"], c.rms_eps))
        a = st(silu(linear(w[p + "w_gate"], y)) * linear(w[p + "w_up"], y))
        return st(h + linear(w[p + "w_down"], a))

    def block_forward(self, tokens, F, ctx):
        """Forward of [anchor, mask x n] at positions F..F+n against context.

        ctx: dict with 'pos' [N] and per-layer 'k', 'v' lists of [N, Hkv, d].
        Returns the final residual h [n+1, H].
        """
        pos = F + np.arange(len(tokens), dtype=np.float64)
        h = self.w.rows("embed", [int(t) for t in tokens])
        cpos = np.asarray(ctx["pos"], dtype=np.float64)
        for l in range(self.cfg.n_layers):
            h = self.block_layer(l, h, pos, ctx["k"][l], ctx["v"][l], cpos)
        return h

    def select_block(self, logits, current, temperature, seed, rnd, seq):
        """DFlash2's candidate selector over rows 1..n (R28; dflash.go
        selectBlock, the BlockSelector branch): each position's token is
        drawn from its candidates conditioned on its predecessor.  Returns
        tokens [n], candidate ids [n, k], their probabilities [n, k] (one-hot
        on the token at T = 0) and q(token) [n]."""
        c = self.cfg
        logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
        n, V = logits.shape
        k = min(c.sel_candidates, V)
        A, B = self.w["sel_prev"], self.w["sel_next"]
        toks = np.zeros(n, dtype=np.int64)
        ids = np.zeros((n, k), dtype=np.int64)
        probs = np.zeros((n, k))
        prev = int(current)
        for i in range(n):
            row = logits[i]
            cand = np.lexsort((np.arange(V), -row))[:k]
            score = row[cand] + B[cand] @ A[prev]
            if temperature == 0:
                j = int(np.argmax(score))
                probs[i, j] = 1.0
            else:
                z = score / temperature + gumbel(seed, rnd, STREAM_DRAFT, seq, i + 1, cand)
                j = int(np.argmax(z))
                probs[i] = softmax(score / temperature)
            ids[i] = cand
            toks[i] = prev = int(cand[j])
        return toks, ids, probs, probs[np.arange(n), np.argmax(ids == toks[:, None], axis=1)]

    def unembed(self, h_rows, lo=0, hi=None):
        """Raw draft logits of block rows (final norm, then the unembedding);
        lo/hi select a slice of the vocabulary."""
        z = self.st(rmsnorm(h_rows, self.w["final_norm"], self.cfg.rms_eps))
        U = self.w.src["unembed"]
        return linear(np.asarray(U[lo:hi], dtype=np.float64), z)


# ---------------------------------------------------------------------------
# Sampling and verification
# ---------------------------------------------------------------------------

def truncated_support(s, top_k=0, top_p=1.0, min_p=0.0):
    """The ids a truncating sampler keeps for one row of scaled scores s = l/T.

    dflash.go selectBlock draws from the sampler's Distribution, whose IDs
    are the kept tokens.  The truncation (reading R24): order the row by
    value, descending, then by id; keep the first top_k (0: all); take the
    softmax over what is kept; keep an entry while the probability mass
    strictly before it is below top_p; keep entries whose probability is at
    least min_p times the largest.  Every step keeps a prefix of the order,
    so the result is a prefix too.  NaN scores are never kept.
    Returns the kept ids in that order.
    """
    s = np.asarray(s, dtype=np.float64)
    ids = np.arange(len(s))
    ok = ~np.isnan(s)
    order = ids[ok][np.lexsort((ids[ok], -s[ok]))]
    if top_k:
        order = order[:top_k]
    e = np.exp(s[order] - s[order[0]])
    p = e / e.sum()
    keep = len(order)
    if top_p < 1.0:
        before = np.cumsum(p) - p
        keep = min(keep, int(np.count_nonzero(before < top_p)))
    if min_p > 0.0:
        keep = min(keep, int(np.count_nonzero(p >= min_p * p[0])))
    return order[:keep]


def truncation_active(trunc) -> bool:
    return trunc is not None and (trunc[0] > 0 or trunc[1] < 1.0 or trunc[2] > 0.0)


def apply_penalties(logits_row, history, repeat=1.0, presence=0.0, frequency=0.0):
    """One row of logits after the sampler's penalties over `history` (R25).

    For every id that occurs c > 0 times in the history: a positive logit is
    divided by `repeat` and a non-positive one multiplied by it; then
    `presence` is subtracted once and `frequency` c times.  Ids that do not
    occur are unchanged.  ("Ollama DFlash block-diffusion draft model in
    mlxrunner", Facts: penalties see only committed history, not other rows
    of the block; dflash.go selectBlock.)
    """
    out = np.array(logits_row, dtype=np.float64)
    ids, counts = np.unique(np.asarray(history, dtype=np.int64), return_counts=True)
    for v, c in zip(ids, counts):
        x = out[v]
        x = x / repeat if x > 0 else x * repeat
        out[v] = x - presence - frequency * float(c)
    return out


def penalties_active(pen) -> bool:
    return pen is not None and (pen[0] != 1.0 or pen[1] != 0.0 or pen[2] != 0.0)


def penalized(logits_row, pen, extra=()):
    """The row after the penalties `pen` = (repeat, presence, frequency,
    history), with `extra` tokens appended to the history; unchanged when no
    penalty is active."""
    if not penalties_active(pen):
        return np.asarray(logits_row, dtype=np.float64)
    return apply_penalties(logits_row, list(pen[3]) + [int(t) for t in extra], *pen[:3])


def sample_rows(logits, temperature, seed, rnd, seq, trunc=None):
    """One batched draw for rows 1..n of a block (dflash.go selectBlock).

    T == 0: argmax (lowest index on ties), q(token) = 1.
    T > 0: token = argmax_v(l_v/T + Gumbel_v), which is an exact draw from
    softmax(l/T); q(token) = exp(l_token/T - logsumexp(l/T)).
    trunc = (top_k, top_p, min_p) at T > 0: the same draw over the kept ids
    only (truncated_support), with the log-sum-exp over them; T == 0 is
    unchanged (the best id is always kept).
    Returns tokens [n], q(token) [n], lse [n] (nan when T == 0).
    """
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    n, V = logits.shape
    toks = np.zeros(n, dtype=np.int64)
    qtok = np.ones(n)
    lse = np.full(n, np.nan)
    for i in range(n):
        if temperature == 0:
            toks[i] = int(np.argmax(logits[i]))
            continue
        s = logits[i] / temperature
        g = gumbel(seed, rnd, STREAM_DRAFT, seq, i + 1, np.arange(V))
        if truncation_active(trunc):
            kept = truncated_support(s, *trunc)
            lse[i] = logsumexp(s[kept])
            score = np.full(V, -np.inf)
            score[kept] = s[kept] + g[kept]
        else:
            lse[i] = logsumexp(s)
            score = s + g
        toks[i] = int(np.argmax(score))
        qtok[i] = np.exp(s[toks[i]] - lse[i])
    return toks, qtok, lse


def sampler_distribution(logits_row, temperature, trunc=None):
    """softmax(l/T), restricted to the kept ids and renormalised when trunc is active."""
    s = np.asarray(logits_row, dtype=np.float64) / temperature
    if not truncation_active(trunc):
        return softmax(s)
    kept = truncated_support(s, *trunc)
    p = np.zeros(len(s))
    p[kept] = softmax(s[kept])
    return p


def proposal_distribution(draft_logits_row, draft_temperature, proposed_token, trunc=None, cands=None):
    """q of one block row: the sampler's distribution at T > 0, one-hot of the
    proposal at T == 0; cands = (ids, probs): a DFlash2 candidate distribution."""
    if cands is not None and draft_temperature > 0:
        q = np.zeros(len(draft_logits_row))
        q[np.asarray(cands[0], dtype=np.int64)] = cands[1]
        return q
    if draft_temperature == 0:
        q = np.zeros(len(draft_logits_row))
        q[int(proposed_token)] = 1.0
        return q
    return sampler_distribution(draft_logits_row, draft_temperature, trunc)


def verify(target_logits, draft_tokens, draft_logits, proposed_tokens, draft_temperature,
           temperature, seed, rnd, seq, trunc=None, draft_trunc=None, penalties=None, draft_cands=None):
    """Accepted prefix length a and bonus token b.

    target_logits [n+1, V]: row r scores the token after [current, d_1..d_r].
    draft_tokens [n]: the tokens under test (normally the proposal).
    draft_logits [n, V], proposed_tokens [n], draft_temperature: what the last
    propose drew from; q_i is that distribution.

    T == 0: accept while argmax(target row i-1) == d_i; b = argmax(row a).
    T > 0: accept d_i iff r_i * q_i(d_i) < p_i(d_i) (that is r_i < p/q), with
    p_i = softmax(target row i-1 / T); at the first rejection draw b from
    max(0, p_i - q_i) (from p_i if that is all zero, R15); if all n pass,
    draw b from p of row n.
    trunc: the sampler's truncation of the target rows (p is the truncated,
    renormalised distribution); draft_trunc: the one the proposal was drawn
    with (q likewise).  The rule is unchanged, so the emitted tokens follow
    the truncated target distribution.
    penalties = (repeat, presence, frequency, history): target row r is
    penalised over the history plus d_1..d_r (R26); draft_logits are the
    logits the proposal was drawn from, its penalties already applied.
    draft_cands = (ids [n, k], probs [n, k]): DFlash2's per-position candidate
    distributions, which are q (the DFlash2 commit note: verification uses
    each position's candidate distribution to keep the output exact).
    """
    tl = np.atleast_2d(np.asarray(target_logits, dtype=np.float64))
    if penalties_active(penalties):
        tl = np.stack([penalized(tl[r], penalties, draft_tokens[:r]) for r in range(len(tl))])
    n = len(draft_tokens)
    V = tl.shape[1]
    if temperature == 0:
        a = 0
        while a < n and int(np.argmax(tl[a])) == int(draft_tokens[a]):
            a += 1
        return a, int(np.argmax(tl[a]))
    for i in range(1, n + 1):
        p = sampler_distribution(tl[i - 1], temperature, trunc)
        q = proposal_distribution(draft_logits[i - 1], draft_temperature, proposed_tokens[i - 1], draft_trunc,
                                  None if draft_cands is None else (draft_cands[0][i - 1], draft_cands[1][i - 1]))
        d = int(draft_tokens[i - 1])
        r = uniform_open(random_u32(seed, rnd, STREAM_ACCEPT, seq, i, 0))
        if r * q[d] < p[d]:
            continue
        res = np.maximum(p - q, 0.0)
        if not np.sum(res) > 0:
            res = p
        with np.errstate(divide="ignore"):
            score = np.log(res) + gumbel(seed, rnd, STREAM_BONUS, seq, i, np.arange(V))
        return i - 1, int(np.argmax(score))
    p = sampler_distribution(tl[n], temperature, trunc)
    with np.errstate(divide="ignore"):
        score = np.log(p) + gumbel(seed, rnd, STREAM_BONUS, seq, n + 1, np.arange(V))
    return n, int(np.argmax(score))


# ---------------------------------------------------------------------------
# The drafter session (dflash.go: open / committed / takePending /
# commitBlock / flush / propose / selectBlock)
# ---------------------------------------------------------------------------

class OracleSession:
    """One request's drafting state.

    F (ctxOffset) is the slot after the last feature row written to the
    cache; P rows are buffered past it, so F + P is the slot after the last
    reported token.  The cache maps slot -> (K [L,Hkv,d], V [L,Hkv,d]).
    """

    def __init__(self, draft: OracleDraft, restored_offset: int = 0, seq: int = 0,
                 restored_cache=None):
        self.draft = draft
        self.cfg = draft.cfg
        self.F = int(restored_offset)
        self.pending = []
        self.P = 0
        self.block_outstanding = False
        self.block_kv = None           # the outstanding block's K/V (never persisted)
        self.cache = dict(restored_cache or {})
        self.seq = seq
        self.last = None               # what the last propose drew from
        self.sampler = None            # (top_k, top_p, min_p) truncation, None: full distributions
        self.penalties = None          # (repeat, presence, frequency, history), None: no penalties
        self.stats = dict(rounds=0, proposed=0, accepted=0)

    def set_penalties(self, repeat: float = 1.0, presence: float = 0.0, frequency: float = 0.0, history=()):
        """The sampler's penalties and the committed token history they count."""
        self.penalties = (float(repeat), float(presence), float(frequency), tuple(int(t) for t in history))

    def set_sampler(self, top_k: int = 0, top_p: float = 1.0, min_p: float = 0.0):
        """The session's truncation, used for its draft rows and its target rows."""
        self.sampler = (int(top_k), float(top_p), float(min_p))

    # dflash.go draftLimit
    @property
    def draft_limit(self) -> int:
        return self.cfg.block_size - 1

    def committed(self, features, position: int):
        """Append the rows of a committed run that the session does not hold yet."""
        features = np.atleast_2d(features)
        n = len(features)
        start = self.F + self.P - int(position)
        if start < 0:
            raise ContextGap(f"committed run at {position} leaves a context gap at {self.F + self.P}")
        if start < n:
            self.pending.append(np.asarray(features[start:n]))
            self.P += n - start
            if self.P >= PENDING_FLUSH_TOKENS:
                self.flush()

    def take_pending(self):
        if not self.pending:
            return None, self.F
        rows = np.concatenate(self.pending)
        first = self.F
        self.pending = []
        self.F += self.P
        self.P = 0
        return rows, first

    def commit_block(self):
        """Rewind the outstanding block: the cache keeps only context rows."""
        if not self.block_outstanding:
            return
        self.block_kv = None
        self.block_outstanding = False

    def _write_context(self, rows, first):
        """Context-only forward of rows at slots first.. (drops rows no future
        query can see when the draft has a window: Laguna PR, window drop)."""
        if rows is None or len(rows) == 0:
            return
        slots = first + np.arange(len(rows))
        if self.cfg.window:
            keep = slots > self.F - self.cfg.window
            rows, slots = rows[keep], slots[keep]
            for s in [s for s in self.cache if s <= self.F - self.cfg.window]:
                del self.cache[s]
            if len(rows) == 0:
                return
        Ks, Vs = self.draft.context_kv(rows, slots)
        for j, s in enumerate(slots):
            self.cache[int(s)] = (np.stack([K[j] for K in Ks]), np.stack([V[j] for V in Vs]))

    def flush(self):
        self.commit_block()
        if not self.pending:
            return
        rows, first = self.take_pending()
        self._write_context(rows, first)

    def context(self):
        """Cached context rows below F as arrays for the attention."""
        c = self.cfg
        slots = sorted(s for s in self.cache if s < self.F)
        L = c.n_layers
        if not slots:
            z = np.zeros((0, c.n_kv_heads, c.head_dim))
            return dict(pos=np.zeros(0), k=[z] * L, v=[z] * L)
        K = np.stack([self.cache[s][0] for s in slots])   # [N, L, Hkv, d]
        V = np.stack([self.cache[s][1] for s in slots])
        return dict(pos=np.asarray(slots, dtype=np.float64),
                    k=[K[:, l] for l in range(L)], v=[V[:, l] for l in range(L)])

    def propose(self, current: int, max_tokens: int, temperature: float = 0.0,
                seed: int = 0, rnd: int = 0):
        """Draft n = min(max_tokens, B_s - 1) tokens after `current`.

        Returns None (the pages' nil) when n <= 0 or nothing has been
        committed; otherwise dict(tokens, q, logits, lse, hidden).
        """
        c = self.cfg
        n = min(int(max_tokens), c.block_size - 1)
        if n <= 0 or self.F + self.P == 0:
            return None
        if c.variant == "dflash2":
            n = min(DFLASH2_DEPTH, c.block_size - 1)      # the fixed depth overrides max_tokens (R29)
        self.commit_block()
        rows, first = self.take_pending()
        self._write_context(rows, first)
        self.block_outstanding = True
        tokens = [int(current)] + [c.mask_token] * n
        h = self.draft.block_forward(tokens, self.F, self.context())
        logits = self.draft.unembed(h[1:])          # the anchor row is unused
        if c.variant == "dflash2":
            # the selector draws at the request temperature only (DFlash2 note)
            toks, ids, probs, q = self.draft.select_block(logits, current, temperature, seed, rnd, self.seq)
            lse = np.full(n, np.nan)
            self.last = dict(tokens=toks, logits=logits, temperature=temperature, trunc=None, cands=(ids, probs))
            self.stats["rounds"] += 1
            self.stats["proposed"] += n
            return dict(tokens=toks, q=q, logits=logits, lse=lse, hidden=h, n=n, cand_ids=ids, cand_probs=probs)
        # every row sees the same committed history (R26)
        logits = np.stack([penalized(row, self.penalties) for row in logits])
        toks, q, lse = sample_rows(logits, temperature, seed, rnd, self.seq, self.sampler)
        self.last = dict(tokens=toks, logits=logits, temperature=temperature, trunc=self.sampler, cands=None)
        self.stats["rounds"] += 1
        self.stats["proposed"] += n
        return dict(tokens=toks, q=q, logits=logits, lse=lse, hidden=h, n=n)

    def verify(self, target_logits, draft_tokens, temperature, seed=0, rnd=0):
        if self.last is None:
            raise RuntimeError("verify without a proposal")
        a, b = verify(target_logits, draft_tokens, self.last["logits"], self.last["tokens"],
                      self.last["temperature"], temperature, seed, rnd, self.seq, self.sampler,
                      self.last["trunc"], self.penalties, self.last["cands"])
        self.stats["accepted"] += a
        return a, b

    def close(self):
        self.flush()
