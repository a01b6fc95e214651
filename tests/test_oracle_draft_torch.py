"""Pin of the draft oracle (oracle/dflash_oracle.py) against an independent
torch float64 build of the same round.

The build below shares nothing with the oracle but the seeded inputs.  It
takes torch's own RMSNorm (F.rms_norm), RoPE as a complex rotation of the
pairs (x_j, x_{j+d/2}), torch's scaled_dot_product_attention with an explicit
visibility mask over [context | block] and the KV heads repeated for grouped
queries, F.silu and F.linear, and a storage rounding written with frexp /
ldexp (bf16: 8 significant bits, ties to even) instead of the oracle's bit
manipulation.  It covers the whole path the pages give:
  * the context path: aux_hidden_norms per tap, fc, hidden_norm, then each
    layer's input_layernorm before the K/V rows of the fused projection, the
    k norm and RoPE at the slot (mlxcel PR #1771, summary, and the note on
    where the landed code and the issue text disagree);
  * the block layer: fused q | k | v (+ g_proj), per-head q/k norms, RoPE,
    attention, the per-head sigmoid gate, the O residual, post-norm, SwiGLU
    and the down residual;
  * final_norm and the unembedding of rows 1..n, the anchor row dropped
    ("Ollama DFlash block-diffusion draft model in mlxrunner", Facts).
Planted mistakes in the oracle (a dropped gain, SiLU on the wrong half, a
missing gate) must make the comparison fail, which shows the pin has teeth.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synthetic as S
from oracle import dflash_oracle as O


def _store(cfg):
    """Storage rounding of the build: fp32 by cast, bf16 by keeping 8
    significant bits of the frexp mantissa (ties to even)."""
    if cfg.dtype == "f32":
        return lambda x: x.to(torch.float32).to(torch.float64)

    def bf16(x):
        m, e = torch.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
        return torch.ldexp(torch.round(m * 256.0) / 256.0, e)
    return bf16


class TorchDraft:
    def __init__(self, cfg, w):
        self.cfg = cfg
        self.w = {k: torch.from_numpy(np.asarray(v, dtype=np.float64)) for k, v in w.items()}
        self.st = _store(cfg)

    def _norm(self, x, g):
        return F.rms_norm(x, (x.shape[-1],), weight=g, eps=self.cfg.rms_eps)

    def _rope(self, x, pos):
        """x [rows, heads, d] at absolute positions pos [rows]."""
        d = x.shape[-1]
        half = d // 2
        freq = self.cfg.rope_theta ** (-torch.arange(half, dtype=torch.float64) * 2.0 / d)
        rot = torch.polar(torch.ones(len(pos), half, dtype=torch.float64), pos[:, None] * freq[None, :])
        z = torch.complex(x[..., :half], x[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    def context_kv(self, feats, slots):
        """Per-layer cached K, V [rows, Hkv, d] of feature rows at absolute slots."""
        c, w, st = self.cfg, self.w, self.st
        f = torch.from_numpy(np.asarray(feats, dtype=np.float64))
        taps = [st(self._norm(f[:, k * c.target_hidden:(k + 1) * c.target_hidden], w["aux_norms"][k]))
                for k in range(c.n_taps)]
        hid = st(self._norm(F.linear(torch.cat(taps, dim=-1), w["w_fc"]), w["hidden_norm"]))
        pos = torch.as_tensor(np.asarray(slots, dtype=np.float64))
        qd, kd = c.n_q_heads * c.head_dim, c.n_kv_heads * c.head_dim
        out = []
        for l in range(c.n_layers):
            p = f"layers.{l}."
            x = st(self._norm(hid, w[p + "in_norm"]))
            kv = F.linear(x, w[p + "w_qkv"][qd:qd + 2 * kd])
            k = kv[:, :kd].reshape(-1, c.n_kv_heads, c.head_dim)
            v = kv[:, kd:].reshape(-1, c.n_kv_heads, c.head_dim)
            out.append((st(self._rope(self._norm(k, w[p + "k_norm"]), pos)), st(v)))
        return out

    def block(self, tokens, Fpos, ctx_kv, ctx_pos):
        """Logits of rows 1..n for the block [anchor, mask x n] at Fpos."""
        c, w, st = self.cfg, self.w, self.st
        nb = len(tokens)
        qd, kd = c.n_q_heads * c.head_dim, c.n_kv_heads * c.head_dim
        pos = Fpos + torch.arange(nb, dtype=torch.float64)
        cpos = torch.as_tensor(np.asarray(ctx_pos, dtype=np.float64))
        # visibility of [context | block] keys for each block query
        kpos = torch.cat([cpos, pos])
        vis = torch.ones(nb, len(kpos), dtype=torch.bool)
        if c.window:
            vis &= (pos[:, None] - kpos[None, :]) < c.window
        if c.causal_block:
            blk = torch.arange(nb)
            vis[:, len(cpos):] &= blk[None, :] <= blk[:, None]
        group = c.n_q_heads // c.n_kv_heads
        h = w["embed"][torch.tensor(tokens)]
        for l in range(c.n_layers):
            p = f"layers.{l}."
            x = st(self._norm(h, w[p + "in_norm"]))
            qkv = F.linear(x, w[p + "w_qkv"])
            q = qkv[:, :qd].reshape(nb, c.n_q_heads, c.head_dim)
            k = qkv[:, qd:qd + kd].reshape(nb, c.n_kv_heads, c.head_dim)
            v = qkv[:, qd + kd:].reshape(nb, c.n_kv_heads, c.head_dim)
            q = st(self._rope(self._norm(q, w[p + "q_norm"]), pos))
            k = st(self._rope(self._norm(k, w[p + "k_norm"]), pos))
            v = st(v)
            ck, cv = ctx_kv[l]
            keys = torch.cat([ck, k]).transpose(0, 1).repeat_interleave(group, dim=0)     # [Hq, N, d]
            vals = torch.cat([cv, v]).transpose(0, 1).repeat_interleave(group, dim=0)
            o = F.scaled_dot_product_attention(q.transpose(0, 1), keys, vals, attn_mask=vis)  # [Hq, nb, d]
            o = o.transpose(0, 1)
            if c.gated_attention:
                o = o * torch.sigmoid(F.linear(x, w[p + "w_g"]))[:, :, None]
            o = st(o.reshape(nb, qd))
            h = st(h + F.linear(o, w[p + "w_o"]))
            y = st(self._norm(h, w[p + "post_norm"]))
            a = st(F.silu(F.linear(y, w[p + "w_gate"])) * F.linear(y, w[p + "w_up"]))
            h = st(h + F.linear(a, w[p + "w_down"]))
        z = st(self._norm(h[1:], w["final_norm"]))
        return F.linear(z, w["unembed"]).numpy()


def _round(cfg, w, odraft, n_ctx, n_pend, anchor=5, seed=3):
    """One propose on both sides: n_ctx rows flushed, n_pend rows held, then
    the block of block_size - 1 mask rows.  Returns (oracle logits, torch
    logits, oracle session, torch cached K/V)."""
    feats = S.make_features(cfg, n_ctx + n_pend, seed=seed)
    s = O.OracleSession(odraft)
    s.committed(feats[:n_ctx], 0)
    s.flush()
    s.committed(feats[n_ctx:], n_ctx)
    n = cfg.block_size - 1
    out = s.propose(anchor, n)
    td = TorchDraft(cfg, w)
    Fpos = n_ctx + n_pend
    kv = td.context_kv(feats, np.arange(Fpos))
    logits = td.block([anchor] + [cfg.mask_token] * n, Fpos, kv, np.arange(Fpos))
    return out["logits"], logits, s, kv


CASES = ["tiny_fp32", "small_bf16", "small_laguna_bf16"]


@pytest.mark.parametrize("name", CASES)
def test_draft_oracle_equals_an_independent_torch_build(name):
    cfg = S.CONFIGS[name]
    w = S.make_weights(cfg, seed=0)
    n_ctx = 150 if cfg.window else 40
    o_lg, t_lg, s, kv = _round(cfg, w, O.OracleDraft(cfg, w), n_ctx, 5)
    assert o_lg.shape == t_lg.shape == (cfg.block_size - 1, cfg.vocab)
    np.testing.assert_allclose(o_lg, t_lg, rtol=1e-9, atol=1e-9)
    # the cached context rows the oracle keeps (the window keeps the newest only)
    for slot in sorted(s.cache)[-3:] + sorted(s.cache)[:2]:
        for l in range(cfg.n_layers):
            np.testing.assert_allclose(s.cache[slot][0][l], kv[l][0][slot].numpy(), rtol=1e-9, atol=1e-9)
            np.testing.assert_allclose(s.cache[slot][1][l], kv[l][1][slot].numpy(), rtol=1e-9, atol=1e-9)


def _planted(cfg, w, mistake):
    """An oracle given a plausible mistake through its inputs alone."""
    w2 = dict(w)
    if mistake == "post_norm gain dropped":
        for l in range(cfg.n_layers):
            w2[f"layers.{l}.post_norm"] = np.ones_like(w[f"layers.{l}.post_norm"])
    elif mistake == "SiLU on the up half":
        for l in range(cfg.n_layers):
            w2[f"layers.{l}.w_gate"], w2[f"layers.{l}.w_up"] = w[f"layers.{l}.w_up"], w[f"layers.{l}.w_gate"]
    elif mistake == "hidden_norm gain dropped":
        w2["hidden_norm"] = np.ones_like(w["hidden_norm"])
    elif mistake == "final_norm gain dropped":
        w2["final_norm"] = np.ones_like(w["final_norm"])
    elif mistake == "k norm gain dropped":
        for l in range(cfg.n_layers):
            w2[f"layers.{l}.k_norm"] = np.ones_like(w[f"layers.{l}.k_norm"])
    elif mistake == "gate of the wrong head":
        for l in range(cfg.n_layers):
            w2[f"layers.{l}.w_g"] = np.roll(w[f"layers.{l}.w_g"], 1, axis=0)
    return O.OracleDraft(cfg, w2)


@pytest.mark.parametrize("mistake", ["post_norm gain dropped", "SiLU on the up half", "hidden_norm gain dropped",
                                     "final_norm gain dropped", "k norm gain dropped", "gate of the wrong head"])
def test_the_torch_build_catches_planted_mistakes(mistake):
    cfg = S.CONFIGS["small_laguna_bf16"]
    w = S.make_weights(cfg, seed=0)
    o_lg, t_lg, _, _ = _round(cfg, w, _planted(cfg, w, mistake), 100, 3)
    assert np.max(np.abs(o_lg - t_lg)) > 1e-4, mistake


def test_storage_rounding_of_the_build_is_round_to_nearest_even():
    """The frexp rounding of the build against torch's own bf16 cast on values
    that are exact in fp32 (so that the cast rounds once)."""
    x = torch.from_numpy(S.normal(1, "rt", (4096,), std=3.0).astype(np.float64))
    x = torch.cat([x, torch.tensor([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.0 - 2.0 ** -7, 0.0])])
    got = _store(S.CONFIGS["small_bf16"])(x)
    assert torch.equal(got, x.to(torch.float32).to(torch.bfloat16).to(torch.float64))
