"""Seeded synthetic inputs for the DFlash draft round.

This module only describes shapes and draws random numbers: draft configs,
random-init draft weights, target feature rows (the concatenated hidden taps
of the target's layers), pre-filled K/V caches and synthetic target logits.
It holds none of the draft round's arithmetic.  Both the CPU oracle (through
the tests) and the CUDA library consume what it produces, so the two sides
see exactly the same inputs.

Recipe (the pages ship no checkpoints, prompts or benchmark suite, so every
input is synthetic):
  * matrices ~ N(0, 0.02); norm gains ~ 1 + N(0, 0.02) so that a skipped or
    misplaced norm is visible; features ~ N(0, 1);
  * bf16 configs round each fp32 draw to the nearest bf16 (ties to even), so
    the stored values are exactly representable in both bf16 and fp64;
  * every tensor has its own stream: numpy's Philox bit generator keyed by
    (seed, crc32(tensor name)).
"""
from __future__ import annotations

import dataclasses
import zlib
from dataclasses import dataclass

import numpy as np

__all__ = [
    "DraftConfig", "CONFIGS", "rng_for", "normal", "to_dtype_values",
    "make_weights", "make_features", "make_target_logits", "make_kv",
    "weight_shapes",
]


@dataclass(frozen=True)
class DraftConfig:
    """Shape of a DFlash draft model and its block parameters."""

    name: str
    dtype: str              # "f32" or "bf16": storage type of weights/activations
    n_taps: int             # K: target layers whose hidden states are tapped
    target_hidden: int      # H_t: width of one tap
    hidden: int             # H
    n_layers: int           # L
    n_q_heads: int          # Hq
    n_kv_heads: int         # Hkv
    head_dim: int           # d
    intermediate: int       # I (SwiGLU width)
    vocab: int              # V
    block_size: int         # B_s
    mask_token: int         # m
    window: int = 0         # W; 0 = full attention over the context
    causal_block: bool = False   # causal (True) or bidirectional (False) inside the block
    gated_attention: bool = False  # per-head sigmoid gate (g_proj) on the attention output
    rope_theta: float = 1e6
    rms_eps: float = 1e-6
    # DFlash2 (block-local dynamic convolutions and a candidate selector):
    # "dflash" or "dflash2"; the convolution's width, the selector tables'
    # rank and the number of candidates per position are not on the pages
    variant: str = "dflash"
    conv_taps: int = 4
    sel_rank: int = 64
    sel_candidates: int = 8

    @property
    def feature_width(self) -> int:
        return self.n_taps * self.target_hidden

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def draft_limit(self) -> int:
        return self.block_size - 1

    def replace(self, **kw) -> "DraftConfig":
        return dataclasses.replace(self, **kw)


CONFIGS: dict[str, DraftConfig] = {
    # Tiny fp32 draft: 5 taps x hidden 256, fc 1280->256, 2 layers, 4x64 MHA,
    # causal inside the block, SwiGLU 512, vocab 32, block 8, mask id 31.
    "tiny_fp32": DraftConfig(
        name="tiny_fp32", dtype="f32", n_taps=5, target_hidden=256, hidden=256,
        n_layers=2, n_q_heads=4, n_kv_heads=4, head_dim=64, intermediate=512,
        vocab=32, block_size=8, mask_token=31, causal_block=True),
    # Qwen3-8B-shaped bf16 draft: fc 20480->4096, 5 layers, 32 Q / 8 KV heads
    # of 128, bidirectional block, SwiGLU 12288, vocab 151936, block 16.
    "qwen3_8b_bf16": DraftConfig(
        name="qwen3_8b_bf16", dtype="bf16", n_taps=5, target_hidden=4096,
        hidden=4096, n_layers=5, n_q_heads=32, n_kv_heads=8, head_dim=128,
        intermediate=12288, vocab=151936, block_size=16, mask_token=151935),
    # Laguna-style bf16 draft: fused QKV + per-head sigmoid gate, sliding
    # window 512, 4 layers, hidden 3072, 24 Q / 8 KV heads of 128, vocab 100352.
    # The MLP width is not given on the pages; 8192 is assumed.
    "laguna_bf16": DraftConfig(
        name="laguna_bf16", dtype="bf16", n_taps=5, target_hidden=3072,
        hidden=3072, n_layers=4, n_q_heads=24, n_kv_heads=8, head_dim=128,
        intermediate=8192, vocab=100352, block_size=16, mask_token=100351,
        window=512, gated_attention=True),
    # Small bf16 drafts for parity at sizes the oracle finishes in seconds:
    # several GEMM tiles, a ragged vocabulary tail, GQA groups of 4 and 3.
    "small_bf16": DraftConfig(
        name="small_bf16", dtype="bf16", n_taps=3, target_hidden=512, hidden=512,
        n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128, intermediate=1024,
        vocab=1000, block_size=16, mask_token=999),
    "small_laguna_bf16": DraftConfig(
        name="small_laguna_bf16", dtype="bf16", n_taps=3, target_hidden=384,
        hidden=384, n_layers=2, n_q_heads=6, n_kv_heads=2, head_dim=128,
        intermediate=768, vocab=1000, block_size=8, mask_token=999, window=64,
        gated_attention=True),
    # DFlash2 drafts: the tiny fp32 and small bf16 shapes with the dynamic
    # convolutions and the candidate selector
    "tiny_dflash2_fp32": DraftConfig(
        name="tiny_dflash2_fp32", dtype="f32", n_taps=5, target_hidden=256, hidden=256,
        n_layers=2, n_q_heads=4, n_kv_heads=4, head_dim=64, intermediate=512,
        vocab=32, block_size=8, mask_token=31, causal_block=True, variant="dflash2"),
    "small_dflash2_bf16": DraftConfig(
        name="small_dflash2_bf16", dtype="bf16", n_taps=3, target_hidden=512, hidden=512,
        n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128, intermediate=1024,
        vocab=1000, block_size=16, mask_token=999, variant="dflash2"),
}


def rng_for(seed: int, name: str) -> np.random.Generator:
    """Independent stream per (seed, tensor name)."""
    return np.random.Generator(np.random.Philox(key=[int(seed) & (2**64 - 1), zlib.crc32(name.encode())]))


def to_dtype_values(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 draws to the storage type; returns float32 holding exact values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype != "bf16":
        raise ValueError(dtype)
    # round-to-nearest-even on the top 16 bits of the fp32 pattern
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def normal(seed: int, name: str, shape, std: float = 1.0, mean: float = 0.0,
           dtype: str = "f32") -> np.ndarray:
    g = rng_for(seed, name)
    x = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return to_dtype_values(x, dtype)


def weight_shapes(cfg: DraftConfig) -> dict[str, tuple]:
    """Every draft tensor, row-major [out, in] for matrices."""
    H, K, Ht = cfg.hidden, cfg.n_taps, cfg.target_hidden
    s = {
        "aux_norms": (K, Ht),
        "w_fc": (H, K * Ht),
        "hidden_norm": (H,),
        "final_norm": (H,),
        "embed": (cfg.vocab, H),
        "unembed": (cfg.vocab, H),
    }
    for l in range(cfg.n_layers):
        p = f"layers.{l}."
        s[p + "in_norm"] = (H,)
        s[p + "w_qkv"] = (cfg.qkv_rows, H)
        s[p + "q_norm"] = (cfg.head_dim,)
        s[p + "k_norm"] = (cfg.head_dim,)
        if cfg.gated_attention:
            s[p + "w_g"] = (cfg.n_q_heads, H)
        s[p + "w_o"] = (H, cfg.n_q_heads * cfg.head_dim)
        s[p + "post_norm"] = (H,)
        s[p + "w_gate"] = (cfg.intermediate, H)
        s[p + "w_up"] = (cfg.intermediate, H)
        s[p + "w_down"] = (H, cfg.intermediate)
        if cfg.variant == "dflash2":
            s[p + "conv_norm"] = (H,)
            s[p + "w_dc"] = (cfg.n_q_heads * cfg.conv_taps, H)
    if cfg.variant == "dflash2":
        s["sel_prev"] = (cfg.vocab, cfg.sel_rank)
        s["sel_next"] = (cfg.vocab, cfg.sel_rank)
    return s


def make_weights(cfg: DraftConfig, seed: int = 0, names=None) -> dict[str, np.ndarray]:
    """Random-init draft weights (float32 arrays holding storage-type values)."""
    out = {}
    for name, shape in weight_shapes(cfg).items():
        if names is not None and name not in names:
            continue
        if name.endswith("norm") or name == "aux_norms":
            out[name] = normal(seed, name, shape, std=0.02, mean=1.0, dtype=cfg.dtype)
        elif name in ("sel_prev", "sel_next"):
            # selector tables: a transition term of std ~0.125 next to the logits
            out[name] = normal(seed, name, shape, std=0.125, dtype=cfg.dtype)
        else:
            out[name] = normal(seed, name, shape, std=0.02, dtype=cfg.dtype)
    return out


def make_features(cfg: DraftConfig, n_rows: int, seed: int = 0, name: str = "features") -> np.ndarray:
    """Target feature rows [n_rows, K*H_t] ~ N(0, 1) in the storage type."""
    return normal(seed, name, (n_rows, cfg.feature_width), dtype=cfg.dtype)


def make_kv(cfg: DraftConfig, n_rows: int, seed: int, name: str) -> np.ndarray:
    """Directly seeded context K or V rows [L, Hkv, n_rows, d] ~ N(0, 1).

    Used where filling a long cache through real flushes would take the CPU
    oracle too long; both sides then read the same rows.
    """
    return normal(seed, name, (cfg.n_layers, cfg.n_kv_heads, n_rows, cfg.head_dim), dtype=cfg.dtype)


def make_target_logits(batch: int, rows: int, vocab: int, draft_tokens: np.ndarray,
                       seed: int = 0, std: float = 3.0, boost: float = 6.0,
                       p_boost: float = 0.6) -> np.ndarray:
    """Synthetic target logits [B, rows, V] fp32: N(0, std) plus `boost` on the
    draft's proposal token at each verified position with probability p_boost.

    Row r scores the token after position r, so row r-1 is the one that
    checks draft token d_r; the last row (the bonus row) gets no boost.
    """
    g = rng_for(seed, "target_logits")
    x = g.standard_normal(size=(batch, rows, vocab), dtype=np.float32)
    x *= np.float32(std)
    coin = rng_for(seed, "target_boost").random(size=(batch, rows - 1)) < p_boost
    n = draft_tokens.shape[1]
    for b in range(batch):
        for r in range(min(rows - 1, n)):
            if coin[b, r]:
                x[b, r, int(draft_tokens[b, r])] += np.float32(boost)
    return x
