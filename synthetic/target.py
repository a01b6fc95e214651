"""Seeded weights of the small synthetic target that drives speculative rounds.

The pages run the draft against a real target (Qwen 3.5, Laguna); no target
checkpoint exists here, so a random-init dense decoder stands in for it:
hidden 256, 4 heads of 64 (MHA), SwiGLU 512, vocabulary 32, 2 layers, RoPE
with theta 1e6, its own seed.  Its forward produces what a DFlash draft
consumes: five hidden taps per position (the embedding output, then the
residual stream after each attention and each MLP) and raw next-token logits.

This module only draws the weights (float64, row-major [out, in]); the CPU
forward lives with the oracle and the GPU forward in the library.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import normal

__all__ = ["TargetShape", "make_target_weights", "TARGET_TINY"]


@dataclass(frozen=True)
class TargetShape:
    hidden: int = 256
    n_heads: int = 4
    head_dim: int = 64
    intermediate: int = 512
    vocab: int = 32
    n_layers: int = 2
    rope_theta: float = 1e6
    rms_eps: float = 1e-6

    @property
    def n_taps(self) -> int:
        return 2 * self.n_layers + 1

    def as_dict(self) -> dict:
        return dict(hidden=self.hidden, n_heads=self.n_heads, head_dim=self.head_dim,
                    intermediate=self.intermediate, vocab=self.vocab, n_layers=self.n_layers,
                    rope_theta=self.rope_theta, rms_eps=self.rms_eps)


TARGET_TINY = TargetShape()


def make_target_weights(seed: int = 1, shape: TargetShape = TARGET_TINY, logit_scale: float = 8.0) -> dict:
    """embed [V,H] N(0,1); unembed [V,H] N(0, 0.02*logit_scale) (a wider
    unembedding keeps greedy choices well separated); norm gains 1 + N(0, .02);
    every other matrix N(0, 0.02)."""
    H, qd, I, V = shape.hidden, shape.n_heads * shape.head_dim, shape.intermediate, shape.vocab
    f64 = lambda name, shp, std=0.02, mean=0.0: normal(seed, "target." + name, shp, std=std,
                                                        mean=mean).astype(np.float64)
    w = dict(embed=f64("embed", (V, H), std=1.0), unembed=f64("unembed", (V, H), std=0.02 * logit_scale),
             final_norm=f64("final_norm", (H,), mean=1.0), layers=[])
    for l in range(shape.n_layers):
        p = f"layers.{l}."
        w["layers"].append(dict(
            n1=f64(p + "n1", (H,), mean=1.0), wq=f64(p + "wq", (qd, H)), wk=f64(p + "wk", (qd, H)),
            wv=f64(p + "wv", (qd, H)), wo=f64(p + "wo", (H, qd)), n2=f64(p + "n2", (H,), mean=1.0),
            wg=f64(p + "wg", (I, H)), wu=f64(p + "wu", (I, H)), wd=f64(p + "wd", (H, I))))
    return w
