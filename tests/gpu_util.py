"""Shared helpers of the GPU parity tests: one seeded input set handed to both
the CUDA library (through the C ABI binding) and the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import synthetic as S
from oracle import dflash_oracle as O

# tolerances of the parity bar
TOL_LOGITS = {"f32": 1e-4, "bf16": 2e-2}
TOL_Q = 1e-3
MARGIN = 1e-3


def lib():
    import block_diffusion_speculative_flush_gb300 as D
    return D


def upload(cfg, w: dict) -> dict:
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(device="cuda", dtype=dt) for k, v in w.items()}


class Pair:
    """The same draft on both sides."""

    def __init__(self, cfg, seed=0, flags=0, weights=None):
        D = lib()
        self.cfg = cfg
        self.w = weights if weights is not None else S.make_weights(cfg, seed=seed)
        self.model = D.dflash_model_create(cfg, upload(cfg, self.w), flags=flags)
        self.oracle = O.OracleDraft(cfg, self.w)
        self.dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32

    def feats(self, rows, seed=0, name="features"):
        f = S.make_features(self.cfg, rows, seed=seed, name=name)
        return f, torch.from_numpy(f).to(device="cuda", dtype=self.dt)


def export_kv(D, sess, cfg, layer, first, n):
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    k = torch.empty((cfg.n_kv_heads, n, cfg.head_dim), device="cuda", dtype=dt)
    v = torch.empty_like(k)
    D.dflash_kv_export(sess, layer, first, n, k, v)
    torch.cuda.synchronize()
    return k.double().cpu().numpy(), v.double().cpu().numpy()


def oracle_scores(logits, T, seed, rnd, seq):
    """The score whose argmax is the drawn token, and its top-2 margin, per row."""
    logits = np.atleast_2d(logits)
    out, margins = [], []
    for i, row in enumerate(logits):
        s = row / T if T > 0 else row.copy()
        if T > 0:
            s = s + O.gumbel(seed, rnd, O.STREAM_DRAFT, seq, i + 1, np.arange(len(row)))
        top = np.sort(s)[-2:]
        out.append(s)
        margins.append(top[1] - top[0])
    return np.array(out), np.array(margins)


def assert_tokens(gpu_tok, ora_tok, margins, margin=MARGIN):
    gpu_tok = np.asarray(gpu_tok).reshape(-1)
    ora_tok = np.asarray(ora_tok).reshape(-1)
    margins = np.asarray(margins).reshape(-1)
    bad = (gpu_tok != ora_tok) & (margins >= margin)
    assert not bad.any(), f"token mismatch at rows {np.nonzero(bad)[0]}: gpu {gpu_tok[bad]} oracle {ora_tok[bad]} " \
                          f"margins {margins[bad]}"
    return int(((gpu_tok != ora_tok)).sum())
