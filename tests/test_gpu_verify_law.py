"""The output law of speculative verification on the GPU.

Rejection sampling with the proposal's own distribution q emits tokens whose
law is the target's p, whatever q is (Leviathan, Kalman & Matias 2023,
Theorem 1; the dflash.go propose comment: verification keeps the output exact
because it uses the actual proposal probabilities).  The test draws the draft
tokens d_i ~ q_i on the host from the logits each GPU session kept from its
proposal, runs dflash_verify over many sessions and rounds (each (session,
round) pair has its own Philox counters), and histograms the token emitted at
block position `pos`.  Pearson chi-square over 2^20 trials on the tiny
draft's 32-token vocabulary must stay below chi2.ppf(1 - 1e-4, 31) = 69.11.
"""
import numpy as np
import pytest
import torch

import synthetic as S
from tests.gpu_util import Pair, lib

pytestmark = pytest.mark.gpu

CHI2_CRIT = 69.11   # chi-square quantile 1 - 1e-4 at 31 degrees of freedom


def _softmax(x):
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


@pytest.mark.parametrize("n,pos", [(1, 0), (3, 1)])
def test_gpu_verify_reproduces_target_law(n, pos):
    D = lib()
    p = Pair(S.CONFIGS["tiny_fp32"])
    V, T, B, R = p.cfg.vocab, 0.8, 512, 2048
    _, f = p.feats(24, seed=70)
    sess = []
    for _ in range(B):
        s = D.dflash_open(p.model, max_ctx=64)
        D.dflash_committed(s, f, 0)
        sess.append(s)
    cur = torch.full((B,), 4, dtype=torch.int32, device="cuda")
    tok = torch.empty((B, n), dtype=torch.int32, device="cuda")
    q = torch.empty((B, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((B, n, V), dtype=torch.float32, device="cuda")
    assert D.dflash_propose(sess, cur, n, T, 3, 0, tok, q, lg) == [n] * B
    torch.cuda.synchronize()
    # each session's proposal distribution, as the session keeps it
    qd = _softmax(lg.double().cpu().numpy() / T)                      # [B, n, V]
    rng = np.random.default_rng(12)
    tl = (rng.standard_normal((n + 1, V)) * 1.5).astype(np.float32)   # the fixed target rows
    tl_dev = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(tl, (B, n + 1, V)))).cuda()
    # d ~ q for every (round, session, position), by inversion of the CDF
    cdf = np.cumsum(qd, axis=-1)
    u = rng.random((R, B, n))
    d = np.minimum((u[..., None] > cdf[None]).sum(axis=-1), V - 1).astype(np.int32)  # [R, B, n]
    d_dev = torch.from_numpy(d).cuda()
    acc = torch.empty((R, B), dtype=torch.int32, device="cuda")
    bon = torch.empty((R, B), dtype=torch.int32, device="cuda")
    for r in range(R):
        D.dflash_verify(sess, tl_dev, d_dev[r], n, T, 42, r, acc[r], bon[r])
    torch.cuda.synchronize()
    D.dflash_device_status(p.model)
    a, b = acc.cpu().numpy(), bon.cpu().numpy()
    assert a.min() >= 0 and a.max() <= n and b.min() >= 0 and b.max() < V
    # emitted tokens: d_1..d_a, then the bonus
    if pos == 0:
        emitted = np.where(a >= 1, d[..., 0], b)
        valid = np.ones_like(a, dtype=bool)
    else:
        emitted = np.where(a >= 2, d[..., 1], b)
        valid = a >= 1
    counts = np.bincount(emitted[valid].ravel(), minlength=V).astype(np.float64)
    total = counts.sum()
    assert total > B * R // 8
    pt = _softmax(tl[pos].astype(np.float64) / T)
    chi2 = float(np.sum((counts - total * pt) ** 2 / (total * pt)))
    assert chi2 < CHI2_CRIT, chi2
    # the acceptance rate matches sum_v min(p, q) at the first position
    qa = qd[:, 0, :].mean(axis=0)
    expect = np.minimum(_softmax(tl[0].astype(np.float64) / T), qa).sum()
    assert abs(np.mean(a >= 1) - expect) < 0.01, (np.mean(a >= 1), expect)
    for s in sess:
        D.dflash_close(s)
