"""Pins of the oracle's elementary steps against facts fixed outside it:
published known-answer vectors, closed forms, textbook identities and
library routines.  CPU only."""
import os

import numpy as np
import pytest
import torch
from scipy import stats

from oracle import dflash_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    """Philox4x32-10 reproduces the Random123 known-answer vectors."""
    n = 0
    for line in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        assert f[0] == "philox4x32" and f[1] == "10"
        v = [int(x, 16) for x in f[2:]]
        out = O.philox4x32_10(*v[0:6])
        assert [int(o) for o in out] == v[6:10]
        n += 1
    assert n == 3


def test_uniform_is_open_and_fp32_exact():
    x = np.array([0, 1, 511, 512, 2**32 - 1, 2**31], dtype=np.uint64)
    u = O.uniform_open(x)
    assert np.all(u > 0) and np.all(u < 1)
    assert u[0] == 0.5 * 2.0 ** -23 and u[1] == u[0] and u[3] == 1.5 * 2.0 ** -23
    assert u[4] == 1 - 0.5 * 2.0 ** -23
    assert np.all(u.astype(np.float32).astype(np.float64) == u)


def test_uniform_stream_is_uniform():
    """Kolmogorov-Smirnov against U(0,1) over 2^16 counters."""
    u = O.uniform_open(O.random_u32(123, 7, 0, 3, 5, np.arange(1 << 16)))
    assert stats.kstest(u, "uniform").pvalue > 1e-4


def test_gumbel_max_draws_softmax():
    """argmax(l + Gumbel) is a draw from softmax(l): Pearson chi-square over
    2^16 independent rows (the textbook Gumbel-max property)."""
    V = 8
    logits = np.array([1.0, 0.5, -0.3, 2.0, 0.0, -1.0, 1.5, 0.2])
    p = O.softmax(logits)
    N = 1 << 16
    cnt = np.zeros(V)
    rows = np.arange(N)
    # counter v varies fastest; a different seq per draw gives independent rows
    g = np.stack([O.gumbel(99, 0, O.STREAM_DRAFT, rows, 1, v) for v in range(V)], axis=1)
    np.add.at(cnt, np.argmax(logits[None, :] + g, axis=1), 1)
    chi2 = np.sum((cnt - N * p) ** 2 / (N * p))
    assert chi2 < stats.chi2.ppf(1 - 1e-4, V - 1)


def test_round_bf16_against_torch():
    """Nearest-even rounding agrees with torch's fp32 -> bf16 conversion on
    fp32 inputs, including exact ties."""
    rng = np.random.default_rng(0)
    x = rng.standard_normal(100000).astype(np.float32) * np.float32(10.0)
    ties = np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 3 * 2**-9 + 2**-17], dtype=np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_bf16(x.astype(np.float64)), ref)
    assert O.round_bf16(np.array([1 + 2**-8]))[0] == 1.0
    assert O.round_bf16(np.array([1 + 3 * 2**-8]))[0] == 1 + 2**-6


def test_rmsnorm_closed_forms():
    x = np.array([3.0, 4.0])
    np.testing.assert_allclose(O.rmsnorm(x, np.ones(2), 0.0), x / np.sqrt(12.5), rtol=1e-15)
    rng = np.random.default_rng(1)
    y = rng.standard_normal((5, 64))
    g = 1 + 0.1 * rng.standard_normal(64)
    n1 = O.rmsnorm(y, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(n1 ** 2, axis=-1)), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.rmsnorm(7.5 * y, g, 0.0), O.rmsnorm(y, g, 0.0), rtol=1e-13)
    # eps enters under the root: a zero row stays zero, a tiny row is damped
    assert np.all(O.rmsnorm(np.zeros(4), np.ones(4), 1e-6) == 0)
    t = np.full(4, 1e-3)
    np.testing.assert_allclose(O.rmsnorm(t, np.ones(4), 1e-6), t / np.sqrt(1e-6 + 1e-6))


def test_rope_is_a_rotation():
    # d = 2: the pair (1, 0) turns by exactly pos radians (theta^0 = 1)
    for pos in [0.0, 0.3, 2.0, -1.0]:
        np.testing.assert_allclose(O.rope(np.array([1.0, 0.0]), pos, 1e6), [np.cos(pos), np.sin(pos)], atol=1e-15)
        np.testing.assert_allclose(O.rope(np.array([0.0, 1.0]), pos, 1e6), [-np.sin(pos), np.cos(pos)], atol=1e-15)
    rng = np.random.default_rng(2)
    d = 128
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    assert np.array_equal(O.rope(q, 0.0, 1e6), q)
    # pairs (j, j+d/2) keep their length
    r = O.rope(q, 37.0, 1e6)
    np.testing.assert_allclose(r[:64] ** 2 + r[64:] ** 2, q[:64] ** 2 + q[64:] ** 2, rtol=1e-12)
    # scores depend only on the position difference
    s1 = O.rope(q, 100.0, 1e6) @ O.rope(k, 40.0, 1e6)
    s2 = O.rope(q, 1060.0, 1e6) @ O.rope(k, 1000.0, 1e6)
    np.testing.assert_allclose(s1, s2, rtol=1e-9)
    # the j-th pair turns with frequency theta^(-2j/d): check pair 1 at d = 4
    x = np.array([0.0, 1.0, 0.0, 0.0])
    np.testing.assert_allclose(O.rope(x, 5.0, 100.0), [0, np.cos(0.5), 0, np.sin(0.5)], atol=1e-15)


class _Cfg:
    def __init__(self, **kw):
        self.__dict__.update(dict(n_q_heads=4, n_kv_heads=2, head_dim=16, window=0,
                                  causal_block=False, dtype="f32"))
        self.__dict__.update(kw)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (False, 5), (True, 7)])
def test_attention_matches_library_sdpa(causal, window):
    """The oracle's per-row attention equals torch's scaled_dot_product_attention
    (float64) over [context | block] keys with an explicit boolean mask and
    K/V heads repeated to the query heads."""
    cfg = _Cfg(causal_block=causal, window=window)
    d = O.OracleDraft.__new__(O.OracleDraft)
    d.cfg, d.group = cfg, cfg.n_q_heads // cfg.n_kv_heads
    rng = np.random.default_rng(3)
    N, nb, F = 11, 6, 20
    cpos = np.array([2, 5, 9, 10, 12, 13, 14, 15, 17, 18, 19], dtype=np.float64)
    ck, cv = rng.standard_normal((2, N, 2, 16))
    q = rng.standard_normal((nb, 4, 16))
    k, v = rng.standard_normal((2, nb, 2, 16))
    pos = F + np.arange(nb, dtype=np.float64)
    o = d.attention(q, k, v, pos, ck, cv, cpos)
    keys = np.concatenate([ck, k])                        # [N+nb, 2, 16]
    vals = np.concatenate([cv, v])
    kpos = np.concatenate([cpos, pos])
    mask = np.ones((nb, N + nb), dtype=bool)
    for i in range(nb):
        if window:
            mask[i] &= (pos[i] - kpos) < window
        if causal:
            mask[i, N:] &= np.arange(nb) <= i
    Q = torch.from_numpy(q).permute(1, 0, 2)              # [H, nb, d]
    Kt = torch.from_numpy(keys).permute(1, 0, 2).repeat_interleave(2, dim=0)
    Vt = torch.from_numpy(vals).permute(1, 0, 2).repeat_interleave(2, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt, attn_mask=torch.from_numpy(mask))
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_single_key_attention_returns_its_value():
    cfg = _Cfg(n_q_heads=2, n_kv_heads=1, head_dim=4)
    d = O.OracleDraft.__new__(O.OracleDraft)
    d.cfg, d.group = cfg, 2
    v = np.array([[[1.0, -2.0, 3.0, 0.5]]])
    o = d.attention(np.ones((1, 2, 4)), np.zeros((1, 1, 4)), v, np.array([0.0]),
                    np.zeros((0, 1, 4)), np.zeros((0, 1, 4)), np.zeros(0))
    assert np.array_equal(o[0, 0], v[0, 0]) and np.array_equal(o[0, 1], v[0, 0])
    # two keys with equal scores average their values
    k2 = np.zeros((2, 1, 4))
    v2 = np.array([[[2.0, 0, 0, 0]], [[0, 4.0, 0, 0]]])
    o2 = d.attention(np.ones((1, 2, 4)), k2[:1], v2[:1], np.array([1.0]), k2[1:], v2[1:], np.array([0.0]))
    np.testing.assert_allclose(o2[0, 0], [1.0, 2.0, 0, 0])


def test_window_visibility_by_hand():
    cfg = _Cfg(window=3)
    d = O.OracleDraft.__new__(O.OracleDraft)
    d.cfg = cfg
    vis = d.visible(10.0, np.arange(12, dtype=np.float64), 0, None)
    # a query at 10 sees 8, 9, 10 (W counts the query itself) and later rows
    assert list(np.nonzero(vis)[0]) == [8, 9, 10, 11]


def test_sampling_greedy_and_cold_limit():
    logits = np.array([[0.1, 3.0, 2.9, -1.0], [5.0, 5.0, 1.0, 0.0]])
    toks, q, lse = O.sample_rows(logits, 0.0, 0, 0, 0)
    assert list(toks) == [1, 0] and np.all(q == 1) and np.all(np.isnan(lse))
    # T -> 0 with separated logits: the Gumbel draw is the argmax
    toks, q, _ = O.sample_rows(np.array([[0.1, 3.0, 2.0, -1.0]]), 1e-3, 5, 9, 2)
    assert toks[0] == 1 and q[0] > 0.999999
    # q(token) is the softmax probability of the drawn token
    l = np.array([[0.3, -0.2, 1.1, 0.0]])
    toks, q, lse = O.sample_rows(l, 0.7, 1, 2, 3)
    np.testing.assert_allclose(q[0], O.softmax(l[0] / 0.7)[toks[0]], rtol=1e-14)
    np.testing.assert_allclose(lse[0], np.log(np.sum(np.exp(l[0] / 0.7))), rtol=1e-14)


def test_greedy_verify_by_hand():
    V = 5
    tl = np.full((4, V), -1.0)
    tl[0, 2] = tl[1, 4] = tl[2, 1] = tl[3, 0] = 1.0   # argmaxes 2, 4, 1, 0
    dl = np.zeros((3, V))
    assert O.verify(tl, [2, 4, 1], dl, [2, 4, 1], 0.0, 0.0, 0, 0, 0) == (3, 0)
    assert O.verify(tl, [2, 3, 1], dl, [2, 3, 1], 0.0, 0.0, 0, 0, 0) == (1, 4)
    assert O.verify(tl, [0, 4, 1], dl, [0, 4, 1], 0.0, 0.0, 0, 0, 0) == (0, 2)


@pytest.mark.parametrize("n,pos", [(1, 0), (3, 1)])
def test_speculative_verify_reproduces_target_law(n, pos):
    """Rejection sampling with the proposal's own q returns tokens distributed
    as the target p (Leviathan et al. 2023, Theorem 1): draws d_i ~ q_i,
    verifies, and histograms the token emitted at block position `pos`.
    Pearson chi-square over 2^16 rounds on a 32-token vocabulary."""
    V = 32
    rng = np.random.default_rng(11)
    tl = rng.standard_normal((n + 1, V)) * 1.5      # target logits
    dl = rng.standard_normal((n, V)) * 1.5          # draft logits
    T = 0.8
    R = 1 << 16
    counts = np.zeros(V)
    qs = [O.softmax(dl[i] / T) for i in range(n)]
    cq = [np.cumsum(q) for q in qs]
    for r in range(R):
        u = rng.random(n)
        d = [min(int(np.searchsorted(cq[i], u[i], side="right")), V - 1) for i in range(n)]
        a, b = O.verify(tl, d, dl, d, T, T, 42, r, 0)
        emitted = list(d[:a]) + [b]
        if len(emitted) > pos:
            counts[emitted[pos]] += 1
    # the token emitted at block position j follows p_{j+1} (target row j):
    # position 0 always exists; position 1 exists when d_1 was accepted and
    # is then drawn (accept or residual) against the fixed target row 1
    p = O.softmax(tl[pos] / T)
    total = counts.sum()
    assert total > R // 8
    chi2 = np.sum((counts - total * p) ** 2 / (total * p))
    assert chi2 < stats.chi2.ppf(1 - 1e-4, V - 1)
