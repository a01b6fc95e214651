"""Pins of the oracle's truncated distributions (top-k, top-p, min-p):
supports worked by hand, the no-op and top-1 limits, ties and NaN, the
Gumbel-max draw over a truncated support, and speculative verification
reproducing the truncated target law (Leviathan et al. 2023, Theorem 1,
with p and q the sampler's truncated distributions)."""
import numpy as np
import pytest
from scipy import stats

from oracle import dflash_oracle as O

# s = [0, 2, 1, -1]: the order is ids 1, 2, 0, 3.  Worked by hand:
# Z = e^2 + e + 1 + e^-1 = 7.389 + 2.718 + 1 + 0.368 = 11.475
# p = 0.6439, 0.2369, 0.0871, 0.0321 (in that order); mass before each entry
# 0, 0.6439, 0.8808, 0.9679; p / p_max = 1, 0.3679, 0.1353, 0.0498.
# Over the top two only: p = 0.7311, 0.2689 (mass before: 0, 0.7311).
S4 = np.array([0.0, 2.0, 1.0, -1.0])


@pytest.mark.parametrize("trunc,kept", [
    ((0, 1.0, 0.0), [1, 2, 0, 3]),
    ((3, 1.0, 0.0), [1, 2, 0]),
    ((0, 0.6, 0.0), [1]),
    ((0, 0.7, 0.0), [1, 2]),
    ((0, 0.9, 0.0), [1, 2, 0]),
    ((0, 0.97, 0.0), [1, 2, 0, 3]),
    ((0, 1.0, 0.1), [1, 2, 0]),
    ((0, 1.0, 0.2), [1, 2]),
    ((0, 1.0, 0.4), [1]),
    ((2, 0.75, 0.0), [1, 2]),
    ((2, 0.7, 0.0), [1]),
    ((0, 0.95, 0.2), [1, 2]),
])
def test_support_worked_by_hand(trunc, kept):
    assert list(O.truncated_support(S4, *trunc)) == kept


def test_support_ties_and_nan():
    assert list(O.truncated_support(np.array([1.0, 1.0, 1.0, 0.0]), 2)) == [0, 1]
    assert list(O.truncated_support(np.array([np.nan, 1.0, 0.0]), 0)) == [1, 2]
    assert list(O.truncated_support(np.array([3.0, np.nan, 3.0]), 1)) == [0]
    # a tie straddling the top-p boundary keeps the lower id only
    assert list(O.truncated_support(np.array([0.0, 0.0]), 0, 0.5)) == [0]


def test_no_op_truncation_equals_full_sampling():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((6, 50)) * 2
    t0, q0, l0 = O.sample_rows(logits, 0.8, 7, 3, 1)
    t1, q1, l1 = O.sample_rows(logits, 0.8, 7, 3, 1, (50, 1.0, 0.0))
    assert np.array_equal(t0, t1)
    np.testing.assert_allclose(q1, q0, rtol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=1e-12)


def test_top1_is_greedy_at_any_temperature():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((8, 40))
    for T in (0.3, 1.0, 5.0):
        t, q, _ = O.sample_rows(logits, T, 1, 2, 0, (1, 1.0, 0.0))
        assert np.array_equal(t, np.argmax(logits, axis=1)) and np.all(q == 1.0)


def test_gumbel_max_over_the_support_draws_the_truncated_softmax():
    V = 8
    logits = np.array([1.0, 0.5, -0.3, 2.0, 0.0, -1.0, 1.5, 0.2])
    trunc = (6, 0.9, 0.0)
    p = O.sampler_distribution(logits, 1.0, trunc)
    assert np.count_nonzero(p) < 6                       # top-p cut inside the top 6
    N = 1 << 15
    cnt = np.zeros(V)
    for r in range(N):
        t, q, _ = O.sample_rows(logits[None], 1.0, 5, r, 0, trunc)
        cnt[t[0]] += 1
        assert abs(q[0] - p[t[0]]) < 1e-12
    assert np.all(cnt[p == 0] == 0)
    k = p > 0
    chi2 = np.sum((cnt[k] - N * p[k]) ** 2 / (N * p[k]))
    assert chi2 < stats.chi2.ppf(1 - 1e-4, int(k.sum()) - 1)


@pytest.mark.parametrize("pos", [0, 1])
def test_speculative_verify_reproduces_the_truncated_target_law(pos):
    """Draft and target truncate differently (the draft keeps ids the target
    drops and the reverse): the emitted token still follows the target's
    truncated distribution."""
    V, n, T = 24, 2, 0.9
    rng = np.random.default_rng(12)
    tl = rng.standard_normal((n + 1, V)) * 1.5
    dl = rng.standard_normal((n, V)) * 1.5
    tt, dt = (8, 0.9, 0.0), (10, 1.0, 0.05)
    qs = [O.sampler_distribution(dl[i], T, dt) for i in range(n)]
    cq = [np.cumsum(q) for q in qs]
    R = 1 << 15
    counts = np.zeros(V)
    for r in range(R):
        u = rng.random(n)
        d = [min(int(np.searchsorted(cq[i], u[i] * cq[i][-1], side="right")), V - 1) for i in range(n)]
        a, b = O.verify(tl, d, dl, d, T, T, 42, r, 0, tt, dt)
        emitted = list(d[:a]) + [b]
        if len(emitted) > pos:
            counts[emitted[pos]] += 1
    p = O.sampler_distribution(tl[pos], T, tt)
    assert np.all(counts[p == 0] == 0)
    k = p > 0
    total = counts.sum()
    assert total > R // 8
    chi2 = np.sum((counts[k] - total * p[k]) ** 2 / (total * p[k]))
    assert chi2 < stats.chi2.ppf(1 - 1e-4, int(k.sum()) - 1)


def test_top1_target_truncation_makes_verify_greedy():
    """With the target truncated to its top token, p is one-hot on the
    target's argmax: a draft token equal to it has ratio p/q >= 1 and is
    accepted, any other has p = 0 and is rejected, and the residual's only
    support is the target's argmax."""
    rng = np.random.default_rng(2)
    V, n = 16, 3
    tl = rng.standard_normal((n + 1, V))
    dl = rng.standard_normal((n, V))
    d = [int(np.argmax(tl[0])), int(np.argmax(tl[1])), (int(np.argmax(tl[2])) + 1) % V]
    a, b = O.verify(tl, d, dl, d, 1.0, 1.0, 3, 0, 0, (1, 1.0, 0.0), (0, 1.0, 0.0))
    assert (a, b) == (2, int(np.argmax(tl[2])))
