"""Pins of the oracle's sampler penalties ("Ollama DFlash block-diffusion draft
model in mlxrunner", Facts: penalties see only committed history, not other
rows of the block; dflash.go selectBlock).

The penalty form is a reading (R25, the sampler's repetition / presence /
frequency penalties); the pins hold it to values worked by hand, to the rule
that every draft row sees the same committed history, and to the output law
of speculative verification when target row r counts d_1..d_r as history
(R26), which is what keeps the output that of classic decoding."""
import numpy as np
import pytest
from scipy import stats

import synthetic as S
from oracle import dflash_oracle as O

TINY = S.CONFIGS["tiny_fp32"]


def test_penalties_by_hand():
    logits = [2.0, -1.0, 0.5, 3.0, 0.0, -0.25]
    history = [0, 0, 3, 5, 5, 5]
    got = O.apply_penalties(logits, history, repeat=1.5, presence=0.2, frequency=0.1)
    # id 0: seen twice, positive: 2 / 1.5 - 0.2 - 2 * 0.1
    # id 3: seen once, positive: 3 / 1.5 - 0.2 - 0.1
    # id 5: seen three times, negative: -0.25 * 1.5 - 0.2 - 3 * 0.1
    want = [2.0 / 1.5 - 0.4, -1.0, 0.5, 1.7, 0.0, -0.875]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)
    # zero is "not positive": multiplied (stays 0), then the shifts apply
    np.testing.assert_allclose(O.apply_penalties([0.0, 1.0], [0], 2.0, 0.5, 0.25), [-0.75, 1.0])


def test_neutral_penalties_and_empty_history_change_nothing():
    row = np.random.default_rng(0).standard_normal(50)
    assert np.array_equal(O.apply_penalties(row, [1, 2, 2, 9], 1.0, 0.0, 0.0), row)
    assert np.array_equal(O.apply_penalties(row, [], 1.3, 0.4, 0.2), row)
    assert not O.penalties_active((1.0, 0.0, 0.0, (1, 2)))
    assert O.penalties_active((1.0, 0.0, 0.1, ()))


def test_every_block_row_sees_the_same_committed_history():
    """A propose with penalties equals the draw over each raw row penalised
    by the committed history alone; the block's own tokens never count."""
    w = S.make_weights(TINY, seed=0)
    d = O.OracleDraft(TINY, w)
    feats = S.make_features(TINY, 40, seed=4)
    hist = [3, 3, 17, 30, 5, 3]
    outs = {}
    for pen in (False, True):
        s = O.OracleSession(d)
        s.committed(feats, 0)
        if pen:
            s.set_penalties(1.3, 0.5, 0.25, hist)
        outs[pen] = s.propose(4, 7, 0.9, 11, 2)
    raw = outs[False]["logits"]
    want = np.stack([O.apply_penalties(r, hist, 1.3, 0.5, 0.25) for r in raw])
    np.testing.assert_allclose(outs[True]["logits"], want, rtol=0, atol=1e-13)
    toks, q, _ = O.sample_rows(want, 0.9, 11, 2, 0)
    assert np.array_equal(outs[True]["tokens"], toks)
    np.testing.assert_allclose(outs[True]["q"], q, rtol=1e-13)
    # the penalties do change the draw's distribution
    assert not np.allclose(outs[True]["q"], outs[False]["q"])


def test_greedy_verify_counts_the_draft_prefix_as_history():
    """Target row 1 favours id 2 by 0.1 over id 4; d_1 = 2 was accepted, so
    with a presence penalty of 0.5 row 1's choice becomes 4 (R26).  Counting
    only the committed history would have kept 2."""
    V = 5
    tl = np.full((3, V), -1.0)
    tl[0, 2] = 1.0                  # row 0 picks 2
    tl[1, 2], tl[1, 4] = 3.0, 2.9   # row 1: 2 by a hair, unless 2 is penalised
    tl[2, 0] = 1.0
    dl = np.zeros((2, V))
    pen = (1.0, 0.5, 0.0, (1,))
    assert O.verify(tl, [2, 4], dl, [2, 4], 0.0, 0.0, 0, 0, 0, penalties=pen) == (2, 0)
    assert O.verify(tl, [2, 2], dl, [2, 2], 0.0, 0.0, 0, 0, 0, penalties=pen) == (1, 4)
    assert O.verify(tl, [2, 2], dl, [2, 2], 0.0, 0.0, 0, 0, 0) == (2, 0)
    # the committed history counts on row 0 too: penalise 2 there and d_1 = 2 fails
    pen0 = (1.0, 3.0, 0.0, (2,))
    assert O.verify(tl, [2, 4], dl, [2, 4], 0.0, 0.0, 0, 0, 0, penalties=pen0)[0] == 0


@pytest.mark.parametrize("pos", [0, 1])
def test_speculative_verify_with_penalties_reproduces_the_penalised_target_law(pos):
    """With d_i ~ q_i and target rows penalised over history + d_1..d_r, the
    token emitted at position 0 follows softmax(pen_h(row 0) / T), and the
    token at position 1, given that position 0 emitted x, follows
    softmax(pen_{h + [x]}(row 1) / T).  Pearson chi-square, 2^15 rounds."""
    V, n, T = 32, 3, 0.8
    rng = np.random.default_rng(21)
    tl = rng.standard_normal((n + 1, V)) * 1.5
    dl = rng.standard_normal((n, V)) * 1.5
    hist = (0, 5, 5, 9)
    pen = (1.4, 0.3, 0.2, hist)
    qs = [O.softmax(dl[i] / T) for i in range(n)]
    cq = [np.cumsum(q) for q in qs]
    R = 1 << 15
    emitted_all = []
    for r in range(R):
        u = rng.random(n)
        d = [min(int(np.searchsorted(cq[i], u[i], side="right")), V - 1) for i in range(n)]
        a, b = O.verify(tl, d, dl, d, T, T, 7, r, 0, penalties=pen)
        emitted_all.append(list(d[:a]) + [b])
    if pos == 0:
        counts = np.bincount([e[0] for e in emitted_all], minlength=V).astype(float)
        p = O.softmax(O.apply_penalties(tl[0], hist, *pen[:3]) / T)
    else:
        firsts = np.bincount([e[0] for e in emitted_all if len(e) > 1], minlength=V)
        x = int(np.argmax(firsts))
        counts = np.bincount([e[1] for e in emitted_all if len(e) > 1 and e[0] == x], minlength=V).astype(float)
        p = O.softmax(O.apply_penalties(tl[1], list(hist) + [x], *pen[:3]) / T)
    total = counts.sum()
    assert total > 500
    keep = total * p >= 5          # Pearson's rule of thumb: pool the sparse cells
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(total * p[keep], total * p[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    chi2 = float(np.sum((obs - exp) ** 2 / exp))
    assert chi2 < stats.chi2.ppf(1 - 1e-4, len(obs) - 1), chi2
