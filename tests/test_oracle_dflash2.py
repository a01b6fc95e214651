"""Pins of the oracle's DFlash2 draft (the DFlash2 commit note and the
BlockSelector branch of selectBlock in ollama's mlxrunner/dflash.go):
block-local dynamic convolutions, a candidate selector that conditions each
token on its predecessor and returns each position's candidate distribution,
verification against those distributions, and the fixed depth of 7.

The convolution's and the selector's shapes are readings (R27, R28); the
pins hold them to an independent torch build, to their locality and
conditioning, and to what the pages fix: exactness of verification with the
candidate distributions (the output law is the target's) and greedy
speculative output equal to plain greedy decoding."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy import stats

import synthetic as S
from oracle import dflash_oracle as O
from oracle.target_oracle import OracleTarget
from synthetic.target import TARGET_TINY, make_target_weights
from tests.test_oracle_round import _speculative_run

TINY2 = S.CONFIGS["tiny_dflash2_fp32"]
SMALL2 = S.CONFIGS["small_dflash2_bf16"]


@pytest.fixture(scope="module")
def tiny2():
    return O.OracleDraft(TINY2, S.make_weights(TINY2, seed=0))


def _session(draft, n_ctx=40, seed=0):
    s = O.OracleSession(draft)
    s.committed(S.make_features(draft.cfg, n_ctx, seed=seed), 0)
    return s


def test_a_dflash2_session_drafts_seven_tokens(tiny2):
    """dflash2Depth: seven tokens every round whatever max_tokens asks for
    (capped by the block), nil when nothing is asked or nothing is committed."""
    s = _session(tiny2)
    for mt in (1, 3, 7, 100):
        out = s.propose(5, mt, 0.0)
        assert out["n"] == 7 and len(out["tokens"]) == 7
        assert out["cand_ids"].shape == out["cand_probs"].shape == (7, TINY2.sel_candidates)
    assert s.propose(5, 0) is None
    small_block = O.OracleDraft(TINY2.replace(block_size=4), S.make_weights(TINY2, seed=0))
    assert _session(small_block).propose(5, 100)["n"] == 3
    assert O.OracleSession(tiny2).propose(5, 4) is None


def _torch_dynamic_conv(cfg, w, l, h):
    """The convolution written with torch: F.rms_norm, F.linear, a softmax
    over the taps, and the windows of a zero-padded unfold."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    nb, H = h.shape
    G, kap = cfg.n_q_heads, cfg.conv_taps
    x = F.rms_norm(t(h), (H,), weight=t(w[f"layers.{l}.conv_norm"]), eps=cfg.rms_eps)
    if cfg.dtype == "f32":
        x = x.to(torch.float32).to(torch.float64)
    else:
        m, e = torch.frexp(x)
        x = torch.ldexp(torch.round(m * 256.0) / 256.0, e)
    wk = torch.softmax(F.linear(x, t(w[f"layers.{l}.w_dc"])).view(nb, G, kap), dim=-1)
    win = F.pad(x, (0, 0, kap - 1, 0)).unfold(0, kap, 1)        # [nb, H, kap]: rows i-kap+1 .. i
    wch = wk.repeat_interleave(H // G, dim=1).flip(-1)           # [nb, H, kap], tap j at window kap-1-j
    return (t(h) + (win * wch).sum(-1)).numpy()


@pytest.mark.parametrize("cfg", [TINY2, SMALL2])
def test_dynamic_conv_equals_an_independent_torch_build(cfg):
    w = S.make_weights(cfg, seed=1)
    d = O.OracleDraft(cfg, w)
    h = S.normal(2, "h", (cfg.block_size, cfg.hidden), std=1.0).astype(np.float64)
    for l in range(cfg.n_layers):
        want = _torch_dynamic_conv(cfg, w, l, h)
        st = O.storage_round(cfg.dtype)
        np.testing.assert_allclose(d.dynamic_conv(l, h), st(want), rtol=1e-12, atol=1e-12)


def test_dynamic_conv_is_causal_and_local_to_the_block(tiny2):
    """Row i mixes rows i-3..i of the block only: a change of row 5 moves rows
    5..8 and nothing else; the first rows see fewer taps (zeros before the
    anchor), so a block of equal rows does not come back unchanged at row 0."""
    h = S.normal(3, "h", (12, TINY2.hidden), std=1.0).astype(np.float64)
    base = tiny2.dynamic_conv(0, h)
    h2 = h.copy()
    h2[5] += 0.5
    moved = np.any(tiny2.dynamic_conv(0, h2) != base, axis=1)
    assert moved.tolist() == [i in (5, 6, 7, 8) for i in range(12)]
    same = np.tile(h[:1], (6, 1))
    out = tiny2.dynamic_conv(0, same)
    assert not np.allclose(out[0], out[5])          # row 0 sees one tap, row 5 all four
    np.testing.assert_allclose(out[3], out[5], rtol=1e-6)   # full windows of equal rows agree


def test_selector_candidates_and_predecessor(tiny2):
    """Candidates are the k largest logits (ties by id); the scores move with
    the predecessor, the candidates do not; q sums to one over them; at T = 0
    each token is the best score given the token before it."""
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((7, 32))
    lg[2, 10] = lg[2, 11] = 9.0                       # a tie among candidates
    toks, ids, probs, q = tiny2.select_block(lg, 3, 0.8, 1, 2, 0)
    k = TINY2.sel_candidates
    for i in range(7):
        want = np.lexsort((np.arange(32), -lg[i]))[:k]
        assert np.array_equal(ids[i], want)
        assert toks[i] in set(ids[i].tolist())
        np.testing.assert_allclose(probs[i].sum(), 1.0, rtol=1e-12)
    assert ids[2][0] == 10 and ids[2][1] == 11
    toks_b, ids_b, probs_b, _ = tiny2.select_block(lg, 17, 0.8, 1, 2, 0)
    assert np.array_equal(ids_b, ids)
    assert not np.allclose(probs_b[0], probs[0])      # the first row's predecessor changed
    A, B = tiny2.w["sel_prev"], tiny2.w["sel_next"]
    g_toks, _, g_probs, g_q = tiny2.select_block(lg, 3, 0.0, 1, 2, 0)
    prev = 3
    for i in range(7):
        score = lg[i][ids[i]] + B[ids[i]] @ A[prev]
        assert g_toks[i] == ids[i][int(np.argmax(score))]
        assert g_q[i] == 1.0
        prev = int(g_toks[i])


@pytest.mark.parametrize("pos", [0, 1])
def test_verify_with_candidate_distributions_reproduces_the_target_law(tiny2, pos):
    """Drafts drawn by the selector (each position conditioned on the drafted
    predecessor, supported on 8 of 32 ids) and verified against their
    candidate distributions emit the target's law: Pearson chi-square over
    2^14 rounds at positions 0 and 1 (the DFlash2 commit note: verification
    uses each position's candidate distribution to keep the output exact)."""
    V, n, T = 32, 3, 0.8
    rng = np.random.default_rng(8)
    tl = rng.standard_normal((n + 1, V)) * 1.5
    lg = tl[:n] + rng.standard_normal((n, V)) * 0.5     # a draft that roughly agrees with the target
    R = 1 << 14
    counts = np.zeros(V)
    for r in range(R):
        toks, ids, probs, _ = tiny2.select_block(lg, 4, T, 9, r, 0)
        a, b = O.verify(tl, toks, lg, toks, T, T, 9, r, 0, draft_cands=(ids, probs))
        emitted = list(toks[:a]) + [b]
        if len(emitted) > pos:
            counts[emitted[pos]] += 1
    p = O.softmax(tl[pos] / T)
    total = counts.sum()
    assert total > R // 8
    keep = total * p >= 5          # Pearson's rule of thumb: pool the sparse cells
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(total * p[keep], total * p[~keep].sum())
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    chi2 = float(np.sum((obs - exp) ** 2 / exp))
    assert chi2 < stats.chi2.ppf(1 - 1e-4, len(obs) - 1), chi2


def test_dflash2_greedy_speculative_equals_greedy_decode(tiny2):
    """The DFlash2 draft drives greedy rounds against the synthetic target:
    the output equals plain greedy decoding, with seven drafted per round."""
    tgt = OracleTarget(make_target_weights(1), TARGET_TINY)
    prompt = list(S.rng_for(0, "prompt").integers(0, 32, size=8))
    ref = tgt.greedy_decode(prompt, 96)
    out, sess = _speculative_run(tiny2, tgt, prompt, 96)
    assert out == ref
    assert sess.stats["proposed"] == 7 * sess.stats["rounds"]
