"""GPU parity of the DFlash2 draft against the oracle (the DFlash2 commit note
and the BlockSelector branch of selectBlock in ollama's mlxrunner/dflash.go):
the dynamic convolutions inside the block forward, the candidate selector,
the fixed depth of 7, and verification against the candidate distributions.

The selector is checked on the GPU's own logits (candidates exactly, tokens
and probabilities by the oracle's decision on the same logits), the logits
against the oracle's forward, verify against the oracle's verify with the
GPU's candidate distributions, and the whole loop by greedy speculative
decoding of the synthetic target and by the output law of rejection sampling."""
import numpy as np
import pytest
import torch

import synthetic as S
from oracle import dflash_oracle as O
from oracle.target_oracle import OracleTarget
from synthetic.target import TARGET_TINY, make_target_weights
from tests.gpu_util import MARGIN, TOL_LOGITS, Pair, lib, top2_margin, verify_parity

pytestmark = pytest.mark.gpu

CASES = ["tiny_dflash2_fp32", "small_dflash2_bf16"]


@pytest.fixture(scope="module")
def D():
    return lib()


def _propose(D, p, sess, cur_np, T, seed, rnd, max_tokens=100):
    cfg = p.cfg
    B, n, k = len(sess), O.DFLASH2_DEPTH, cfg.sel_candidates
    tok = torch.empty((B, n), dtype=torch.int32, device="cuda")
    q = torch.empty((B, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((B, n, cfg.vocab), dtype=torch.float32, device="cuda")
    assert D.dflash_propose(sess, torch.from_numpy(cur_np).cuda(), max_tokens, T, seed, rnd, tok, q, lg) == [n] * B
    ids = torch.empty((B, n, k), dtype=torch.int32, device="cuda")
    probs = torch.empty((B, n, k), dtype=torch.float32, device="cuda")
    for b, s in enumerate(sess):
        D.dflash_candidates(s, ids[b], probs[b])
    torch.cuda.synchronize()
    return (tok.cpu().numpy(), q.cpu().numpy(), lg.double().cpu().numpy(), ids.cpu().numpy(),
            probs.double().cpu().numpy())


def _check_selector(draft, cur, lg, toks, q, ids, probs, T, seed, rnd, seq):
    """The GPU's selection against the oracle's selector run on the GPU's
    logits: candidates exactly; tokens and probabilities position by position
    while the predecessors agree (a near-tie of the draw, margin < 1e-3, ends
    the comparison, since every later position is conditioned on it)."""
    V = lg.shape[1]
    k = ids.shape[1]
    o_toks, o_ids, o_probs, o_q = draft.select_block(lg, cur, T, seed, rnd, seq)
    A, Bt = draft.w["sel_prev"], draft.w["sel_next"]
    prev = cur
    for i in range(len(toks)):
        assert np.array_equal(ids[i], o_ids[i]), i
        if toks[i] != o_toks[i]:
            score = lg[i][ids[i]] + Bt[ids[i]] @ A[prev]
            z = score / T + O.gumbel(seed, rnd, O.STREAM_DRAFT, seq, i + 1, ids[i]) if T > 0 else score
            assert top2_margin(z) < MARGIN, (i, toks[i], o_toks[i])
            return i
        np.testing.assert_allclose(probs[i], o_probs[i], rtol=1e-4, atol=1e-5)
        np.testing.assert_allclose(q[i], o_q[i], rtol=1e-4, atol=1e-5)
        prev = int(toks[i])
    return len(toks)


@pytest.mark.parametrize("cfg_name", CASES)
@pytest.mark.parametrize("T", [0.0, 0.8])
def test_dflash2_propose_and_verify_match_the_oracle(D, cfg_name, T):
    p = Pair(S.CONFIGS[cfg_name])
    cfg = p.cfg
    n, V = O.DFLASH2_DEPTH, cfg.vocab
    sess, oss = [], []
    for b, L in enumerate([20, 75, 130]):
        f_np, f = p.feats(L, seed=60 + b)
        s = D.dflash_open(p.model, max_ctx=512)
        D.dflash_committed(s, f, 0)
        o = O.OracleSession(p.oracle, seq=b)
        o.committed(f_np, 0)
        sess.append(s)
        oss.append(o)
    cur = np.array([3, 9, 1], dtype=np.int32)
    toks, q, lg, ids, probs = _propose(D, p, sess, cur, T, 41, 6, max_tokens=3)   # the depth overrides 3
    refs = [o.propose(int(c), 3, T, 41, 6) for o, c in zip(oss, cur)]
    checked = 0
    for b in range(3):
        assert refs[b]["n"] == n
        delta = np.max(np.abs(lg[b] - refs[b]["logits"]))
        assert delta <= TOL_LOGITS[cfg.dtype], delta
        checked += _check_selector(p.oracle, int(cur[b]), lg[b], toks[b], q[b], ids[b], probs[b], T, 41, 6, b)
        if cfg.dtype == "f32":   # the fp32 draft meets the token rule against the oracle's own logits too
            _check_selector(p.oracle, int(cur[b]), refs[b]["logits"], toks[b], q[b], ids[b], probs[b], T, 41, 6, b)
    assert checked >= 3 * n - 2
    # verify against the candidate distributions
    d_np = toks.astype(np.int32)
    tl = S.make_target_logits(3, n + 1, V, d_np, seed=4, std=1.0, boost=3.0)
    acc = torch.empty(3, dtype=torch.int32, device="cuda")
    bon = torch.empty(3, dtype=torch.int32, device="cuda")
    compared = 0
    for Tv in (0.8, 0.0):
        for fn in (D.dflash_verify, D.dflash_verify_noalloc):
            fn(sess, torch.from_numpy(tl).cuda(), torch.from_numpy(d_np).cuda(), n, Tv, 7, 6, acc, bon)
            torch.cuda.synchronize()
            for b in range(3):
                compared += verify_parity((acc[b], bon[b]), tl[b], d_np[b], lg[b], toks[b], T, Tv, 7, 6, b,
                                          draft_cands=(ids[b], probs[b]))
    assert compared >= 10, compared
    D.dflash_device_status(p.model)
    for s in sess:
        D.dflash_close(s)


def test_dflash2_greedy_speculative_output_equals_greedy_decode(D):
    """The DFlash2 tiny draft on the GPU drives greedy rounds against the
    synthetic target: the output equals plain greedy decoding of the target."""
    p = Pair(S.CONFIGS["tiny_dflash2_fp32"])
    n = O.DFLASH2_DEPTH
    tgt = OracleTarget(make_target_weights(1), TARGET_TINY)
    prompt = list(S.rng_for(0, "prompt").integers(0, 32, size=8))
    ref = tgt.greedy_decode(prompt, 80)
    logits, taps = tgt.forward(prompt, 0)
    s = D.dflash_open(p.model, max_ctx=512)
    D.dflash_committed(s, torch.from_numpy(taps).cuda(), 0)
    out = [int(np.argmax(logits[-1]))]
    pos = len(prompt)
    cur = torch.empty(1, dtype=torch.int32, device="cuda")
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    bon = torch.empty(1, dtype=torch.int32, device="cuda")
    rnd = 0
    while len(out) < 80:
        cur.fill_(out[-1])
        assert D.dflash_propose([s], cur, n, 0.0, 0, rnd, tok, q) == [n]
        d = tok[0].cpu().tolist()
        tl, tt = tgt.forward([out[-1]] + d, pos)
        D.dflash_verify([s], torch.from_numpy(tl[None]).cuda(), torch.tensor([d], dtype=torch.int32).cuda(),
                        n, 0.0, 0, rnd, acc, bon)
        a, b = int(acc[0]), int(bon[0])
        tgt.trim(pos + a + 1)
        D.dflash_committed(s, torch.from_numpy(tt[:a + 1]).cuda(), pos)
        out += d[:a] + [b]
        pos += a + 1
        rnd += 1
    assert out[:80] == ref[:80]
    D.dflash_device_status(p.model)
    D.dflash_close(s)


def test_dflash2_rejection_sampling_reproduces_the_target_law(D):
    """Sessions of the tiny DFlash2 draft propose (the selector's Gumbel draws
    vary with the session and the round) and verify at T = 0.8 against fixed
    target rows: the first emitted token follows the target's law whatever the
    candidate distributions were.  Pearson chi-square over 2^17 trials."""
    p = Pair(S.CONFIGS["tiny_dflash2_fp32"])
    n, V, T, B, R = O.DFLASH2_DEPTH, p.cfg.vocab, 0.8, 512, 256
    _, f = p.feats(24, seed=70)
    sess = []
    for _ in range(B):
        s = D.dflash_open(p.model, max_ctx=64)
        D.dflash_committed(s, f, 0)
        sess.append(s)
    rng = np.random.default_rng(13)
    tl = (rng.standard_normal((n + 1, V)) * 1.5).astype(np.float32)
    tl_dev = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(tl, (B, n + 1, V)))).cuda()
    cur = torch.full((B,), 4, dtype=torch.int32, device="cuda")
    tok = torch.empty((R, B, n), dtype=torch.int32, device="cuda")
    q = torch.empty((B, n), dtype=torch.float32, device="cuda")
    acc = torch.empty((R, B), dtype=torch.int32, device="cuda")
    bon = torch.empty((R, B), dtype=torch.int32, device="cuda")
    for r in range(R):
        D.dflash_propose(sess, cur, n, T, 5, r, tok[r], q)
        D.dflash_verify(sess, tl_dev, tok[r], n, T, 6, r, acc[r], bon[r])
    torch.cuda.synchronize()
    D.dflash_device_status(p.model)
    a, b, d = acc.cpu().numpy(), bon.cpu().numpy(), tok.cpu().numpy()
    emitted = np.where(a >= 1, d[..., 0], b).ravel()
    counts = np.bincount(emitted, minlength=V).astype(np.float64)
    e = np.exp(tl[0].astype(np.float64) / T - np.max(tl[0] / T))
    pt = e / e.sum()
    total = counts.sum()
    chi2 = float(np.sum((counts - total * pt) ** 2 / (total * pt)))
    assert chi2 < 69.11, chi2           # chi-square quantile 1 - 1e-4 at 31 degrees of freedom
    assert 0.0 < np.mean(a >= 1) < 1.0
    for s in sess:
        D.dflash_close(s)


def test_dflash2_candidates_call(D):
    p = Pair(S.CONFIGS["tiny_fp32"])
    s = D.dflash_open(p.model, max_ctx=64)
    with pytest.raises(D.DFlashError) as e:
        D.dflash_candidates(s, torch.empty(64, dtype=torch.int32, device="cuda"),
                            torch.empty(64, dtype=torch.float32, device="cuda"))
    assert e.value.status == D.DFLASH_ERR_STATE
    D.dflash_close(s)
