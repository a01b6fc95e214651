"""GPU parity of truncated sampler distributions (dflash_set_sampler): the
cut kernel, the truncated draw and q, and speculative verification with
truncated p and q, against the oracle.

Two kinds of check.  On the GPU's own logits (copied back), the oracle's
truncated support, draw and q must agree exactly up to the fp32/fp64
difference of the kept mass; this isolates the kernels at any vocabulary
size.  On the oracle's logits (small configs), the whole path agrees where
the decision is not within rounding of a boundary (a top-k gap, a top-p or
min-p threshold, a Gumbel score or an acceptance threshold)."""
import numpy as np
import pytest
import torch

import synthetic as S
from oracle import dflash_oracle as O
from tests.gpu_util import MARGIN, TOL_LOGITS, TOL_Q, Pair, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def D():
    return lib()


def _clear(s, trunc, tol):
    """True when the truncated support of the scaled row s is not decided by
    rounding: the top-k boundary gap, the top-p mass and the min-p ratio are
    all farther than tol from their thresholds."""
    top_k, top_p, min_p = trunc
    if not O.truncation_active(trunc):
        return True
    order = np.lexsort((np.arange(len(s)), -s))
    if top_k and top_k < len(s) and s[order[top_k - 1]] - s[order[top_k]] <= tol:
        return False
    # the last kept and the first dropped entry must not swap ranks
    J = len(O.truncated_support(s, *trunc))
    if J < len(s) and s[order[J - 1]] - s[order[J]] <= tol:
        return False
    kept = order[:top_k] if top_k else order
    e = np.exp(s[kept] - s[kept[0]])
    p = e / e.sum()
    before = np.cumsum(p) - p
    if top_p < 1.0 and np.any(np.abs(before - top_p) <= tol):
        return False
    if min_p > 0.0 and np.any(np.abs(p / p[0] - min_p) <= tol):
        return False
    return True


def _masked_scores(row, T, trunc, seed, rnd, seq, prow):
    s = row / T
    g = O.gumbel(seed, rnd, O.STREAM_DRAFT, seq, prow, np.arange(len(row)))
    kept = O.truncated_support(s, *trunc) if O.truncation_active(trunc) else np.arange(len(row))
    out = np.full(len(row), -np.inf)
    out[kept] = s[kept] + g[kept]
    return out, kept


def _check_draw(g_lg, g_tok, g_q, T, trunc, seed, rnd, seq):
    """The GPU's draw against the oracle on the GPU's own logits, row by row."""
    for i in range(len(g_tok)):
        s = g_lg[i] / T
        if not _clear(s, trunc, 1e-5):
            continue
        sc, kept = _masked_scores(g_lg[i], T, trunc, seed, rnd, seq, i + 1)
        t = int(g_tok[i])
        assert t in set(kept.tolist()), f"row {i}: token {t} outside the truncated support"
        top = int(np.argmax(sc))
        assert t == top or sc[top] - sc[t] <= MARGIN
        lse = O.logsumexp(s[kept])
        assert abs(float(g_q[i]) - np.exp(s[t] - lse)) <= TOL_Q


@pytest.mark.parametrize("cfg_name", ["tiny_fp32", "small_bf16"])
def test_truncated_batched_propose_and_verify(D, cfg_name):
    """Three sessions with three samplers (none, top-k + top-p, top-k + top-p
    + min-p) in one batched propose and verify at T = 0.9."""
    p = Pair(S.CONFIGS[cfg_name])
    cfg = p.cfg
    n, V, T = cfg.block_size - 1, cfg.vocab, 0.9
    samplers = [(0, 1.0, 0.0), (min(8, V - 1), 0.85, 0.0), (min(40, V - 1), 0.95, 0.02)]
    sess, oss = [], []
    for b, L in enumerate([20, 75, 130]):
        f_np, f = p.feats(L, seed=30 + b)
        s = D.dflash_open(p.model, max_ctx=512)
        D.dflash_committed(s, f, 0)
        D.dflash_set_sampler(s, *samplers[b])
        o = O.OracleSession(p.oracle, seq=b)
        o.committed(f_np, 0)
        o.set_sampler(*samplers[b])
        sess.append(s)
        oss.append(o)
    cur_np = np.array([5, 2, 7], dtype=np.int32)
    tok = torch.empty((3, n), dtype=torch.int32, device="cuda")
    q = torch.empty((3, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((3, n, V), dtype=torch.float32, device="cuda")
    assert D.dflash_propose(sess, torch.from_numpy(cur_np).cuda(), n, T, 61, 4, tok, q, lg) == [n] * 3
    refs = [o.propose(int(c), n, T, 61, 4) for o, c in zip(oss, cur_np)]
    torch.cuda.synchronize()
    g_lg = lg.double().cpu().numpy()
    g_tok = tok.cpu().numpy()
    g_q = q.cpu().numpy()
    deltas = []
    for b in range(3):
        _check_draw(g_lg[b], g_tok[b], g_q[b], T, samplers[b], 61, 4, b)
        # against the oracle's own logits where the support is not in doubt
        delta = float(np.max(np.abs(g_lg[b] - refs[b]["logits"])))
        deltas.append(delta)
        assert delta <= TOL_LOGITS[cfg.dtype]
        tol = max(MARGIN, 2.0 * delta / T)
        for i in range(n):
            ol = refs[b]["logits"][i]
            if not (_clear(ol / T, samplers[b], tol) and _clear(g_lg[b][i] / T, samplers[b], tol)):
                continue
            sc, _ = _masked_scores(ol, T, samplers[b], 61, 4, b, i + 1)
            t = int(g_tok[b][i])
            assert t == int(refs[b]["tokens"][i]) or sc[int(refs[b]["tokens"][i])] - sc[t] <= tol
    # verify the GPU's tokens against target logits that favour them
    d_np = g_tok.astype(np.int32)
    tl_np = S.make_target_logits(3, n + 1, V, d_np, seed=8, std=1.0, boost=4.0)
    acc = torch.empty(3, dtype=torch.int32, device="cuda")
    bon = torch.empty(3, dtype=torch.int32, device="cuda")
    D.dflash_verify(sess, torch.from_numpy(tl_np).cuda(), torch.from_numpy(d_np).cuda(), n, T, 17, 4, acc, bon)
    torch.cuda.synchronize()
    compared = 0
    for b in range(3):
        tr = samplers[b]
        # the oracle on the GPU's draft logits (q) and the same target logits
        # (p); a support or a decision within rounding of its boundary is
        # exempt, and the test counts the sessions actually compared
        clear = all(_clear(tl_np[b][i].astype(np.float64) / T, tr, 1e-5) for i in range(n + 1)) and \
            all(_clear(g_lg[b][i] / T, tr, 1e-5) for i in range(n))
        if not clear or _near(tl_np[b], d_np[b], g_lg[b], T, tr, 17, 4, b):
            continue
        a_ref, b_ref = O.verify(tl_np[b].astype(np.float64), d_np[b], g_lg[b], d_np[b], T, T, 17, 4, b, tr, tr)
        assert (int(acc[b]), int(bon[b])) == (a_ref, b_ref), (b, int(acc[b]), int(bon[b]), a_ref, b_ref)
        compared += 1
    assert compared >= 2, compared
    D.dflash_device_status(p.model)
    for s in sess:
        D.dflash_close(s)


def _near(tl, d, dl, T, tr, seed, rnd, seq, tol=1e-4):
    """An acceptance ratio or the bonus draw's top two within tol (fp32 against fp64)."""
    n = len(d)
    for i in range(1, n + 1):
        p = O.sampler_distribution(tl[i - 1].astype(np.float64), T, tr)
        q = O.sampler_distribution(dl[i - 1], T, tr)
        r = O.uniform_open(O.random_u32(seed, rnd, O.STREAM_ACCEPT, seq, i, 0))
        x, y = r * q[d[i - 1]], p[d[i - 1]]
        if abs(x - y) <= tol * max(abs(y), 1e-30):
            return True
        if not x < y:
            res = np.maximum(p - q, 0)
            w = res if res.sum() > 0 else p
            break
    else:
        w = O.sampler_distribution(tl[n].astype(np.float64), T, tr)
        i = n + 1
    with np.errstate(divide="ignore"):
        sc = np.log(w) + O.gumbel(seed, rnd, O.STREAM_BONUS, seq, i, np.arange(len(w)))
    top = np.sort(sc)[-2:]
    return top[1] - top[0] < tol


def test_top1_and_wide_top_k_limits(D):
    """top_k = 1 draws the argmax with q = 1 at T > 0; a top_k of at least V
    with no top-p or min-p draws what the untruncated sampler draws."""
    p = Pair(S.CONFIGS["tiny_fp32"])
    cfg = p.cfg
    n, V = cfg.block_size - 1, cfg.vocab
    f_np, f = p.feats(40, seed=3)
    outs = {}
    for name, tr in (("full", (0, 1.0, 0.0)), ("top1", (1, 1.0, 0.0)), ("wide", (1024, 1.0, 0.0))):
        s = D.dflash_open(p.model, max_ctx=256)
        D.dflash_committed(s, f, 0)
        D.dflash_set_sampler(s, *tr)
        tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
        q = torch.empty((1, n), dtype=torch.float32, device="cuda")
        lg = torch.empty((1, n, V), dtype=torch.float32, device="cuda")
        D.dflash_propose([s], torch.tensor([4], dtype=torch.int32, device="cuda"), n, 1.3, 9, 2, tok, q, lg)
        torch.cuda.synchronize()
        outs[name] = (tok.cpu().numpy()[0], q.cpu().numpy()[0], lg.cpu().numpy()[0])
        D.dflash_close(s)
    assert np.array_equal(outs["top1"][0], np.argmax(outs["top1"][2], axis=1))
    assert np.all(outs["top1"][1] == 1.0)
    assert np.array_equal(outs["wide"][0], outs["full"][0])
    np.testing.assert_allclose(outs["wide"][1], outs["full"][1], rtol=1e-5)


def test_verify_with_ties_at_the_cut_keeps_the_lower_ids(D):
    """Target rows of equal logits: a top-3 truncation keeps ids 0, 1, 2
    (ties by id), so the bonus is one of them, and a draft token outside them
    is rejected at once (p = 0)."""
    p = Pair(S.CONFIGS["tiny_fp32"])
    cfg = p.cfg
    n, V = cfg.block_size - 1, cfg.vocab
    f_np, f = p.feats(30, seed=4)
    s = D.dflash_open(p.model, max_ctx=256)
    D.dflash_committed(s, f, 0)
    D.dflash_set_sampler(s, 3, 1.0, 0.0)
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    D.dflash_propose([s], torch.tensor([1], dtype=torch.int32, device="cuda"), n, 1.0, 5, 0, tok, q)
    tl = torch.zeros((1, n + 1, V), dtype=torch.float32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    bon = torch.empty(1, dtype=torch.int32, device="cuda")
    for rnd in range(6):
        d = torch.full((1, n), 9, dtype=torch.int32, device="cuda")          # outside {0, 1, 2}
        D.dflash_verify([s], tl, d, n, 1.0, 3, rnd, acc, bon)
        torch.cuda.synchronize()
        assert int(acc[0]) == 0 and int(bon[0]) in (0, 1, 2)
    D.dflash_device_status(p.model)
    D.dflash_close(s)


def test_truncated_draw_at_full_vocabulary(D):
    """A 151,936-entry vocabulary (the Qwen3-8B unembedding width) on a small
    draft: the cut kernel's radix passes over the whole row, for the proposal
    rows and, in verify, the target rows; checked against the oracle on the
    GPU's own logits."""
    cfg = S.CONFIGS["small_bf16"].replace(vocab=151936, mask_token=151935)
    p = Pair(cfg)
    n, V, T = cfg.block_size - 1, cfg.vocab, 1.0
    tr = (40, 0.9, 0.0)
    f_np, f = p.feats(64, seed=6)
    s = D.dflash_open(p.model, max_ctx=256)
    D.dflash_committed(s, f, 0)
    D.dflash_set_sampler(s, *tr)
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((1, n, V), dtype=torch.float32, device="cuda")
    D.dflash_propose([s], torch.tensor([100], dtype=torch.int32, device="cuda"), n, T, 23, 1, tok, q, lg)
    torch.cuda.synchronize()
    g_lg = lg[0].double().cpu().numpy()
    g_tok = tok[0].cpu().numpy()
    _check_draw(g_lg, g_tok, q[0].cpu().numpy(), T, tr, 23, 1, 0)
    # target rows: N(0, 3) logits with the proposal boosted
    d_np = g_tok[None].astype(np.int32)
    tl_np = S.make_target_logits(1, n + 1, V, d_np, seed=9, std=3.0, boost=6.0)
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    bon = torch.empty(1, dtype=torch.int32, device="cuda")
    clear_q = all(_clear(g_lg[i] / T, tr, 1e-5) for i in range(n))
    compared = 0
    for rnd in range(1, 7):
        D.dflash_verify([s], torch.from_numpy(tl_np).cuda(), torch.from_numpy(d_np).cuda(), n, T, 31, rnd, acc, bon)
        torch.cuda.synchronize()
        a_ref, b_ref = O.verify(tl_np[0].astype(np.float64), d_np[0], g_lg, d_np[0], T, T, 31, rnd, 0, tr, tr)
        clear = clear_q and all(_clear(tl_np[0][i].astype(np.float64) / T, tr, 1e-5) for i in range(n + 1))
        if clear and not _near(tl_np[0], d_np[0], g_lg, T, tr, 31, rnd, 0):
            assert (int(acc[0]), int(bon[0])) == (a_ref, b_ref), rnd
            compared += 1
        # the bonus comes from the residual or from p of the row after the
        # prefix: either way from that row's truncated support
        row = tl_np[0][int(acc[0])].astype(np.float64) / T
        if _clear(row, tr, 1e-5):
            assert int(bon[0]) in set(O.truncated_support(row, *tr).tolist())
    assert compared >= 3, compared
    D.dflash_device_status(p.model)
    D.dflash_close(s)


def test_sampler_arguments_are_checked(D):
    p = Pair(S.CONFIGS["tiny_fp32"])
    s = D.dflash_open(p.model, max_ctx=64)
    for bad in ((-1, 1.0, 0.0), (1025, 1.0, 0.0), (0, 0.9, 0.0), (0, 1.0, 0.1), (10, 0.0, 0.0), (10, 1.5, 0.0),
                (10, 1.0, -0.1), (10, 1.0, 1.5)):
        with pytest.raises(D.DFlashError):
            D.dflash_set_sampler(s, *bad)
    D.dflash_set_sampler(s, 1024, 0.5, 1.0)
    D.dflash_close(s)
