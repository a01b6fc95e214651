"""GPU parity of the sampler penalties (dflash_set_penalties) against the
oracle ("Ollama DFlash block-diffusion draft model in mlxrunner", Facts:
penalties see only committed history, not other rows of the block).

The penalised logits of a propose are checked against the oracle's
penalties applied to the same session's unpenalised logits (isolating the
kernel), the draw against the oracle's decision on those logits, the whole
round against the oracle session, and verify -- whose target row r counts
the history plus d_1..d_r -- against the oracle's verify on the same draft
and target logits."""
import numpy as np
import pytest
import torch

import synthetic as S
from oracle import dflash_oracle as O
from tests.gpu_util import (TOL_LOGITS, Pair, check_tokens, check_tokens_for, lib, verify_parity)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def D():
    return lib()


def _hist(ids):
    return torch.tensor(ids, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("cfg_name", ["tiny_fp32", "small_bf16"])
@pytest.mark.parametrize("T", [0.0, 0.8])
def test_penalised_propose_and_verify(D, cfg_name, T):
    p = Pair(S.CONFIGS[cfg_name])
    cfg = p.cfg
    n, V = cfg.block_size - 1, cfg.vocab
    sess, oss = [], []
    for b, L in enumerate([20, 75, 130]):
        f_np, f = p.feats(L, seed=50 + b)
        s = D.dflash_open(p.model, max_ctx=512)
        D.dflash_committed(s, f, 0)
        o = O.OracleSession(p.oracle, seq=b)
        o.committed(f_np, 0)
        sess.append(s)
        oss.append(o)
    cur_np = np.array([3, 9, 1], dtype=np.int32)
    cur = torch.from_numpy(cur_np).cuda()
    tok = torch.empty((3, n), dtype=torch.int32, device="cuda")
    q = torch.empty((3, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((3, n, V), dtype=torch.float32, device="cuda")
    # the unpenalised proposal first (the same block is recomputed below)
    D.dflash_propose(sess, cur, n, T, 77, 5, tok, q, lg)
    torch.cuda.synchronize()
    raw = lg.double().cpu().numpy()
    top = [[int(x) for x in np.argsort(-raw[b].max(axis=0))[:6]] for b in range(3)]
    rng = np.random.default_rng(3)
    pens = [None,
            (1.3, 0.4, 0.1, tuple(top[1] + top[1][:3] + [int(x) for x in rng.integers(0, V, 20)])),
            (1.0, 0.8, 0.0, tuple(int(x) for x in rng.integers(0, V, 300)) + tuple(top[2]))]
    for s, o, pen in zip(sess, oss, pens):
        if pen:
            D.dflash_set_penalties(s, pen[0], pen[1], pen[2], _hist(list(pen[3])))
            o.set_penalties(*pen[:3], history=pen[3])
    assert D.dflash_propose(sess, cur, n, T, 77, 5, tok, q, lg) == [n] * 3
    refs = [o.propose(int(c), n, T, 77, 5) for o, c in zip(oss, cur_np)]
    torch.cuda.synchronize()
    g_lg, g_tok = lg.double().cpu().numpy(), tok.cpu().numpy()
    for b in range(3):
        # the kernel: the same penalties on the same raw logits
        want = np.stack([O.penalized(r, pens[b]) for r in raw[b]])
        np.testing.assert_allclose(g_lg[b], want, rtol=2e-6, atol=2e-6)
        # the draw: the oracle's decision on the GPU's penalised logits
        check_tokens(g_tok[b], g_lg[b], T, 77, 5, b)
        # the round: against the oracle session
        assert np.max(np.abs(g_lg[b] - refs[b]["logits"])) <= TOL_LOGITS[cfg.dtype]
        check_tokens_for(cfg, g_tok[b], g_lg[b], refs[b]["logits"], T, 77, 5, b)
    assert not np.array_equal(g_lg[1], raw[1]) and np.array_equal(g_lg[0], raw[0])
    # verify on both sides: target row r penalised over the history + d_1..d_r
    d_np = g_tok.astype(np.int32)
    tl = S.make_target_logits(3, n + 1, V, d_np, seed=3, std=1.0, boost=3.0)
    acc = torch.empty(3, dtype=torch.int32, device="cuda")
    bon = torch.empty(3, dtype=torch.int32, device="cuda")
    compared = 0
    for Tv in (T, 0.0):
        D.dflash_verify(sess, torch.from_numpy(tl).cuda(), torch.from_numpy(d_np).cuda(), n, Tv, 99, 5, acc, bon)
        torch.cuda.synchronize()
        for b in range(3):
            compared += verify_parity((acc[b], bon[b]), tl[b], d_np[b], g_lg[b], g_tok[b], T, Tv, 99, 5, b,
                                      penalties=pens[b])
    assert compared >= 5, compared
    D.dflash_device_status(p.model)
    for s in sess:
        D.dflash_close(s)


def test_greedy_verify_counts_the_draft_prefix_on_gpu(D):
    """The oracle's worked case on the GPU: target row 1 prefers id 2 by 0.1
    over id 4, d_1 = 2 was accepted, and a presence penalty of 0.5 moves row
    1's choice to 4, so d_2 = 4 is accepted; without the penalties it is not."""
    p = Pair(S.CONFIGS["tiny_fp32"])
    cfg = p.cfg
    n, V = cfg.block_size - 1, cfg.vocab
    _, f = p.feats(30, seed=9)
    s = D.dflash_open(p.model, max_ctx=128)
    D.dflash_committed(s, f, 0)
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    D.dflash_propose([s], torch.tensor([1], dtype=torch.int32, device="cuda"), n, 0.0, 0, 0, tok, q)
    tl = np.full((1, n + 1, V), -1.0, dtype=np.float32)
    tl[0, 0, 2] = 1.0
    tl[0, 1, 2], tl[0, 1, 4] = 3.0, 2.9
    tl[0, 2:, 7] = 1.0
    d = np.array([[2, 4, 7, 7, 7, 7, 7]], dtype=np.int32)
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    bon = torch.empty(1, dtype=torch.int32, device="cuda")
    D.dflash_verify([s], torch.from_numpy(tl).cuda(), torch.from_numpy(d).cuda(), n, 0.0, 0, 0, acc, bon)
    torch.cuda.synchronize()
    assert int(acc[0]) == 1 and int(bon[0]) == 2
    D.dflash_set_penalties(s, 1.0, 0.5, 0.0, _hist([9]))
    tl_dev = torch.from_numpy(tl).cuda()
    D.dflash_verify([s], tl_dev, torch.from_numpy(d).cuda(), n, 0.0, 0, 0, acc, bon)
    torch.cuda.synchronize()
    pen = (1.0, 0.5, 0.0, (9,))
    a_ref, b_ref = O.verify(tl[0].astype(np.float64), d[0], None, d[0], 0.0, 0.0, 0, 0, 0, penalties=pen)
    # rows 2.. favour 7 by 2.0; once 7 is in the history its presence penalty
    # (0.5 per row, once) still leaves it on top
    assert (int(acc[0]), int(bon[0])) == (a_ref, b_ref) == (7, 7)
    # the caller's logits are not written
    assert np.array_equal(tl_dev.cpu().numpy(), tl)
    D.dflash_device_status(p.model)
    D.dflash_close(s)


def test_penalty_arguments_and_the_allocation_free_verify(D):
    p = Pair(S.CONFIGS["tiny_fp32"])
    cfg = p.cfg
    n = cfg.block_size - 1
    s = D.dflash_open(p.model, max_ctx=64)
    for bad in ((0.0, 0.0, 0.0), (-1.0, 0.0, 0.0), (float("inf"), 0.0, 0.0), (1.0, float("nan"), 0.0)):
        with pytest.raises(D.DFlashError):
            D.dflash_set_penalties(s, *bad, _hist([1]))
    with pytest.raises(D.DFlashError):
        D.dflash_set_penalties(s, 1.1, 0.0, 0.0, torch.zeros(4097, dtype=torch.int32, device="cuda"))
    _, f = p.feats(10, seed=2)
    D.dflash_committed(s, f, 0)
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    D.dflash_propose([s], torch.tensor([1], dtype=torch.int32, device="cuda"), n, 0.0, 0, 0, tok, q)
    D.dflash_set_penalties(s, 1.2, 0.0, 0.0, _hist([1, 2]))
    tl = torch.zeros((1, n + 1, cfg.vocab), device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    bon = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(D.DFlashError) as e:
        D.dflash_verify_noalloc([s], tl, tok, n, 0.0, 0, 0, acc, bon)
    assert e.value.status == D.DFLASH_ERR_INVALID_ARG
    D.dflash_set_penalties(s, 1.0, 0.0, 0.0, None)          # off again
    D.dflash_verify_noalloc([s], tl, tok, n, 0.0, 0, 0, acc, bon)
    D.dflash_close(s)
