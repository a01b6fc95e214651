"""dflash_verify_noalloc, the verification entry point that allocates no device
memory, against dflash_verify and against the oracle.

A serving runtime that owns all GPU memory under a fixed budget, or a decode
loop that cannot take cudaMalloc's implicit device synchronisation between
rounds, calls the allocation-free variant; it must return the same accept
lengths and bonus tokens as the regular call on the same inputs, call after
call (its scratch keeps the previous call's contents), with and without a
truncating sampler, and it must leave the device's free memory unchanged
where the regular call would grow its workspace.  This file runs last, so a
failure here leaves every other test already run."""
import numpy as np
import pytest
import torch

import synthetic as S
from tests.gpu_util import Pair, lib, verify_parity

pytestmark = pytest.mark.gpu


def _proposed_batch(D, p, T, lens=(20, 75, 130), sampler=None):
    cfg = p.cfg
    n = cfg.block_size - 1
    sess = []
    for b, L in enumerate(lens):
        _, f = p.feats(L, seed=30 + b)
        s = D.dflash_open(p.model, max_ctx=512)
        D.dflash_committed(s, f, 0)
        if sampler:
            D.dflash_set_sampler(s, *sampler)
        sess.append(s)
    B = len(sess)
    cur = torch.tensor([(4 + 7 * b) % cfg.vocab for b in range(B)], dtype=torch.int32, device="cuda")
    tok = torch.empty((B, n), dtype=torch.int32, device="cuda")
    q = torch.empty((B, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((B, n, cfg.vocab), dtype=torch.float32, device="cuda")
    assert D.dflash_propose(sess, cur, n, T, 5, 1, tok, q, lg) == [n] * B
    torch.cuda.synchronize()
    d = tok.cpu().numpy()
    tl = torch.from_numpy(S.make_target_logits(B, n + 1, cfg.vocab, d, seed=9, std=1.0, boost=4.0)).cuda()
    return sess, tok, tl, lg, n


@pytest.mark.parametrize("T,sampler", [(0.0, None), (0.7, None), (0.7, (40, 0.9, 0.0))])
def test_noalloc_verify_equals_verify_twice(T, sampler):
    D = lib()
    p = Pair(S.CONFIGS["small_bf16"])
    sess, tok, tl, lg, n = _proposed_batch(D, p, T, sampler=sampler)
    B = len(sess)
    outs = []
    for fn in (D.dflash_verify, D.dflash_verify_noalloc, D.dflash_verify_noalloc):
        acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        bon = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        fn(sess, tl, tok, n, T, 11, 1, acc, bon)
        torch.cuda.synchronize()
        outs.append((acc.cpu().numpy(), bon.cpu().numpy()))
    for a, b in outs[1:]:
        np.testing.assert_array_equal(a, outs[0][0])
        np.testing.assert_array_equal(b, outs[0][1])
    assert np.all((outs[0][0] >= 0) & (outs[0][0] <= n))
    # and against the oracle's verify on the same draft and target logits
    g_lg, g_tok, t_np = lg.double().cpu().numpy(), tok.cpu().numpy(), tl.double().cpu().numpy()
    compared = sum(verify_parity((outs[2][0][b], outs[2][1][b]), t_np[b], g_tok[b], g_lg[b], g_tok[b], T, T, 11, 1, b,
                                 sampler, sampler if T > 0 else None) for b in range(B))
    assert compared >= B - 1, compared
    D.dflash_device_status(p.model)
    for s in sess:
        D.dflash_close(s)


def test_noalloc_verify_leaves_free_memory_unchanged():
    """A first call with a batch the model's workspace has never seen: the
    regular verify would grow its workspace; this one must not allocate.
    The timing records count it as a verify."""
    D = lib()
    p = Pair(S.CONFIGS["small_bf16"])
    lens = tuple(16 + 5 * b for b in range(100))
    sess, tok, tl, _, n = _proposed_batch(D, p, 0.7, lens=lens, sampler=(40, 0.9, 0.0))
    B = len(sess)
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bon = torch.empty(B, dtype=torch.int32, device="cuda")
    # the same kernels once on a small batch, timed, so that neither lazily
    # loaded code nor the timing events are created inside the window below
    D.dflash_timing_enable(p.model, True)
    D.dflash_verify_noalloc(sess[:2], tl[:2], tok[:2], n, 0.7, 3, 0, acc[:2], bon[:2])
    D.dflash_timing_enable(p.model, False)
    D.dflash_timing_enable(p.model, True)      # clears the records; the event pair is reused
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    D.dflash_verify_noalloc(sess, tl, tok, n, 0.7, 3, 1, acc, bon)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    rec = D.dflash_timing_read(p.model)
    D.dflash_timing_enable(p.model, False)
    assert free1 == free0, (free0, free1)
    assert rec["verify"]["launches"] == 1 and rec["verify"]["total_ms"] > 0
    assert rec["all"]["launches"] == 3 + 1 + 2
    a = acc.cpu().numpy()
    assert np.all((a >= 0) & (a <= n))
    D.dflash_device_status(p.model)
    for s in sess:
        D.dflash_close(s)


def test_noalloc_verify_refuses_a_batch_beyond_its_scratch():
    D = lib()
    p = Pair(S.CONFIGS["tiny_fp32"])
    cfg = p.cfg
    n = cfg.block_size - 1
    sess = [D.dflash_open(p.model, max_ctx=16) for _ in range(129)]
    tl = torch.zeros((129, n + 1, cfg.vocab), device="cuda")
    tok = torch.zeros((129, n), dtype=torch.int32, device="cuda")
    acc = torch.empty(129, dtype=torch.int32, device="cuda")
    bon = torch.empty(129, dtype=torch.int32, device="cuda")
    with pytest.raises(D.DFlashError) as e:
        D.dflash_verify_noalloc(sess, tl, tok, n, 0.0, 0, 0, acc, bon)
    assert e.value.status == D.DFLASH_ERR_CAPACITY
    assert "128" in str(e.value)
    for s in sess:
        D.dflash_close(s)
