"""dflash_verify_noalloc, the verification entry point that allocates no device
memory, against dflash_verify.

A serving runtime that owns all GPU memory under a fixed budget, or a decode
loop that cannot take cudaMalloc's implicit device synchronisation between
rounds, calls the allocation-free variant; it must return the same accept
lengths and bonus tokens as the regular call on the same inputs, call after
call (its scratch keeps the previous call's contents)."""
import numpy as np
import pytest
import torch

import synthetic as S
from tests.gpu_util import Pair, lib

pytestmark = pytest.mark.gpu


def _proposed_batch(D, p, T, lens=(20, 75, 130)):
    cfg = p.cfg
    n = cfg.block_size - 1
    sess = []
    for b, L in enumerate(lens):
        _, f = p.feats(L, seed=30 + b)
        s = D.dflash_open(p.model, max_ctx=512)
        D.dflash_committed(s, f, 0)
        sess.append(s)
    B = len(sess)
    cur = torch.tensor([4, 8, 15][:B], dtype=torch.int32, device="cuda")
    tok = torch.empty((B, n), dtype=torch.int32, device="cuda")
    q = torch.empty((B, n), dtype=torch.float32, device="cuda")
    assert D.dflash_propose(sess, cur, n, T, 5, 1, tok, q) == [n] * B
    torch.cuda.synchronize()
    d = tok.cpu().numpy()
    tl = torch.from_numpy(S.make_target_logits(B, n + 1, cfg.vocab, d, seed=9, std=1.0, boost=4.0)).cuda()
    return sess, tok, tl, n


@pytest.mark.parametrize("T", [0.0, 0.7])
def test_noalloc_verify_equals_verify_twice(T):
    D = lib()
    p = Pair(S.CONFIGS["small_bf16"])
    sess, tok, tl, n = _proposed_batch(D, p, T)
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
