"""The synthetic target on the GPU (dflash_target_*): its logits and hidden
taps against the target oracle, the rollback trim, block-versus-chain
exactness, and a whole greedy speculative decode (draft and target both on
the GPU) against plain greedy decoding of the target oracle."""
import numpy as np
import pytest
import torch

import synthetic as S
from oracle.target_oracle import OracleTarget, exactness_rows, exactness_summary
from synthetic.target import TARGET_TINY, make_target_weights
from tests.gpu_util import Pair, lib

pytestmark = pytest.mark.gpu


def upload_target(D, seed: int = 1, shape=TARGET_TINY, max_ctx: int = 512):
    w = make_target_weights(seed, shape)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    dw = dict(embed=f32(w["embed"]), unembed=f32(w["unembed"]), final_norm=f32(w["final_norm"]),
              layers=[{k: f32(v) for k, v in lw.items()} for lw in w["layers"]])
    return D.dflash_target_create(shape.as_dict(), dw, max_ctx=max_ctx)


def oracle_target(seed: int = 1, shape=TARGET_TINY):
    return OracleTarget(make_target_weights(seed, shape), shape)


def _fwd(D, t, tokens, start, V, NT):
    tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
    lg = torch.empty((len(tokens), V), dtype=torch.float32, device="cuda")
    tp = torch.empty((len(tokens), NT), dtype=torch.float32, device="cuda")
    D.dflash_target_forward(t, tok, start, lg, tp)
    torch.cuda.synchronize()
    return lg.cpu().numpy(), tp.cpu().numpy()


def _close(g, r, tol):
    assert np.all(np.abs(g - r) <= tol * np.maximum(1.0, np.abs(r))), float(np.max(np.abs(g - r)))


def test_target_forward_and_trim_match_the_cpu_target():
    """Prompt rows, a 5-row verify chunk, a trim to 10 rows and 3 more rows:
    logits and taps equal the CPU target's within the fp32 bar, 1e-4
    (relative above 1; fp32 against float64 arithmetic)."""
    D = lib()
    ref = oracle_target()
    t = upload_target(D)
    V, NT = ref.V, ref.n_taps * ref.H
    prompt = list(S.rng_for(0, "prompt").integers(0, V, size=8))
    for tokens, start, trim in ((prompt, 0, None), ([3, 7, 1, 30, 12], 8, 10), ([5, 9, 2], 10, None)):
        lg, tp = _fwd(D, t, tokens, start, V, NT)
        rl, rt = ref.forward(tokens, start)
        _close(lg, rl, 1e-4)
        _close(tp, rt, 1e-4)
        if trim is not None:
            D.dflash_target_trim(t, trim)
            ref.trim(trim)
        assert D.dflash_target_length(t) == ref.length
    D.dflash_target_device_status(t)


def test_target_refuses_a_gap_and_a_bad_trim():
    D = lib()
    ref = oracle_target()
    t = upload_target(D)
    _fwd(D, t, [1, 2, 3], 0, ref.V, ref.n_taps * ref.H)
    with pytest.raises(D.DFlashError) as e:
        _fwd(D, t, [4], 5, ref.V, ref.n_taps * ref.H)
    assert e.value.status == D.DFLASH_ERR_CONTEXT_GAP
    with pytest.raises(D.DFlashError):
        D.dflash_target_trim(t, 4)
    assert D.dflash_target_length(t) == 3


def test_gpu_speculative_decode_equals_greedy_decode():
    """Draft and target both on the GPU: 128 tokens of greedy speculative
    decoding (propose, a multi-row target forward, verify, trim, commit the
    accepted taps) equal plain greedy decoding of the CPU target."""
    D = lib()
    p = Pair(S.CONFIGS["tiny_fp32"])
    cfg = p.cfg
    n = cfg.block_size - 1
    cpu = oracle_target()
    prompt = list(S.rng_for(0, "prompt").integers(0, 32, size=8))
    ref = cpu.greedy_decode(prompt, 200)
    t = upload_target(D)
    V, NT = cpu.V, cpu.n_taps * cpu.H
    lg = torch.empty((n + 1, V), dtype=torch.float32, device="cuda")
    tp = torch.empty((n + 1, NT), dtype=torch.float32, device="cuda")
    first = torch.empty(1, dtype=torch.int32, device="cuda")
    lg_p = torch.empty((len(prompt), V), dtype=torch.float32, device="cuda")
    tp_p = torch.empty((len(prompt), NT), dtype=torch.float32, device="cuda")
    D.dflash_target_forward(t, torch.tensor(prompt, dtype=torch.int32, device="cuda"), 0, lg_p, tp_p)
    D.dflash_target_argmax(t, lg_p[-1:], first)
    s = D.dflash_open(p.model, max_ctx=512)
    D.dflash_committed(s, tp_p, 0)
    out = [int(first.item())]
    pos = len(prompt)
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    bon = torch.empty(1, dtype=torch.int32, device="cuda")
    cur = torch.empty(1, dtype=torch.int32, device="cuda")
    rnd, accepted = 0, 0
    while len(out) < 128:
        cur.fill_(out[-1])
        assert D.dflash_propose([s], cur, n, 0.0, 0, rnd, tok, q) == [n]
        D.dflash_target_forward(t, torch.cat([cur, tok[0]]), pos, lg, tp)
        D.dflash_verify([s], lg[None], tok, n, 0.0, 0, rnd, acc, bon)
        a, b = int(acc.item()), int(bon.item())
        D.dflash_target_trim(t, pos + a + 1)
        D.dflash_committed(s, tp[:a + 1], pos)
        out += tok[0, :a].cpu().tolist() + [b]
        pos += a + 1
        accepted += a
        rnd += 1
    assert out[:128] == ref[:128]
    assert D.dflash_target_length(t) == pos
    st = D.dflash_stats(s)
    assert st["rounds"] == rnd and st["accepted"] == accepted
    D.dflash_target_device_status(t)
    D.dflash_device_status(p.model)
    D.dflash_close(s)


def test_target_block_forward_equals_chain_forward_bitwise():
    """Every row of the target is computed on its own (GEMMs with a fixed k
    order, attention splits fixed by absolute position): an 8-row verify
    forward and 8 one-row forwards give bit-identical logits and taps, so
    greedy speculative output cannot diverge from greedy decoding."""
    D = lib()
    ref = oracle_target()
    V, NT = ref.V, ref.n_taps * ref.H
    prompt = [int(x) for x in S.rng_for(0, "prompt").integers(0, V, size=250)]
    block = [4, 17, 9, 9, 30, 1, 0, 22]   # rows 250..257 cross the 256-key split boundary
    ta = upload_target(D)
    tb = upload_target(D)
    _fwd(D, ta, prompt, 0, V, NT)
    _fwd(D, tb, prompt, 0, V, NT)
    lg_b, tp_b = _fwd(D, ta, block, len(prompt), V, NT)
    rows = [_fwd(D, tb, [x], len(prompt) + i, V, NT) for i, x in enumerate(block)]
    assert np.array_equal(lg_b, np.concatenate([r[0] for r in rows]))
    assert np.array_equal(tp_b, np.concatenate([r[1] for r in rows]))


def _planted_pair(rows=6, V=1000, seed=5):
    """Block and chain logits that differ where planted: an ulp flip, a sign
    flip, an exact tie in the chain arm that moves its argmax, a NaN."""
    rng = np.random.default_rng(seed)
    block = (rng.standard_normal((rows, V)) * 4).astype(np.float32)
    chain = block.copy()
    u = chain.view(np.uint32)
    u[1, 17] ^= 1                                   # last mantissa bit: one byte differs
    chain[2, 5] = -chain[2, 5]                      # sign: one byte
    b3 = int(np.argmax(block[3]))
    other = (b3 + 7) % V
    chain[3, other] = block[3, b3]                  # an exact tie: the lower id wins in the chain arm
    chain[4, 3] = np.nan
    block[5, :] = chain[5, :] = 1.0                 # a constant row: ids 0 and 1
    return block, chain


def test_logits_compare_matches_the_oracle():
    D = lib()
    block, chain = _planted_pair()
    rows = block.shape[0]
    out = torch.zeros(rows * D.EXACTNESS_ROW_BYTES, dtype=torch.uint8, device="cuda")
    D.dflash_logits_compare(torch.from_numpy(block).cuda(), torch.from_numpy(chain).cuda(), out)
    torch.cuda.synchronize()
    got = D.exactness_rows(out)
    want = exactness_rows(block, chain)
    for g, w in zip(got, want):
        assert g["differing_bytes"] == w["differing_bytes"]
        assert g["block_top"] == w["block_top"] and g["chain_top"] == w["chain_top"]
        assert g["block_val"] == w["block_val"] and g["chain_val"] == w["chain_val"]
    assert D.dflash_exactness_summarize(out) == exactness_summary(want)


def test_exactness_probe_allows_the_synthetic_target_and_leaves_its_cache():
    D = lib()
    t = upload_target(D)
    V = TARGET_TINY.vocab
    prompt = [int(x) for x in S.rng_for(0, "prompt").integers(0, V, size=250)]
    _fwd(D, t, prompt, 0, V, TARGET_TINY.n_taps * TARGET_TINY.hidden)
    block = torch.tensor([4, 17, 9, 9, 30, 1, 0, 22], dtype=torch.int32, device="cuda")
    bl = torch.empty((8, V), dtype=torch.float32, device="cuda")
    cl = torch.empty_like(bl)
    out = torch.zeros(8 * D.EXACTNESS_ROW_BYTES, dtype=torch.uint8, device="cuda")
    s = D.dflash_target_exactness_probe(t, block, len(prompt), bl, cl, out)
    assert s == dict(rows=8, differing_bytes=0, first_row_differing_bytes=0, disagreements=0, allows=1)
    assert D.dflash_target_length(t) == len(prompt)
    ref = oracle_target()
    ref.forward(prompt, 0)
    rl, _ = ref.forward(block.cpu().tolist(), len(prompt))
    _close(bl.cpu().numpy(), rl, 1e-4)
    rows = D.exactness_rows(out)
    assert [r["block_top"][0] for r in rows] == list(np.argmax(bl.cpu().numpy(), axis=1))
    D.dflash_target_device_status(t)
