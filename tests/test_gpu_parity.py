"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on
the same seeded inputs, at sizes the oracle finishes in seconds that still
span several GEMM tiles, ragged vocabulary tails, GQA groups and the window
ring."""
import numpy as np
import pytest
import torch

import synthetic as S
from oracle import dflash_oracle as O
from oracle.target_oracle import OracleTarget
from synthetic.target import TARGET_TINY, make_target_weights
from tests.gpu_util import (TOL_LOGITS, TOL_Q, Pair, assert_cache_close, check_tokens, check_tokens_for, export_kv,
                            lib, verify_parity)

pytestmark = pytest.mark.gpu

SMALL = ["tiny_fp32", "small_bf16", "small_laguna_bf16"]


@pytest.fixture(scope="module")
def D():
    return lib()


@pytest.fixture(scope="module", params=SMALL)
def pair(request):
    return Pair(S.CONFIGS[request.param])


def _oracle_session(p, feats):
    s = O.OracleSession(p.oracle)
    s.committed(feats, 0)
    return s


@pytest.mark.parametrize("rows", [37, 300])
def test_flush_writes_oracle_kv(D, pair, rows):
    """Context-only forward: every cached K/V row equals the oracle's row at
    its slot (rows no query can see are dropped under a window)."""
    cfg = pair.cfg
    f_np, f = pair.feats(rows, seed=1)
    s = D.dflash_open(pair.model, max_ctx=1024)
    D.dflash_committed(s, f, 0)
    D.dflash_flush([s])
    assert D.dflash_session_state(s) == (rows, 0, False)
    os_ = _oracle_session(pair, f_np)
    os_.flush()
    lo = max(0, rows - cfg.window + 1) if cfg.window else 0
    tol = TOL_LOGITS[cfg.dtype]
    for l in range(cfg.n_layers):
        k, v = export_kv(D, s, cfg, l, lo, rows - lo)
        ok = np.stack([os_.cache[j][0][l] for j in range(lo, rows)], axis=1)
        ov = np.stack([os_.cache[j][1][l] for j in range(lo, rows)], axis=1)
        if cfg.dtype == "bf16":
            assert_cache_close(k, ok)
            assert_cache_close(v, ov)
        else:
            assert np.max(np.abs(k - ok)) <= tol and np.max(np.abs(v - ov)) <= tol
        if cfg.dtype == "bf16":   # storage values agree except for rare rounding-boundary flips
            assert np.mean(k != ok) < 0.02 and np.mean(v != ov) < 0.02
    D.dflash_close(s)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_propose_matches_oracle(D, pair, T):
    """Two rounds: propose over held rows, then commit more rows (rewinding
    the block) and propose again.  Logits, tokens and q against the oracle."""
    cfg = pair.cfg
    n = cfg.block_size - 1
    V = cfg.vocab
    f_np, f = pair.feats(90, seed=2)
    s = D.dflash_open(pair.model, max_ctx=1024)
    D.dflash_committed(s, f[:80], 0)
    os_ = _oracle_session(pair, f_np[:80])
    cur = torch.tensor([5], dtype=torch.int32, device="cuda")
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((1, n, V), dtype=torch.float32, device="cuda")
    for rnd in range(2):
        if rnd == 1:
            D.dflash_committed(s, f[80:90], 80)
            os_.committed(f_np[80:90], 80)
        out_n = D.dflash_propose([s], cur, 100, T, 1234, rnd, tok, q, lg)
        assert out_n == [n]
        ref = os_.propose(5, 100, T, 1234, rnd)
        torch.cuda.synchronize()
        g_lg = lg[0].double().cpu().numpy()
        err = np.max(np.abs(g_lg - ref["logits"]))
        assert err <= TOL_LOGITS[cfg.dtype], err
        g_tok = tok[0].cpu().numpy()
        check_tokens_for(cfg, g_tok, g_lg, ref["logits"], T, 1234, rnd, 0)
        same = g_tok == ref["tokens"]
        assert np.max(np.abs(q[0].cpu().numpy()[same] - ref["q"][same])) <= TOL_Q
        assert D.dflash_session_state(s) == (os_.F, 0, True)
    D.dflash_device_status(pair.model)
    D.dflash_close(s)


def test_nil_proposals(D):
    p = Pair(S.CONFIGS["tiny_fp32"])
    s = D.dflash_open(p.model, max_ctx=64)
    cur = torch.tensor([1], dtype=torch.int32, device="cuda")
    tok = torch.empty((1, 7), dtype=torch.int32, device="cuda")
    q = torch.empty((1, 7), dtype=torch.float32, device="cuda")
    assert D.dflash_propose([s], cur, 4, 0.0, 0, 0, tok, q) == [0]      # nothing committed
    _, f = p.feats(3)
    D.dflash_committed(s, f, 0)
    assert D.dflash_propose([s], cur, 0, 0.0, 0, 0, tok, q) == [0]      # n <= 0
    assert D.dflash_propose([s], cur, 3, 0.0, 0, 0, tok, q) == [3]
    assert D.dflash_draft_limit(p.model) == 7
    D.dflash_close(s)


def test_context_gap_is_refused(D):
    p = Pair(S.CONFIGS["tiny_fp32"])
    s = D.dflash_open(p.model, max_ctx=64)
    _, f = p.feats(10)
    D.dflash_committed(s, f[:4], 0)
    with pytest.raises(D.DFlashError) as e:
        D.dflash_committed(s, f[4:6], 5)
    assert e.value.status == D.DFLASH_ERR_CONTEXT_GAP
    assert D.dflash_session_state(s) == (0, 4, False)
    D.dflash_committed(s, f[2:6], 2)          # rows 2, 3 held already
    assert D.dflash_session_state(s) == (0, 6, False)
    with pytest.raises(D.DFlashError) as e:
        D.dflash_committed(s, p.feats(60)[1], 6)
    assert e.value.status == D.DFLASH_ERR_CAPACITY
    D.dflash_close(s)


def test_pending_rows_flush_at_256(D):
    p = Pair(S.CONFIGS["tiny_fp32"])
    s = D.dflash_open(p.model, max_ctx=1024)
    _, f = p.feats(300)
    D.dflash_committed(s, f[:255], 0)
    assert D.dflash_session_state(s) == (0, 255, False)
    D.dflash_committed(s, f[255:256], 255)
    assert D.dflash_session_state(s) == (256, 0, False)
    D.dflash_committed(s, f[256:], 256)
    assert D.dflash_session_state(s) == (256, 44, False)
    D.dflash_close(s)


@pytest.mark.parametrize("cfg_name", ["tiny_fp32", "small_bf16"])
def test_incremental_flush_is_bit_identical(D, cfg_name):
    """A context entry depends only on its own features: flushing in pieces
    gives the same cache bytes as one flush.  One flush of 300 rows takes the
    grouped many-row path (every layer's norm, K/V product and cache write in
    one launch each); pieces of up to 120 rows take the per-layer path."""
    p = Pair(S.CONFIGS[cfg_name])
    cfg = p.cfg
    _, f = p.feats(300, seed=4)
    a = D.dflash_open(p.model, max_ctx=512)
    D.dflash_committed(a, f, 0)
    D.dflash_flush([a])
    b = D.dflash_open(p.model, max_ctx=512)
    for lo, hi in [(0, 1), (1, 9), (9, 70), (70, 190), (190, 300)]:
        D.dflash_committed(b, f[lo:hi], lo)
        D.dflash_flush([b])
    for l in range(cfg.n_layers):
        ka, va = export_kv(D, a, cfg, l, 0, 300)
        kb, vb = export_kv(D, b, cfg, l, 0, 300)
        assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    D.dflash_close(a)
    D.dflash_close(b)


@pytest.mark.parametrize("cfg_name", ["tiny_fp32", "small_bf16"])
def test_rewind_then_flush_equals_never_drafting(D, cfg_name):
    p = Pair(S.CONFIGS[cfg_name])
    cfg = p.cfg
    _, f = p.feats(40, seed=5)
    n = cfg.block_size - 1
    a = D.dflash_open(p.model, max_ctx=256)
    D.dflash_committed(a, f[:30], 0)
    cur = torch.tensor([2], dtype=torch.int32, device="cuda")
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    D.dflash_propose([a], cur, n, 0.0, 0, 0, tok, q)
    assert D.dflash_session_state(a) == (30, 0, True)
    D.dflash_committed(a, f[30:33], 30)      # fewer rows than the block: stale block slots stay past F
    D.dflash_flush([a])
    assert D.dflash_session_state(a) == (33, 0, False)
    b = D.dflash_open(p.model, max_ctx=256)
    D.dflash_committed(b, f[:33], 0)
    D.dflash_flush([b])
    for l in range(cfg.n_layers):
        ka, va = export_kv(D, a, cfg, l, 0, 33)
        kb, vb = export_kv(D, b, cfg, l, 0, 33)
        assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    D.dflash_close(a)
    D.dflash_close(b)


def test_tensor_core_gemm_matches_cuda_core_gemm(D):
    """The tcgen05 path and the CUDA-core path both give the oracle's round
    (they sum in different orders, so each is held to the oracle)."""
    cfg = S.CONFIGS["small_bf16"]
    w = S.make_weights(cfg, seed=0)
    outs = []
    ref = None
    for flags in (0, D.DFLASH_FLAG_SIMT_GEMM):
        p = Pair(cfg, weights=w, flags=flags)
        f_np, f = p.feats(50, seed=6)
        if ref is None:
            o = O.OracleSession(p.oracle)
            o.committed(f_np, 0)
            ref = o.propose(7, cfg.block_size - 1, 0.0, 0, 0)["logits"]
        s = D.dflash_open(p.model, max_ctx=256)
        D.dflash_committed(s, f, 0)
        n = cfg.block_size - 1
        cur = torch.tensor([7], dtype=torch.int32, device="cuda")
        tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
        q = torch.empty((1, n), dtype=torch.float32, device="cuda")
        lg = torch.empty((1, n, cfg.vocab), dtype=torch.float32, device="cuda")
        D.dflash_propose([s], cur, n, 0.0, 0, 0, tok, q, lg)
        torch.cuda.synchronize()
        outs.append(lg.double().cpu().numpy())
        D.dflash_close(s)
    for out in outs:
        assert np.max(np.abs(out[0] - ref)) <= TOL_LOGITS["bf16"]


@pytest.mark.parametrize("cfg_name", ["tiny_fp32", "small_bf16"])
@pytest.mark.parametrize("T", [0.0, 0.7])
def test_batched_propose_and_verify(D, cfg_name, T):
    """Three sessions with different context lengths in one batched propose
    and verify; each against its own oracle session (seq id = batch index)."""
    p = Pair(S.CONFIGS[cfg_name])
    cfg = p.cfg
    n = cfg.block_size - 1
    V = cfg.vocab
    lens = [20, 75, 130]
    sess, oss = [], []
    for b, L in enumerate(lens):
        f_np, f = p.feats(L, seed=10 + b)
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
    assert D.dflash_propose(sess, cur, n, T, 77, 5, tok, q, lg) == [n] * 3
    refs = [o.propose(int(c), n, T, 77, 5) for o, c in zip(oss, cur_np)]
    torch.cuda.synchronize()
    g_lg = lg.double().cpu().numpy()
    g_tok = tok.cpu().numpy()
    for b in range(3):
        assert np.max(np.abs(g_lg[b] - refs[b]["logits"])) <= TOL_LOGITS[cfg.dtype]
        check_tokens_for(cfg, g_tok[b], g_lg[b], refs[b]["logits"], T, 77, 5, b)
    # verify on both sides: the oracle reads the draft logits that the GPU
    # session keeps from its proposal and the same target logits
    d_np = np.stack([r["tokens"] for r in refs]).astype(np.int32)
    tl_np = S.make_target_logits(3, n + 1, V, d_np, seed=3, std=1.0, boost=4.0)
    acc = torch.empty(3, dtype=torch.int32, device="cuda")
    bon = torch.empty(3, dtype=torch.int32, device="cuda")
    D.dflash_verify(sess, torch.from_numpy(tl_np).cuda(), torch.from_numpy(d_np).cuda(), n, T, 99, 5, acc, bon)
    torch.cuda.synchronize()
    compared = 0
    for b in range(3):
        compared += verify_parity((acc[b], bon[b]), tl_np[b], d_np[b], g_lg[b], g_tok[b], T, T, 99, 5, b)
    assert compared >= 2, compared
    D.dflash_device_status(p.model)
    for s in sess:
        D.dflash_close(s)


def test_greedy_speculative_output_equals_greedy_decode(D):
    """The tiny fp32 draft on the GPU drives greedy rounds against the
    synthetic 2-layer target for 128 tokens: the output equals plain greedy
    decoding of the target, with the real draft and with forced accept
    lengths 0, 1, 2 and full."""
    p = Pair(S.CONFIGS["tiny_fp32"])
    cfg = p.cfg
    n = cfg.block_size - 1
    tgt = OracleTarget(make_target_weights(1), TARGET_TINY)
    prompt = list(S.rng_for(0, "prompt").integers(0, 32, size=8))
    ref = tgt.greedy_decode(prompt, 200)
    plan = [0, 1, 2, n]
    for forced in (False, True):
        tgt.reset()
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
        while len(out) < 128:
            cur.fill_(out[-1])
            assert D.dflash_propose([s], cur, n, 0.0, 0, rnd, tok, q) == [n]
            d = tok[0].cpu().tolist()
            k = None
            if forced:
                k = plan[rnd % len(plan)]
                t = len(out)
                d = [ref[t + j] for j in range(k)] + ([(ref[t + k] + 1) % 32] if k < n else [])
                d += [0] * (n - len(d))
            tl, tt = tgt.forward([out[-1]] + d, pos)
            D.dflash_verify([s], torch.from_numpy(tl[None]).cuda(), torch.tensor([d], dtype=torch.int32).cuda(),
                            n, 0.0, 0, rnd, acc, bon)
            a, b = int(acc[0]), int(bon[0])
            if forced:
                assert a == k and b == ref[len(out) + a]
            tgt.trim(pos + a + 1)
            D.dflash_committed(s, torch.from_numpy(tt[:a + 1]).cuda(), pos)
            out += d[:a] + [b]
            pos += a + 1
            rnd += 1
        assert out[:128] == ref[:128]
        st = D.dflash_stats(s)
        assert st["rounds"] == rnd and st["proposed"] == rnd * n
        D.dflash_close(s)


@pytest.mark.parametrize("block", [8, 16])
def test_windowed_rounds_follow_the_oracle(D, block):
    """Many rounds on a window-64 gated draft: as the frontier moves, a block
    row can find whole 64-key tiles of its range outside its window.  Every
    round must stay finite and follow the oracle (logits, tokens)."""
    cfg = S.CONFIGS["small_laguna_bf16"].replace(block_size=block)
    p = Pair(cfg)
    n = block - 1
    f_np, f = p.feats(700 + 4 * 24, seed=12)
    s = D.dflash_open(p.model, max_ctx=1024)
    D.dflash_committed(s, f[:700], 0)
    o = O.OracleSession(p.oracle)
    o.committed(f_np[:700], 0)
    cur = torch.tensor([6], dtype=torch.int32, device="cuda")
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((1, n, cfg.vocab), dtype=torch.float32, device="cuda")
    for r in range(24):
        lo = 700 + 4 * r
        D.dflash_committed(s, f[lo:lo + 4], lo)
        o.committed(f_np[lo:lo + 4], lo)
        assert D.dflash_propose([s], cur, n, 1.0, 3, r, tok, q, lg) == [n]
        ref = o.propose(6, n, 1.0, 3, r)
        torch.cuda.synchronize()
        g_lg = lg[0].double().cpu().numpy()
        assert np.all(np.isfinite(g_lg)), f"round {r}: non-finite logits"
        assert np.max(np.abs(g_lg - ref["logits"])) <= TOL_LOGITS["bf16"], r
        check_tokens_for(cfg, tok[0].cpu().numpy(), g_lg, ref["logits"], 1.0, 3, r, 0)
    D.dflash_device_status(p.model)
    D.dflash_close(s)


@pytest.mark.parametrize("block", [12, 16, 24, 32])
def test_query_row_counts_and_key_tile_counts(D, block):
    """The tensor-core attention runs one softmax stream over 128 TMEM rows
    when a KV head's query rows (block x group) exceed 64, and two streams
    (even and odd key tiles) when they fit in 64.  Blocks of 12, 16, 24 and
    32 rows with groups of 4 give 48, 64, 96 and 128 query rows.  76
    sessions x 2 KV heads fill one wave of work items, so each item takes a
    session's whole key range: contexts of 20, 40, 663 and 700 rows give one
    key tile (the odd stream idle), two, an odd count and an even count."""
    cfg = S.CONFIGS["small_bf16"].replace(block_size=block)
    p = Pair(cfg)
    n, V = block - 1, cfg.vocab
    ctxs = [20, 40, 663, 700]
    B = 76
    feats = [p.feats(L, seed=31 + i) for i, L in enumerate(ctxs)]
    sess = []
    for b in range(B):
        f_np, f = feats[b % 4]
        s = D.dflash_open(p.model, max_ctx=1024)
        D.dflash_committed(s, f, 0)
        sess.append(s)
    cur_np = np.array([9 + b % 4 for b in range(B)], dtype=np.int32)
    refs = [_oracle_session(p, f_np).propose(int(cur_np[i]), n, 1.0, 8, 0)["logits"]
            for i, (f_np, _) in enumerate(feats)]
    tok = torch.empty((B, n), dtype=torch.int32, device="cuda")
    q = torch.empty((B, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((B, n, V), dtype=torch.float32, device="cuda")
    assert D.dflash_propose(sess, torch.from_numpy(cur_np).cuda(), n, 1.0, 8, 0, tok, q, lg) == [n] * B
    torch.cuda.synchronize()
    g_lg = lg.double().cpu().numpy()
    g_tok = tok.cpu().numpy()
    assert np.all(np.isfinite(g_lg))
    for b in range(B):
        ref = refs[b % 4]
        err = np.max(np.abs(g_lg[b] - ref))
        assert err <= TOL_LOGITS["bf16"], (b, err)
        check_tokens_for(cfg, g_tok[b], g_lg[b], ref, 1.0, 8, 0, b)
    D.dflash_device_status(p.model)
    for s in sess:
        D.dflash_close(s)


@pytest.mark.parametrize("T", [0.0, 0.8])
def test_batched_draw_on_a_32000_entry_vocabulary(D, T):
    """A batch of many rows over a 32000-entry vocabulary: the unembedding
    runs on 256-wide persistent tiles and the draw on 4096-entry chunks.  On
    the GPU's own logits every token is the oracle's Gumbel-max (or argmax)
    decision, q(token) is the oracle's softmax at the token, and verify
    against the kept log-sum-exp follows the oracle's verify; the block
    logits also follow the oracle's."""
    cfg = S.CONFIGS["small_bf16"].replace(vocab=32000, mask_token=31999)
    p = Pair(cfg)
    n, V, B = cfg.block_size - 1, cfg.vocab, 12
    sess, refs = [], []
    for b in range(B):
        f_np, f = p.feats(30 + 7 * b, seed=60 + b)
        s = D.dflash_open(p.model, max_ctx=512)
        D.dflash_committed(s, f, 0)
        sess.append(s)
        if b < 2:
            o = O.OracleSession(p.oracle, seq=b)
            o.committed(f_np, 0)
            refs.append(o)
    cur_np = (np.arange(B, dtype=np.int32) * 131) % V
    tok = torch.empty((B, n), dtype=torch.int32, device="cuda")
    q = torch.empty((B, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((B, n, V), dtype=torch.float32, device="cuda")
    assert D.dflash_propose(sess, torch.from_numpy(cur_np).cuda(), n, T, 41, 3, tok, q, lg) == [n] * B
    torch.cuda.synchronize()
    g_lg, g_tok, g_q = lg.double().cpu().numpy(), tok.cpu().numpy(), q.double().cpu().numpy()
    for b in range(B):
        check_tokens(g_tok[b], g_lg[b], T, 41, 3, b)
        if T > 0:
            for i in range(n):
                want = O.softmax(g_lg[b, i] / T)[g_tok[b, i]]
                assert abs(g_q[b, i] - want) <= 1e-5 * want + 1e-9, (b, i, g_q[b, i], want)
        else:
            assert np.all(g_q[b] == 1.0)
    for b, o in enumerate(refs):
        ref = o.propose(int(cur_np[b]), n, T, 41, 3)
        assert np.max(np.abs(g_lg[b] - ref["logits"])) <= TOL_LOGITS["bf16"]
        check_tokens_for(cfg, g_tok[b], g_lg[b], ref["logits"], T, 41, 3, b)
    # verify reads each session's kept log-sum-exp of the fused draw
    tl_np = S.make_target_logits(B, n + 1, V, g_tok.astype(np.int32), seed=9, std=2.0, boost=5.0)
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bon = torch.empty(B, dtype=torch.int32, device="cuda")
    D.dflash_verify(sess, torch.from_numpy(tl_np).cuda(), tok, n, T, 17, 3, acc, bon)
    torch.cuda.synchronize()
    a_g, b_g = acc.cpu().numpy(), bon.cpu().numpy()
    compared = sum(verify_parity((a_g[b], b_g[b]), tl_np[b], g_tok[b], g_lg[b], g_tok[b], T, T, 17, 3, b)
                   for b in range(B))
    assert compared >= B - 1, compared
    D.dflash_device_status(p.model)
    for s_ in sess:
        D.dflash_close(s_)


@pytest.mark.parametrize("intermediate", [1024, 12288])
def test_rows_do_not_depend_on_the_batch(D, intermediate):
    """A session's block logits are bit-identical whether it proposes alone
    or among 127 other sessions: the K order of every product depends on the
    weight shape only, so the 16-row and the 2048-row schedules (split
    clusters; persistent tiles 128 or 256 rows wide, with several K splits,
    and the one-split SwiGLU of a wide MLP) sum alike."""
    p = Pair(S.CONFIGS["small_bf16"].replace(intermediate=intermediate))
    cfg = p.cfg
    n = cfg.block_size - 1
    B = 128
    _, f = p.feats(48, seed=21)
    sess = []
    for b in range(B):
        s = D.dflash_open(p.model, max_ctx=128)
        D.dflash_committed(s, f[: 16 + (b % 32)], 0)
        D.dflash_flush([s])
        sess.append(s)
    cur = (torch.arange(B, dtype=torch.int32, device="cuda") * 7) % cfg.vocab
    tok = torch.empty((B, n), dtype=torch.int32, device="cuda")
    q = torch.empty((B, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((B, n, cfg.vocab), dtype=torch.float32, device="cuda")
    assert D.dflash_propose(sess, cur, n, 0.7, 5, 1, tok, q, lg) == [n] * B
    tok1 = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q1 = torch.empty((1, n), dtype=torch.float32, device="cuda")
    lg1 = torch.empty((1, n, cfg.vocab), dtype=torch.float32, device="cuda")
    for b in (0, 37, 127):
        # alone, the session is batch entry 0: same logits, tokens drawn with seq 0
        assert D.dflash_propose([sess[b]], cur[b:b + 1], n, 0.7, 5, 1, tok1, q1, lg1) == [n]
        torch.cuda.synchronize()
        assert torch.equal(lg1[0], lg[b]), float((lg1[0] - lg[b]).abs().max())
    D.dflash_device_status(p.model)
    for s in sess:
        D.dflash_close(s)


def test_sessions_called_back_to_back_keep_their_own_tables(D):
    """Six sessions with different context lengths propose one after another
    on one stream, twice round: each call's kernels must read that call's
    tables (work items, frontiers, cache maps), never the previous call's, so
    every proposal equals its own session's oracle."""
    p = Pair(S.CONFIGS["small_bf16"])
    cfg = p.cfg
    n = cfg.block_size - 1
    lens = [12, 300, 40, 190, 75, 260]
    sess, oss = [], []
    for b, L in enumerate(lens):
        f_np, f = p.feats(L, seed=40 + b)
        s = D.dflash_open(p.model, max_ctx=512)
        D.dflash_committed(s, f, 0)
        o = O.OracleSession(p.oracle)
        o.committed(f_np, 0)
        sess.append(s)
        oss.append(o)
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    lgs = [torch.empty((1, n, cfg.vocab), dtype=torch.float32, device="cuda") for _ in lens]
    for rnd in range(2):
        for b in range(len(lens)):
            cur = torch.tensor([(5 * b + rnd) % cfg.vocab], dtype=torch.int32, device="cuda")
            assert D.dflash_propose([sess[b]], cur, n, 0.0, 0, rnd, tok, q, lgs[b]) == [n]
        torch.cuda.synchronize()
        for b in range(len(lens)):
            ref = oss[b].propose((5 * b + rnd) % cfg.vocab, n, 0.0, 0, rnd)
            assert np.max(np.abs(lgs[b][0].double().cpu().numpy() - ref["logits"])) <= TOL_LOGITS["bf16"]
            oss[b].commit_block()
    D.dflash_device_status(p.model)
    for s in sess:
        D.dflash_close(s)


@pytest.mark.parametrize("rows", [37, 300])
def test_committed_taps_equals_concatenated_features(D, rows):
    """dflash_committed_taps (the target's taps in separate buffers, read in
    place) leaves the same cache and the same next proposal as
    dflash_committed with the concatenated rows: staged (37 rows) and
    flushed at the threshold (300 rows)."""
    p = Pair(S.CONFIGS["small_bf16"])
    cfg = p.cfg
    n, Ht, K = cfg.block_size - 1, cfg.target_hidden, cfg.n_taps
    _, f = p.feats(rows, seed=41)
    a = D.dflash_open(p.model, max_ctx=512)
    b = D.dflash_open(p.model, max_ctx=512)
    c = D.dflash_open(p.model, max_ctx=512)
    D.dflash_committed(a, f, 0)
    D.dflash_committed_taps(b, [f[:, k * Ht:(k + 1) * Ht] for k in range(K)], 0)          # one strided buffer
    D.dflash_committed_taps(c, [f[:, k * Ht:(k + 1) * Ht].contiguous() for k in range(K)], 0)  # K buffers
    assert D.dflash_session_state(b) == D.dflash_session_state(c) == D.dflash_session_state(a)
    outs = []
    for s in (a, b, c):
        tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
        q = torch.empty((1, n), dtype=torch.float32, device="cuda")
        lg = torch.empty((1, n, cfg.vocab), dtype=torch.float32, device="cuda")
        D.dflash_propose([s], torch.tensor([9], dtype=torch.int32, device="cuda"), n, 0.8, 3, 2, tok, q, lg)
        torch.cuda.synchronize()
        outs.append((tok.clone(), lg.clone(), [export_kv(D, s, cfg, l, 0, rows) for l in range(cfg.n_layers)]))
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0]) and torch.equal(o[1], outs[0][1])
        for (k0, v0), (k1, v1) in zip(outs[0][2], o[2]):
            assert np.array_equal(k0, k1) and np.array_equal(v0, v1)
    with pytest.raises(ValueError):
        D.dflash_committed_taps(a, [f[:, :Ht]] * (K - 1), rows)
    D.dflash_device_status(p.model)
    for s in (a, b, c):
        D.dflash_close(s)


def _propose_logits(D, model, cfg, feats_dev, first, max_tokens, cur=5, restored=0):
    s = D.dflash_open(model, restored_offset=restored, max_ctx=restored + len(feats_dev) + 64)
    D.dflash_committed(s, feats_dev, first)
    n = min(max_tokens, cfg.block_size - 1)
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((1, n, cfg.vocab), dtype=torch.float32, device="cuda")
    assert D.dflash_propose([s], torch.tensor([cur], dtype=torch.int32, device="cuda"), max_tokens, 0.0, 0, 0, tok,
                            q, lg) == [n]
    torch.cuda.synchronize()
    out = lg[0].double().cpu().numpy()
    D.dflash_close(s)
    return out


def test_causal_prefix_forward_on_gpu(D):
    """The mask-token shortcut on the GPU: for the causal tiny draft, drafting
    n + 1 rows gives rows 1..n of the full block's forward ("Ollama DFlash
    block-diffusion draft model in mlxrunner", Facts: exact for causal
    layers)."""
    p = Pair(S.CONFIGS["tiny_fp32"])
    _, f = p.feats(64, seed=71)
    full = _propose_logits(D, p.model, p.cfg, f, 0, p.cfg.block_size - 1)
    for k in (1, 3, 6):
        part = _propose_logits(D, p.model, p.cfg, f, 0, k)
        assert np.max(np.abs(part - full[:k])) <= 1e-6, k


def _windowed_block_logits(D, model, cfg, F, K, V):
    """Block logits of a windowed draft whose visible context (the W - 1 rows
    before F) holds the given K/V rows [L, Hkv, W - 1, d]."""
    s = D.dflash_open(model, restored_offset=F, max_ctx=F + 64)
    first = F - cfg.window + 1
    for l in range(cfg.n_layers):
        D.dflash_kv_import(s, l, first, cfg.window - 1, torch.from_numpy(K[l]).cuda().to(torch.bfloat16),
                           torch.from_numpy(V[l]).cuda().to(torch.bfloat16))
    n = cfg.block_size - 1
    tok = torch.empty((1, n), dtype=torch.int32, device="cuda")
    q = torch.empty((1, n), dtype=torch.float32, device="cuda")
    lg = torch.empty((1, n, cfg.vocab), dtype=torch.float32, device="cuda")
    assert D.dflash_propose([s], torch.tensor([5], dtype=torch.int32, device="cuda"), n, 0.0, 0, 0, tok, q,
                            lg) == [n]
    torch.cuda.synchronize()
    out = lg[0].double().cpu().numpy()
    D.dflash_close(s)
    return out


def test_block_depends_on_rope_offset_and_qkv_row_order_on_gpu(D):
    """The PR's two dependence tests on the GPU (mlxcel PR #1771: the tests
    that the block depends on RoPE and on the order of the fused q/k/v rows).
    The same visible context K/V read from a frontier 5 positions later
    changes the logits; so does a permutation of the fused projection's rows."""
    cfg = S.CONFIGS["small_laguna_bf16"]
    p = Pair(cfg)
    K = S.make_kv(cfg, cfg.window - 1, 75, "rope.k")
    V = S.make_kv(cfg, cfg.window - 1, 75, "rope.v")
    base = _windowed_block_logits(D, p.model, cfg, 100, K, V)
    again = _windowed_block_logits(D, p.model, cfg, 100, K, V)
    assert np.array_equal(base, again)
    shifted = _windowed_block_logits(D, p.model, cfg, 105, K, V)
    assert np.max(np.abs(base - shifted)) > 1e-2
    w = dict(p.w)
    qd, kd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    for l in range(cfg.n_layers):
        qkv = p.w[f"layers.{l}.w_qkv"]
        w[f"layers.{l}.w_qkv"] = np.ascontiguousarray(np.concatenate([qkv[qd:qd + kd], qkv[:qd], qkv[qd + kd:]]))
    perm = _windowed_block_logits(D, Pair(cfg, weights=w).model, cfg, 100, K, V)
    assert np.max(np.abs(base - perm)) > 1e-2


def test_rows_older_than_the_window_do_not_change_the_block_on_gpu(D):
    """Window W: context rows at positions <= F - W can be seen by no query
    of the block, so replacing their features leaves the logits bit for bit
    unchanged (mlxcel PR #1771: rows older than the window are dropped before
    aux_hidden_norms and fc)."""
    cfg = S.CONFIGS["small_laguna_bf16"]
    p = Pair(cfg)
    f_np, f = p.feats(300, seed=73)
    g_np = S.make_features(cfg, 300, seed=74, name="other")
    mixed = f_np.copy()
    F = 300
    mixed[: F - cfg.window + 1] = g_np[: F - cfg.window + 1]
    a = _propose_logits(D, p.model, cfg, f, 0, 7)
    b = _propose_logits(D, p.model, cfg, torch.from_numpy(mixed).cuda().to(torch.bfloat16), 0, 7)
    assert np.array_equal(a, b)
    mixed[F - cfg.window + 1] = g_np[F - cfg.window + 1]      # the oldest visible row does matter
    c = _propose_logits(D, p.model, cfg, torch.from_numpy(mixed).cuda().to(torch.bfloat16), 0, 7)
    assert not np.array_equal(a, c)


def test_committed_batch_flushes_together_and_equals_single_commits(D):
    """dflash_committed_batch: sessions that reach 256 held rows flush in one
    batched forward, sessions below it stage their rows, a restored prefix is
    skipped, and the caches and cursors equal those of one dflash_committed
    per session, bit for bit.  A gap in any session changes no session."""
    p = Pair(S.CONFIGS["small_bf16"])
    cfg = p.cfg
    n = cfg.block_size - 1
    f_np, f = p.feats(300, seed=80)
    offs = [0, 64, 128, 192, 256, 320]
    rows = [256, 100, 256, 300, 30, 256]
    held = [0, 0, 20, 0, 0, 5]
    single, batch = [], []
    for j in range(len(offs)):
        for group in (single, batch):
            s = D.dflash_open(p.model, restored_offset=offs[j], max_ctx=offs[j] + 600)
            if held[j]:
                D.dflash_committed(s, f[:held[j]], offs[j])
            if j % 2:   # an outstanding block that the flush must rewind
                D.dflash_propose([s], torch.tensor([3], dtype=torch.int32, device="cuda"), n, 0.0, 0, 0,
                                 torch.empty((1, n), dtype=torch.int32, device="cuda"),
                                 torch.empty((1, n), dtype=torch.float32, device="cuda"))
            group.append(s)
    # the batch call: each session's run starts where its held rows start
    feats = [f[:held[j] + rows[j]] for j in range(len(offs))]
    before = [D.dflash_session_state(s) for s in batch]
    bad_pos = [offs[j] for j in range(len(offs))]
    bad_pos[3] += 1 + held[3]                                   # session 3: a gap
    with pytest.raises(D.DFlashError) as e:
        D.dflash_committed_batch(batch, feats, bad_pos)
    assert e.value.status == D.DFLASH_ERR_CONTEXT_GAP
    assert [D.dflash_session_state(s) for s in batch] == before
    D.dflash_committed_batch(batch, feats, offs)
    for j, s in enumerate(single):
        D.dflash_committed(s, feats[j], offs[j])
    for a, b in zip(single, batch):
        assert D.dflash_session_state(a) == D.dflash_session_state(b)
    for j, (a, b) in enumerate(zip(single, batch)):
        F_, P_, _ = D.dflash_session_state(a)
        assert (P_ == 0) == (held[j] + rows[j] >= 256)
        if F_ == offs[j]:
            continue                # staged only: nothing in the cache yet
        for l in (0, cfg.n_layers - 1):
            ka, va = export_kv(D, a, cfg, l, offs[j], F_ - offs[j])
            kb, vb = export_kv(D, b, cfg, l, offs[j], F_ - offs[j])
            assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    # the staged rows (one batched copy for all staged sessions) flush to the
    # same caches as the rows each dflash_committed staged
    D.dflash_flush(single)
    D.dflash_flush(batch)
    for j, (a, b) in enumerate(zip(single, batch)):
        F_, P_, _ = D.dflash_session_state(a)
        assert D.dflash_session_state(b) == (F_, P_, _) and P_ == 0
        for l in (0, cfg.n_layers - 1):
            ka, va = export_kv(D, a, cfg, l, offs[j], F_ - offs[j])
            kb, vb = export_kv(D, b, cfg, l, offs[j], F_ - offs[j])
            assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    # the flushed rows equal the oracle's
    o = O.OracleSession(p.oracle, restored_offset=offs[0])
    o.committed(f_np[:256], offs[0])
    k, v = export_kv(D, batch[0], cfg, 1, 0, 256)
    assert_cache_close(k, np.stack([o.cache[s][0][1] for s in range(256)], axis=1))
    assert_cache_close(v, np.stack([o.cache[s][1][1] for s in range(256)], axis=1))
    D.dflash_device_status(p.model)
    for s in single + batch:
        D.dflash_close(s)
