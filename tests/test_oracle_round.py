"""Pins of the oracle's draft round against the invariants the pages fix.
CPU only; sizes are the tiny fp32 draft and small variants of it."""
import numpy as np
import pytest

import synthetic as S
from oracle import dflash_oracle as O
from oracle.target_oracle import OracleTarget
from synthetic.target import TARGET_TINY, make_target_weights

TINY = S.CONFIGS["tiny_fp32"]


@pytest.fixture(scope="module")
def tiny():
    return O.OracleDraft(TINY, S.make_weights(TINY, seed=0))


def _session(draft, n_ctx=64, seed=0, **kw):
    s = O.OracleSession(draft, **kw)
    s.committed(S.make_features(draft.cfg, n_ctx, seed=seed), 0)
    return s


# -- dflash.go draftLimit / propose: n = min(maxTokens, blockSize-1) -------

def test_draft_limit_and_block_rows(tiny):
    s = _session(tiny)
    assert s.draft_limit == TINY.block_size - 1 == 7
    for max_tokens, n in [(100, 7), (7, 7), (3, 3), (1, 1)]:
        out = s.propose(5, max_tokens)
        assert out["n"] == n and len(out["tokens"]) == n and out["logits"].shape == (n, TINY.vocab)
        assert out["hidden"].shape[0] == n + 1          # anchor row + n mask rows
    assert s.propose(5, 0) is None and s.propose(5, -2) is None
    empty = O.OracleSession(tiny)
    assert empty.propose(5, 4) is None                  # nothing committed yet


def test_anchor_row_is_unused(tiny):
    """Row i predicts its own position: the logits are rows 1..n of the
    forward, and the anchor's own output never reaches them."""
    s = _session(tiny)
    out = s.propose(3, 7)
    h = out["hidden"]
    np.testing.assert_array_equal(out["logits"], tiny.unembed(h[1:]))


def test_causal_prefix_forward_is_exact(tiny):
    """Mask-token shortcut: drafting only n+1 rows reproduces rows 0..n of the
    full-block forward bit for bit when the draft is causal in the block."""
    s = _session(tiny)
    s.flush()
    ctx = s.context()
    full = tiny.block_forward([3] + [TINY.mask_token] * (TINY.block_size - 1), s.F, ctx)
    for n in [1, 3, 6]:
        part = tiny.block_forward([3] + [TINY.mask_token] * n, s.F, ctx)
        assert np.array_equal(part, full[:n + 1])


def test_bidirectional_prefix_forward_differs():
    cfg = TINY.replace(causal_block=False)
    d = O.OracleDraft(cfg, S.make_weights(cfg, seed=0))
    s = _session(d)
    s.flush()
    ctx = s.context()
    full = d.block_forward([3] + [cfg.mask_token] * 7, s.F, ctx)
    part = d.block_forward([3] + [cfg.mask_token] * 3, s.F, ctx)
    assert not np.array_equal(part, full[:4])


def test_block_depends_on_rope_offset(tiny):
    """Laguna PR test draft_block_depends_on_rope: the same context read at a
    shifted frontier changes the block's logits."""
    s = _session(tiny)
    s.flush()
    ctx = s.context()
    toks = [3] + [TINY.mask_token] * 4
    h0 = tiny.block_forward(toks, s.F, ctx)
    shifted = dict(ctx, pos=ctx["pos"] + 5)
    h1 = tiny.block_forward(toks, s.F + 5, shifted)
    assert not np.allclose(tiny.unembed(h0[1:]), tiny.unembed(h1[1:]), atol=1e-6)


def test_permuting_fused_qkv_rows_changes_logits():
    """Laguna PR test: permuting the fused q/k/v rows changes the logits."""
    w = S.make_weights(TINY, seed=0)
    d0 = O.OracleDraft(TINY, w)
    w2 = dict(w)
    qkv = w["layers.0.w_qkv"]
    qd, kd = TINY.n_q_heads * TINY.head_dim, TINY.n_kv_heads * TINY.head_dim
    w2["layers.0.w_qkv"] = np.concatenate([qkv[qd:qd + kd], qkv[:qd], qkv[qd + kd:]])  # k|q|v
    d1 = O.OracleDraft(TINY, w2)
    feats = S.make_features(TINY, 16)
    out = []
    for d in (d0, d1):
        s = O.OracleSession(d)
        s.committed(feats, 0)
        out.append(s.propose(3, 7)["logits"])
    assert not np.allclose(out[0], out[1], atol=1e-6)


# -- context path --------------------------------------------------------

def test_context_rows_are_independent(tiny):
    """A context entry at slot S derives only from the features at S: flushing
    rows one run at a time equals one combined flush, bit for bit (Laguna PR
    test: incremental appends draft exactly like one combined append)."""
    feats = S.make_features(TINY, 40, seed=3)
    a = O.OracleSession(tiny)
    a.committed(feats, 0)
    a.flush()
    b = O.OracleSession(tiny)
    for lo, hi in [(0, 1), (1, 7), (7, 20), (20, 40)]:
        b.committed(feats[lo:hi], lo)
        b.flush()
    assert a.F == b.F == 40
    for s in range(40):
        assert np.array_equal(a.cache[s][0], b.cache[s][0]) and np.array_equal(a.cache[s][1], b.cache[s][1])


def test_each_tap_is_normed_on_its_own():
    """aux_hidden_norms: scaling one tap's features leaves the context row
    unchanged (one RMSNorm per tap); with eps = 0 the norm is scale-free."""
    cfg = TINY.replace(rms_eps=0.0)
    d = O.OracleDraft(cfg, S.make_weights(cfg, seed=0))
    f = S.make_features(cfg, 3, seed=4).astype(np.float64)
    g = f.copy()
    g[:, cfg.target_hidden:2 * cfg.target_hidden] *= 8.0      # tap 1 scaled by a power of two
    np.testing.assert_array_equal(d.context_hidden(f), d.context_hidden(g))


def test_context_kv_rope_uses_the_slot(tiny):
    """The context K at slot S is the slot-0 K turned by S."""
    f = S.make_features(TINY, 1, seed=5)
    K0, V0 = tiny.context_kv(f, [0])
    K9, V9 = tiny.context_kv(f, [9])
    cfg32 = lambda x: x.astype(np.float32).astype(np.float64)
    for l in range(TINY.n_layers):
        np.testing.assert_allclose(K9[l], cfg32(O.rope(K0[l], 9.0, TINY.rope_theta)), rtol=0, atol=2e-6)
        assert np.array_equal(V0[l], V9[l])


def test_window_drops_unseeable_context():
    """Laguna-style window: rows older than the window never change the block
    (they are dropped before the fc); a window wider than everything equals
    full attention."""
    cfg = TINY.replace(window=16, causal_block=False)
    w = S.make_weights(cfg, seed=0)
    feats = S.make_features(cfg, 60, seed=6)
    d = O.OracleDraft(cfg, w)
    s1 = O.OracleSession(d)
    s1.committed(feats, 0)
    o1 = s1.propose(3, 7)
    # different features for every row no block query can see (r <= F - W)
    feats2 = feats.copy()
    feats2[:60 - 16 + 1] = S.make_features(cfg, 45, seed=7)
    s2 = O.OracleSession(d)
    s2.committed(feats2, 0)
    o2 = s2.propose(3, 7)
    assert np.array_equal(o1["logits"], o2["logits"])
    assert min(s1.cache) == 60 - 16 + 1        # only W-1 rows kept
    wide = cfg.replace(window=1 << 20)
    full = cfg.replace(window=0)
    outs = []
    for c in (wide, full):
        s = O.OracleSession(O.OracleDraft(c, w))
        s.committed(feats, 0)
        outs.append(s.propose(3, 7)["logits"])
    assert np.array_equal(outs[0], outs[1])


def test_zero_gate_halves_attention_output():
    """Per-head sigmoid gate: W_g = 0 gives gate 0.5 on every head, which is
    exactly the ungated draft with W_o halved."""
    base = S.CONFIGS["small_laguna_bf16"].replace(n_layers=1, window=0)
    gated = base
    ungated = base.replace(gated_attention=False)
    w = S.make_weights(gated, seed=0)
    w["layers.0.w_g"] = np.zeros_like(w["layers.0.w_g"])
    wu = {k: v for k, v in w.items() if k != "layers.0.w_g"}
    wu["layers.0.w_o"] = w["layers.0.w_o"] * 0.5
    feats = S.make_features(gated, 10, seed=8)
    outs = []
    for c, ww in ((gated, w), (ungated, wu)):
        s = O.OracleSession(O.OracleDraft(c, ww))
        s.committed(feats, 0)
        outs.append(s.propose(3, 5)["hidden"])
    assert np.array_equal(outs[0], outs[1])


# -- session state machine (dflash.go) -------------------------------------

def test_gap_is_refused_and_prefix_skipped(tiny):
    s = O.OracleSession(tiny)
    f = S.make_features(TINY, 10, seed=9)
    s.committed(f, 0)
    assert (s.F, s.P) == (0, 10)
    with pytest.raises(O.ContextGap):
        s.committed(f[:2], 11)
    assert (s.F, s.P) == (0, 10)                          # nothing changed
    s.committed(f[5:10], 5)                              # fully restored: skipped
    assert s.P == 10
    g = S.make_features(TINY, 6, seed=10)
    s.committed(g, 8)                                    # rows 8, 9 held; 10..13 new
    assert s.P == 14
    s.flush()
    assert (s.F, s.P) == (14, 0)
    # the held slots keep the first run's features
    ref = O.OracleSession(tiny)
    ref.committed(np.concatenate([f, g[2:]]), 0)
    ref.flush()
    for k in range(14):
        assert np.array_equal(s.cache[k][0], ref.cache[k][0])


def test_restored_offset_syncs_the_session(tiny):
    s = O.OracleSession(tiny, restored_offset=20)
    assert s.F == 20
    s.committed(S.make_features(TINY, 25, seed=1), 0)     # rows 0..19 restored
    assert s.P == 5
    with pytest.raises(O.ContextGap):
        O.OracleSession(tiny, restored_offset=3).committed(S.make_features(TINY, 2), 4)


def test_pending_rows_flush_at_256(tiny):
    s = O.OracleSession(tiny)
    f = S.make_features(TINY, 300, seed=2)
    s.committed(f[:255], 0)
    assert (s.F, s.P) == (0, 255)
    s.committed(f[255:256], 255)
    assert (s.F, s.P) == (256, 0)
    s.committed(f[256:300], 256)
    assert (s.F, s.P) == (256, 44)


def test_propose_takes_pending_then_rewind_restores(tiny):
    """Rewind then flush equals never having drafted: the cache rows below the
    frontier and the cursors are bit-identical (dflash.go commitBlock)."""
    f = S.make_features(TINY, 30, seed=3)
    a = O.OracleSession(tiny)
    a.committed(f[:20], 0)
    out = a.propose(4, 7)
    assert (a.F, a.P, a.block_outstanding) == (20, 0, True)
    assert out is not None
    a.committed(f[20:30], 20)
    a.flush()
    assert (a.F, a.P, a.block_outstanding) == (30, 0, False)
    b = O.OracleSession(tiny)
    b.committed(f, 0)
    b.flush()
    assert sorted(a.cache) == sorted(b.cache) == list(range(30))
    for k in range(30):
        assert np.array_equal(a.cache[k][0], b.cache[k][0]) and np.array_equal(a.cache[k][1], b.cache[k][1])


# -- whole round against the synthetic target --------------------------------

def _speculative_run(draft, target, prompt, n_new, forced=None, check=None):
    """Greedy speculative decoding: propose, verify on the target's logits,
    commit [current, accepted] with their taps, continue from the bonus."""
    target.reset()
    logits, taps = target.forward(prompt, 0)
    sess = O.OracleSession(draft)
    sess.committed(taps, 0)
    out = [int(np.argmax(logits[-1]))]
    pos = len(prompt)
    rnd = 0
    while len(out) < n_new:
        current = out[-1]
        prop = sess.propose(current, draft.cfg.block_size - 1)
        d = list(prop["tokens"])
        k = None
        if forced is not None:
            d, k = forced(rnd, len(out), len(d))
        tl, tt = target.forward([current] + d, pos)
        a, b = sess.verify(tl, d, 0.0)
        if check is not None:
            check(rnd, len(out), a, b, k)
        target.trim(pos + a + 1)
        sess.committed(tt[:a + 1], pos)
        out += d[:a] + [b]
        pos += a + 1
        rnd += 1
    return out[:n_new], sess


def test_greedy_speculative_equals_greedy_decode(tiny):
    """Speculative output with the real draft equals plain greedy decoding of
    the target, token for token, over 128 tokens."""
    tgt = OracleTarget(make_target_weights(1), TARGET_TINY)
    prompt = list(S.rng_for(0, "prompt").integers(0, 32, size=8))
    ref = tgt.greedy_decode(prompt, 128)
    out, sess = _speculative_run(tiny, tgt, prompt, 128)
    assert out == ref
    assert sess.stats["rounds"] > 0 and sess.stats["proposed"] == 7 * sess.stats["rounds"]


def test_forced_accept_lengths_keep_greedy_output(tiny):
    """Laguna PR greedy_invariant_with_forced_rejections: a drafter that forces
    accept lengths 0, 1, 2 and full; each round must accept exactly the forced
    length with the bonus sitting at the reference index."""
    tgt = OracleTarget(make_target_weights(1), TARGET_TINY)
    prompt = list(S.rng_for(0, "prompt").integers(0, 32, size=8))
    ref = tgt.greedy_decode(prompt, 200)
    plan = [0, 1, 2, 7]

    def forced(rnd, t, n):
        k = plan[rnd % len(plan)]
        d = [ref[t + j] for j in range(min(k, n))]
        if k < n:
            d.append((ref[t + k] + 1) % 32)              # a sure rejection
        d += [0] * (n - len(d))
        return d, min(k, n)

    def check(rnd, t, a, b, k):
        assert a == k
        assert b == ref[t + a]

    out, _ = _speculative_run(tiny, tgt, prompt, 128, forced=forced, check=check)
    assert out == ref[:128]
