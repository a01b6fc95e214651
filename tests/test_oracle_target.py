"""Pins of the target oracle (oracle/target_oracle.py) against facts other
than itself: an independent torch float64 build of the same decoder, RoPE
and attention special cases, and IEEE-754 byte counts worked by hand and a
brute-force top-two for the block-versus-chain probe."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synthetic as S
from oracle.target_oracle import OracleTarget, exactness_rows, exactness_summary
from synthetic.target import TARGET_TINY, TargetShape, make_target_weights


def _torch_forward(w, shape, tokens):
    """The whole sequence at once: torch's RMSNorm, RoPE as a complex
    rotation of (x_j, x_{j+d/2}), torch's causal scaled-dot-product attention,
    SwiGLU.  Returns (logits [T,V], taps [T,(2L+1)H]) in float64."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    T, H, nh, d = len(tokens), shape.hidden, shape.n_heads, shape.head_dim
    half = d // 2
    pos = torch.arange(T, dtype=torch.float64)
    freq = shape.rope_theta ** (-torch.arange(half, dtype=torch.float64) * 2.0 / d)
    rot = torch.polar(torch.ones(T, half, dtype=torch.float64), pos[:, None] * freq[None, :])  # [T, half]

    def rope(x):  # x [T, nh, d]
        z = torch.complex(x[..., :half], x[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    x = t(w["embed"])[torch.tensor(tokens)]
    taps = [x]
    for lw in w["layers"]:
        y = F.rms_norm(x, (H,), weight=t(lw["n1"]), eps=shape.rms_eps)
        q = rope(F.linear(y, t(lw["wq"])).view(T, nh, d)).transpose(0, 1)
        k = rope(F.linear(y, t(lw["wk"])).view(T, nh, d)).transpose(0, 1)
        v = F.linear(y, t(lw["wv"])).view(T, nh, d).transpose(0, 1)
        o = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True)[0]
        x = x + F.linear(o.transpose(0, 1).reshape(T, nh * d), t(lw["wo"]))
        taps.append(x)
        y = F.rms_norm(x, (H,), weight=t(lw["n2"]), eps=shape.rms_eps)
        x = x + F.linear(F.silu(F.linear(y, t(lw["wg"]))) * F.linear(y, t(lw["wu"])), t(lw["wd"]))
        taps.append(x)
    z = F.rms_norm(x, (H,), weight=t(w["final_norm"]), eps=shape.rms_eps)
    return F.linear(z, t(w["unembed"])).numpy(), torch.cat(taps, dim=-1).numpy()


@pytest.mark.parametrize("shape", [TARGET_TINY, TargetShape(hidden=96, n_heads=3, head_dim=16, intermediate=160,
                                                             vocab=50, n_layers=3, rope_theta=1e4)])
def test_target_oracle_equals_an_independent_torch_build(shape):
    w = make_target_weights(3, shape)
    tokens = [int(x) for x in S.rng_for(1, "tokens").integers(0, shape.vocab, size=23)]
    ref_l, ref_t = _torch_forward(w, shape, tokens)
    tgt = OracleTarget(w, shape)
    l0, t0 = tgt.forward(tokens[:9], 0)          # a prompt, then a verify block, then one row
    l1, t1 = tgt.forward(tokens[9:22], 9)
    l2, t2 = tgt.forward(tokens[22:], 22)
    lg, tp = np.concatenate([l0, l1, l2]), np.concatenate([t0, t1, t2])
    assert lg.shape == (23, shape.vocab) and tp.shape == (23, shape.n_taps * shape.hidden)
    # the oracle returns fp32 outputs of float64 arithmetic
    assert np.allclose(lg, ref_l, rtol=2e-7, atol=1e-6)
    assert np.allclose(tp, ref_t, rtol=2e-7, atol=1e-6)


def test_target_trim_then_forward_recomputes_the_same_rows():
    """A rejected verify block is trimmed; re-running the accepted rows and a
    different continuation gives what a fresh decode gives."""
    w = make_target_weights(1)
    a = OracleTarget(w, TARGET_TINY)
    a.forward([1, 2, 3, 4], 0)
    a.forward([5, 6, 7, 8, 9], 4)
    a.trim(6)
    la, ta = a.forward([11, 12], 6)
    b = OracleTarget(w, TARGET_TINY)
    b.forward([1, 2, 3, 4, 5, 6], 0)
    lb, tb = b.forward([11, 12], 6)
    assert np.array_equal(la, lb) and np.array_equal(ta, tb)
    with pytest.raises(ValueError):
        a.trim(9)
    with pytest.raises(ValueError):
        a.forward([1], 3)


def test_target_first_position_attends_only_to_itself():
    """At position 0 RoPE is the identity and the one key gets weight 1, so the
    first attention tap is embed + W_o · W_v · RMSNorm(embed)."""
    w = make_target_weights(2)
    s = TARGET_TINY
    _, taps = OracleTarget(w, s).forward([7], 0)
    e = w["embed"][7]
    L0 = w["layers"][0]
    y = e / np.sqrt(np.mean(e * e) + s.rms_eps) * L0["n1"]
    want = e + L0["wo"] @ (L0["wv"] @ y)
    assert np.allclose(taps[0, :s.hidden], e.astype(np.float32))
    assert np.allclose(taps[0, s.hidden:2 * s.hidden], want, rtol=1e-6, atol=1e-6)


# -- block-versus-chain probe ---------------------------------------------------

def _f32(*v):
    return np.array([v], dtype=np.float32)


@pytest.mark.parametrize("a,b,nbytes", [
    (1.0, 1.0, 0),
    (1.0, float(np.nextafter(np.float32(1.0), np.float32(2.0))), 1),   # 0x3F800000 / 0x3F800001
    (1.0, -1.0, 1),                                                    # 0x3F800000 / 0xBF800000
    (1.0, 2.0, 2),                                                     # 0x3F800000 / 0x40000000
    (0.0, -0.0, 1),                                                    # 0x00000000 / 0x80000000
    (0.5, 3.0, 2),                                                     # 0x3F000000 / 0x40400000
])
def test_probe_counts_differing_bytes_of_the_fp32_encoding(a, b, nbytes):
    r = exactness_rows(_f32(a, 0.25), _f32(b, 0.25))[0]
    assert r["differing_bytes"] == nbytes


def test_probe_top_two_with_ties_and_nan():
    r = exactness_rows(_f32(5, 7, 7, 1), _f32(5, 7, 8, 1))[0]
    assert r["block_top"] == [1, 2] and r["block_val"] == [7.0, 7.0]       # a tie: margin 0, lower id first
    assert r["chain_top"] == [2, 1] and r["chain_val"] == [8.0, 7.0]
    r = exactness_rows(_f32(np.nan, 3, 3), _f32(np.nan, 3, 2))[0]
    assert r["block_top"] == [1, 2] and r["chain_top"] == [1, 2]


def test_probe_top_two_equals_brute_force():
    rng = np.random.default_rng(0)
    x = rng.integers(-3, 4, size=(50, 9)).astype(np.float32)   # many ties
    rows = exactness_rows(x, x)
    for row, r in zip(x, rows):
        beats = lambda i, j: row[i] > row[j] or (row[i] == row[j] and i < j)
        first = next(i for i in range(9) if all(i == j or beats(i, j) for j in range(9)))
        rest = [i for i in range(9) if i != first]
        second = next(i for i in rest if all(i == j or beats(i, j) for j in rest))
        assert r["block_top"] == [first, second] == r["chain_top"]
        assert r["differing_bytes"] == 0


def test_probe_gate_reads_only_the_first_position():
    a = np.zeros((3, 4), dtype=np.float32)
    b = a.copy()
    b[2, 1] = 1.0                                          # a later row differs and disagrees
    s = exactness_summary(exactness_rows(a, b))
    assert s == dict(rows=3, differing_bytes=2, first_row_differing_bytes=0, disagreements=1, allows=1)
    b[0, 3] = -0.0
    s = exactness_summary(exactness_rows(a, b))
    assert s["allows"] == 0 and s["first_row_differing_bytes"] == 1 and s["disagreements"] == 1
