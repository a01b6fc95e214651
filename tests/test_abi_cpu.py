"""The C-ABI library builds, loads and exports every entry point that
include/*.h declares, and its host-side validation answers without a GPU
(no compute calls are made here)."""
import ctypes as C
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _by_path(name, rel):
    spec = importlib.util.spec_from_file_location(name, os.path.join(ROOT, rel))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


# loaded by path so that the package (which loads the library) is not imported first
_build = _by_path("_dflash_build", "block_diffusion_speculative_flush_gb300/build.py")
_abi = _by_path("_dflash_abi", "block_diffusion_speculative_flush_gb300/_abi.py")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _abi.load()


def test_every_header_symbol_is_exported(lib):
    names = _abi.header_symbols()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(_abi.SIGNATURES)   # the binding declares exactly the header


def test_version_and_error_string(lib):
    assert lib.dflash_version() == 200
    assert isinstance(lib.dflash_last_error(), bytes)


def _cfg(**kw):
    base = dict(dtype=_abi.DFLASH_DTYPE_BF16, n_taps=5, target_hidden=256, hidden=256, n_layers=2, n_q_heads=4,
                n_kv_heads=2, head_dim=64, intermediate=512, vocab=32, block_size=8, mask_token=31, window=0,
                causal_block=0, gated_attention=0, flags=0, rope_theta=1e6, rms_eps=1e-6)
    base.update(kw)
    return _abi.dflash_config(**base)


@pytest.mark.parametrize("bad,code", [
    (dict(block_size=1), _abi.DFLASH_ERR_SHAPE),
    (dict(block_size=513), _abi.DFLASH_ERR_SHAPE),
    (dict(window=1), _abi.DFLASH_ERR_SHAPE),
    (dict(window=(1 << 20) + 1), _abi.DFLASH_ERR_SHAPE),
    (dict(n_q_heads=5), _abi.DFLASH_ERR_SHAPE),
    (dict(head_dim=96), _abi.DFLASH_ERR_SHAPE),
    (dict(mask_token=32), _abi.DFLASH_ERR_SHAPE),
    (dict(hidden=200), _abi.DFLASH_ERR_SHAPE),
    (dict(dtype=7), _abi.DFLASH_ERR_INVALID_ARG),
    (dict(causal_block=2), _abi.DFLASH_ERR_INVALID_ARG),
])
def test_config_bounds_are_refused(lib, bad, code):
    """The drafter config is untrusted (Laguna PR): out-of-range fields are
    refused with a status before any device work."""
    c = _cfg(**bad)
    w = _abi.dflash_weights()
    out = C.c_void_p()
    assert lib.dflash_model_create(C.byref(c), C.byref(w), C.byref(out)) == code
    assert out.value is None
    assert len(lib.dflash_last_error()) > 0


def test_null_arguments_are_refused(lib):
    assert lib.dflash_draft_limit(None) == _abi.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_committed(None, None, 0, 0, 0) == _abi.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_committed_taps(None, None, 0, 0, 0) == _abi.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_flush(None, 1) == _abi.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_close(None) == _abi.DFLASH_ERR_INVALID_ARG
    c = _cfg()
    out = C.c_void_p()
    assert lib.dflash_model_create(C.byref(c), None, C.byref(out)) == _abi.DFLASH_ERR_INVALID_ARG
    w = _abi.dflash_weights()   # all weights null
    assert lib.dflash_model_create(C.byref(c), C.byref(w), C.byref(out)) == _abi.DFLASH_ERR_INVALID_ARG


def test_exactness_summary_is_host_code_that_agrees_with_the_oracle(lib):
    """dflash_exactness_summarize reduces row records on the host (no GPU):
    the same gate and counts as the probe oracle on the same records."""
    import numpy as np

    from oracle.target_oracle import exactness_rows, exactness_summary
    rng = np.random.default_rng(4)
    block = rng.standard_normal((5, 40)).astype(np.float32)
    chain = block.copy()
    chain[1, 3] += 1.0
    chain[3] = block[3, ::-1]
    for first_differs in (False, True):
        if first_differs:
            chain[0, 0] = -chain[0, 0]
        rows = exactness_rows(block, chain)
        recs = (_abi.dflash_exactness_row * 5)()
        for rec, r in zip(recs, rows):
            rec.differing_bytes = r["differing_bytes"]
            rec.block_top[:] = r["block_top"]
            rec.chain_top[:] = r["chain_top"]
            rec.block_val[:] = r["block_val"]
            rec.chain_val[:] = r["chain_val"]
        s = _abi.dflash_exactness_summary()
        assert lib.dflash_exactness_summarize(recs, 5, C.byref(s)) == 0
        assert {k: getattr(s, k) for k, _ in s._fields_} == exactness_summary(rows)
    assert lib.dflash_exactness_summarize(None, 5, C.byref(s)) == _abi.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_logits_compare(None, None, 1, 1, None, None) == _abi.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_target_exactness_probe(None, None, 1, 0, None, None, None, None) == _abi.DFLASH_ERR_INVALID_ARG


def test_target_create_refuses_bad_shapes_and_weights_on_the_host(lib):
    cfg = _abi.dflash_target_config(hidden=256, n_heads=4, head_dim=64, intermediate=512, vocab=32, n_layers=1,
                                    rope_theta=1e6, rms_eps=1e-6)
    out = C.c_void_p()
    layers = (_abi.dflash_target_layer * 1)()
    w = _abi.dflash_target_weights(embed=16, unembed=16, final_norm=16, layers=layers)
    # a null layer weight and a misaligned one are refused before anything is allocated
    assert lib.dflash_target_create(C.byref(cfg), C.byref(w), 64, None, C.byref(out)) == _abi.DFLASH_ERR_INVALID_ARG
    for name in ("n1", "wq", "wk", "wv", "wo", "n2", "wg", "wu", "wd"):
        setattr(layers[0], name, 4096)
    layers[0].wo = 4100
    assert lib.dflash_target_create(C.byref(cfg), C.byref(w), 64, None, C.byref(out)) == _abi.DFLASH_ERR_INVALID_ARG
    w.unembed = 20
    assert lib.dflash_target_create(C.byref(cfg), C.byref(w), 64, None, C.byref(out)) == _abi.DFLASH_ERR_INVALID_ARG
    for field, bad in (("head_dim", 66), ("head_dim", 256), ("hidden", 258), ("n_layers", 0)):
        c2 = _abi.dflash_target_config.from_buffer_copy(cfg)
        setattr(c2, field, bad)
        assert lib.dflash_target_create(C.byref(c2), C.byref(w), 64, None, C.byref(out)) == _abi.DFLASH_ERR_SHAPE


def test_binding_refuses_buffers_the_library_would_overrun(lib):
    """The Python binding checks dtype, contiguity, device and size of every
    tensor it hands to the library before the call (host-side; no GPU)."""
    import torch

    import block_diffusion_speculative_flush_gb300 as D
    import synthetic as S
    cfg = S.CONFIGS["tiny_fp32"]
    sess = D.Session(0, D.Model(0, cfg, {}, None))
    n = cfg.block_size - 1
    cur = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError):   # host tensors
        D.dflash_propose([sess], cur, n, 0.0, 0, 0, torch.zeros((1, n), dtype=torch.int32),
                         torch.zeros((1, n)))
    with pytest.raises(ValueError):
        D.dflash_verify([sess], torch.zeros((1, n + 1, cfg.vocab)), torch.zeros((1, n), dtype=torch.int32), n,
                        0.0, 0, 0, torch.zeros(1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError):
        D.dflash_committed(sess, torch.zeros((2, cfg.feature_width + 1)), 0)
