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
    assert lib.dflash_version() == 100
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
    assert lib.dflash_flush(None, 1) == _abi.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_close(None) == _abi.DFLASH_ERR_INVALID_ARG
    c = _cfg()
    out = C.c_void_p()
    assert lib.dflash_model_create(C.byref(c), None, C.byref(out)) == _abi.DFLASH_ERR_INVALID_ARG
    w = _abi.dflash_weights()   # all weights null
    assert lib.dflash_model_create(C.byref(c), C.byref(w), C.byref(out)) == _abi.DFLASH_ERR_INVALID_ARG
