"""ctypes declarations of include/dflash.h (argument marshalling only)."""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash.so")

DFLASH_OK = 0
DFLASH_ERR_INVALID_ARG = -1
DFLASH_ERR_SHAPE = -2
DFLASH_ERR_CONTEXT_GAP = -3
DFLASH_ERR_CAPACITY = -4
DFLASH_ERR_CUDA = -5
DFLASH_ERR_OOM = -6
DFLASH_ERR_STATE = -7
DFLASH_ERR_DEVICE = -8

DFLASH_DTYPE_F32 = 0
DFLASH_DTYPE_BF16 = 1
DFLASH_PENDING_FLUSH_TOKENS = 256
DFLASH_FLAG_SIMT_GEMM = 1
DFLASH_VARIANT_DFLASH = 0
DFLASH_VARIANT_DFLASH2 = 1
DFLASH2_DEPTH = 7


class dflash_config(C.Structure):
    _fields_ = [
        ("dtype", C.c_int32), ("n_taps", C.c_int32), ("target_hidden", C.c_int32), ("hidden", C.c_int32),
        ("n_layers", C.c_int32), ("n_q_heads", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
        ("intermediate", C.c_int32), ("vocab", C.c_int32), ("block_size", C.c_int32), ("mask_token", C.c_int32),
        ("window", C.c_int32), ("causal_block", C.c_int32), ("gated_attention", C.c_int32), ("flags", C.c_uint32),
        ("rope_theta", C.c_float), ("rms_eps", C.c_float),
        ("variant", C.c_int32), ("conv_taps", C.c_int32), ("sel_rank", C.c_int32), ("sel_candidates", C.c_int32),
    ]


class dflash_layer_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("in_norm", "w_qkv", "q_norm", "k_norm", "w_g", "w_o", "post_norm", "w_gate", "w_up", "w_down",
                 "conv_norm", "w_dc")]


class dflash_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("aux_norms", "w_fc", "hidden_norm", "final_norm", "embed", "unembed")] + \
               [("layers", C.POINTER(dflash_layer_weights)), ("sel_prev", C.c_void_p), ("sel_next", C.c_void_p)]


class dflash_counters(C.Structure):
    _fields_ = [("rounds", C.c_int64), ("proposed", C.c_int64), ("accepted", C.c_int64),
                ("flushes", C.c_int64), ("flushed_rows", C.c_int64)]


class dflash_kernel_time(C.Structure):
    _fields_ = [("name", C.c_char * 24), ("launches", C.c_int64), ("total_ms", C.c_double),
                ("bytes", C.c_double), ("flops", C.c_double)]


class dflash_target_config(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_heads", C.c_int32), ("head_dim", C.c_int32), ("intermediate", C.c_int32),
                ("vocab", C.c_int32), ("n_layers", C.c_int32), ("rope_theta", C.c_float), ("rms_eps", C.c_float)]


class dflash_target_layer(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("n1", "wq", "wk", "wv", "wo", "n2", "wg", "wu", "wd")]


class dflash_target_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("unembed", C.c_void_p), ("final_norm", C.c_void_p),
                ("layers", C.POINTER(dflash_target_layer))]


class dflash_exactness_row(C.Structure):
    _fields_ = [("differing_bytes", C.c_int32), ("block_top", C.c_int32 * 2), ("chain_top", C.c_int32 * 2),
                ("block_val", C.c_float * 2), ("chain_val", C.c_float * 2)]


class dflash_exactness_summary(C.Structure):
    _fields_ = [("rows", C.c_int64), ("differing_bytes", C.c_int64), ("first_row_differing_bytes", C.c_int64),
                ("disagreements", C.c_int32), ("allows", C.c_int32)]


P = C.c_void_p
SessArr = C.POINTER(C.c_void_p)

# name -> (restype, argtypes)
SIGNATURES = {
    "dflash_last_error": (C.c_char_p, []),
    "dflash_version": (C.c_int, []),
    "dflash_model_create": (C.c_int, [C.POINTER(dflash_config), C.POINTER(dflash_weights), C.POINTER(C.c_void_p)]),
    "dflash_model_destroy": (C.c_int, [P]),
    "dflash_draft_limit": (C.c_int, [P]),
    "dflash_device_status": (C.c_int, [P]),
    "dflash_open": (C.c_int, [P, C.c_int64, C.c_int64, P, C.POINTER(C.c_void_p)]),
    "dflash_committed": (C.c_int, [P, P, C.c_int64, C.c_int32, C.c_int64]),
    "dflash_committed_taps": (C.c_int, [P, C.POINTER(C.c_void_p), C.c_int64, C.c_int32, C.c_int64]),
    "dflash_committed_batch": (C.c_int, [P, C.c_int32, C.POINTER(C.c_void_p), C.c_int64, C.POINTER(C.c_int32),
                                         C.POINTER(C.c_int64)]),
    "dflash_flush": (C.c_int, [SessArr, C.c_int32]),
    "dflash_settle": (C.c_int, [P]),
    "dflash_commit_block": (C.c_int, [SessArr, C.c_int32]),
    "dflash_propose": (C.c_int, [SessArr, C.c_int32, P, C.c_int32, C.c_float, C.c_uint64, C.c_uint64, P, P, P,
                                 C.POINTER(C.c_int32)]),
    "dflash_verify": (C.c_int, [SessArr, C.c_int32, P, C.c_int32, P, C.c_int32, C.c_float, C.c_uint64, C.c_uint64,
                                P, P]),
    "dflash_verify_noalloc": (C.c_int, [SessArr, C.c_int32, P, C.c_int32, P, C.c_int32, C.c_float, C.c_uint64,
                                        C.c_uint64, P, P]),
    "dflash_close": (C.c_int, [P]),
    "dflash_stats": (C.c_int, [P, C.POINTER(dflash_counters)]),
    "dflash_session_state": (C.c_int, [P, C.POINTER(C.c_int64), C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
    "dflash_kv_export": (C.c_int, [P, C.c_int32, C.c_int64, C.c_int32, P, P]),
    "dflash_kv_import": (C.c_int, [P, C.c_int32, C.c_int64, C.c_int32, P, P]),
    "dflash_timing_enable": (C.c_int, [P, C.c_int32]),
    "dflash_timing_read": (C.c_int, [P, C.POINTER(dflash_kernel_time), C.c_int32, C.POINTER(C.c_int32)]),
    "dflash_set_sampler": (C.c_int, [P, C.c_int32, C.c_float, C.c_float]),
    "dflash_set_penalties": (C.c_int, [P, C.c_float, C.c_float, C.c_float, P, C.c_int32]),
    "dflash_candidates": (C.c_int, [P, P, P]),
    "dflash_target_create": (C.c_int, [C.POINTER(dflash_target_config), C.POINTER(dflash_target_weights), C.c_int64,
                                       P, C.POINTER(C.c_void_p)]),
    "dflash_target_destroy": (C.c_int, [P]),
    "dflash_target_forward": (C.c_int, [P, P, C.c_int32, C.c_int64, P, P]),
    "dflash_target_trim": (C.c_int, [P, C.c_int64]),
    "dflash_target_length": (C.c_int, [P, C.POINTER(C.c_int64)]),
    "dflash_target_argmax": (C.c_int, [P, P, C.c_int32, P]),
    "dflash_target_device_status": (C.c_int, [P]),
    "dflash_logits_compare": (C.c_int, [P, P, C.c_int32, C.c_int32, P, P]),
    "dflash_exactness_summarize": (C.c_int, [C.POINTER(dflash_exactness_row), C.c_int32,
                                             C.POINTER(dflash_exactness_summary)]),
    "dflash_target_exactness_probe": (C.c_int, [P, P, C.c_int32, C.c_int64, P, P, P,
                                                C.POINTER(dflash_exactness_summary)]),
}


def header_symbols(path: str | None = None) -> list[str]:
    """Entry points declared in include/*.h (for the export check)."""
    import re
    inc = os.path.join(os.path.dirname(_HERE), "include")
    names = []
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            names += re.findall(r"DFLASH_API\s+[\w\s\*]*?\b(dflash_\w+)\s*\(", txt)
    return names


def load(path: str = LIB_PATH) -> C.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m block_diffusion_speculative_flush_gb300.build` "
            "(the DFlash path has no fallback)")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib
