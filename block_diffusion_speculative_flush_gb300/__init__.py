"""Python binding of the GB300-native DFlash draft round (libdflash.so).

Each function has the name of the C entry point it marshals and does nothing
else: tensors become device pointers, lists of sessions become host arrays,
negative status codes become DFlashError.  Every step of the round runs in
the CUDA library; if the library is missing, importing this package fails.

PyTorch is used only for device memory (the tensors passed in) and streams.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _abi
from ._abi import (DFLASH_DTYPE_BF16, DFLASH_DTYPE_F32, DFLASH_ERR_CAPACITY, DFLASH_ERR_CONTEXT_GAP,
                   DFLASH_ERR_CUDA, DFLASH_ERR_DEVICE, DFLASH_ERR_INVALID_ARG, DFLASH_ERR_OOM, DFLASH_ERR_SHAPE,
                   DFLASH_ERR_STATE, DFLASH_FLAG_SIMT_GEMM, DFLASH_OK, DFLASH_PENDING_FLUSH_TOKENS,
                   DFLASH_VARIANT_DFLASH, DFLASH_VARIANT_DFLASH2, DFLASH2_DEPTH)

lib = _abi.load()

__all__ = [
    "DFlashError", "Model", "Session", "lib", "torch_dtype",
    "dflash_model_create", "dflash_model_destroy", "dflash_draft_limit", "dflash_device_status", "dflash_open",
    "dflash_committed", "dflash_committed_taps", "dflash_flush", "dflash_settle", "dflash_commit_block", "dflash_propose", "dflash_verify",
    "dflash_close", "dflash_set_sampler", "dflash_set_penalties", "dflash_candidates", "dflash_committed_batch", "dflash_stats", "dflash_session_state", "dflash_kv_export", "dflash_kv_import",
    "dflash_version", "dflash_last_error", "dflash_timing_enable", "dflash_timing_read", "dflash_verify_noalloc",
    "Target", "dflash_target_create", "dflash_target_destroy", "dflash_target_forward", "dflash_target_trim",
    "dflash_target_length", "dflash_target_argmax", "dflash_target_device_status",
    "dflash_logits_compare", "dflash_exactness_summarize", "dflash_target_exactness_probe", "exactness_rows",
]


class DFlashError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dflash status {status}: {message}")
        self.status = status


def _check(rc: int) -> int:
    if rc < 0:
        raise DFlashError(rc, lib.dflash_last_error().decode(errors="replace"))
    return rc


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()


def torch_dtype(cfg) -> torch.dtype:
    return torch.bfloat16 if cfg.dtype == "bf16" else torch.float32


class Model:
    """Handle of a dflash_model; keeps the weight tensors alive."""

    def __init__(self, handle: int, cfg, tensors: dict, layer_structs):
        self.handle = handle
        self.cfg = cfg
        self._tensors = tensors
        self._layers = layer_structs

    def __del__(self):
        if getattr(self, "handle", None):
            lib.dflash_model_destroy(self.handle)
            self.handle = None


class Session:
    def __init__(self, handle: int, model: Model):
        self.handle = handle
        self.model = model


def _sessions(sessions):
    if isinstance(sessions, Session):
        sessions = [sessions]
    arr = (C.c_void_p * len(sessions))(*[s.handle for s in sessions])
    return arr, len(sessions)


def _need(t, dtypes, numel: int, what: str) -> None:
    """The library reads or writes numel elements of t from its data pointer:
    t must be a contiguous CUDA tensor of one of dtypes with at least that many."""
    if t is None:
        return
    if not isinstance(dtypes, tuple):
        dtypes = (dtypes,)
    if not t.is_cuda or t.dtype not in dtypes or not t.is_contiguous() or t.numel() < numel:
        raise ValueError(f"{what}: a contiguous CUDA tensor of {'/'.join(str(d) for d in dtypes)} with at least "
                         f"{numel} elements")


def _model_of(sessions):
    first = sessions if isinstance(sessions, Session) else sessions[0]
    return first.model


def dflash_version() -> int:
    return lib.dflash_version()


def dflash_last_error() -> str:
    return lib.dflash_last_error().decode(errors="replace")


def dflash_model_create(cfg, weights: dict, flags: int = 0) -> Model:
    """cfg: an object with the fields of synthetic.DraftConfig; weights: name ->
    CUDA tensor in the storage type (names as synthetic.weight_shapes)."""
    c = _abi.dflash_config(
        dtype=DFLASH_DTYPE_BF16 if cfg.dtype == "bf16" else DFLASH_DTYPE_F32, n_taps=cfg.n_taps,
        target_hidden=cfg.target_hidden, hidden=cfg.hidden, n_layers=cfg.n_layers, n_q_heads=cfg.n_q_heads,
        n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, intermediate=cfg.intermediate, vocab=cfg.vocab,
        block_size=cfg.block_size, mask_token=cfg.mask_token, window=cfg.window,
        causal_block=int(cfg.causal_block), gated_attention=int(cfg.gated_attention), flags=flags,
        rope_theta=cfg.rope_theta, rms_eps=cfg.rms_eps,
        variant=DFLASH_VARIANT_DFLASH2 if getattr(cfg, "variant", "dflash") == "dflash2" else DFLASH_VARIANT_DFLASH,
        conv_taps=getattr(cfg, "conv_taps", 0), sel_rank=getattr(cfg, "sel_rank", 0),
        sel_candidates=getattr(cfg, "sel_candidates", 0))
    t = {k: v.contiguous() for k, v in weights.items()}
    layers = (_abi.dflash_layer_weights * cfg.n_layers)()
    for l in range(cfg.n_layers):
        p = f"layers.{l}."
        g = t.get(p + "w_g")
        layers[l] = _abi.dflash_layer_weights(
            _ptr(t[p + "in_norm"]), _ptr(t[p + "w_qkv"]), _ptr(t[p + "q_norm"]), _ptr(t[p + "k_norm"]), _ptr(g),
            _ptr(t[p + "w_o"]), _ptr(t[p + "post_norm"]), _ptr(t[p + "w_gate"]), _ptr(t[p + "w_up"]),
            _ptr(t[p + "w_down"]), _ptr(t.get(p + "conv_norm")), _ptr(t.get(p + "w_dc")))
    w = _abi.dflash_weights(_ptr(t["aux_norms"]), _ptr(t["w_fc"]), _ptr(t["hidden_norm"]), _ptr(t["final_norm"]),
                            _ptr(t["embed"]), _ptr(t["unembed"]), layers, _ptr(t.get("sel_prev")),
                            _ptr(t.get("sel_next")))
    out = C.c_void_p()
    _check(lib.dflash_model_create(C.byref(c), C.byref(w), C.byref(out)))
    return Model(out.value, cfg, t, layers)


def dflash_model_destroy(model: Model) -> None:
    if model.handle:
        _check(lib.dflash_model_destroy(model.handle))
        model.handle = None


def dflash_draft_limit(model: Model) -> int:
    return _check(lib.dflash_draft_limit(model.handle))


def dflash_device_status(model: Model) -> None:
    _check(lib.dflash_device_status(model.handle))


def dflash_open(model: Model, restored_offset: int = 0, max_ctx: int = 4096, stream=None) -> Session:
    if stream is None:
        stream = torch.cuda.current_stream()
    out = C.c_void_p()
    _check(lib.dflash_open(model.handle, restored_offset, max_ctx, C.c_void_p(stream.cuda_stream), C.byref(out)))
    return Session(out.value, model)


def dflash_committed(session: Session, features: torch.Tensor, position: int) -> None:
    """features: CUDA tensor [n_rows, K*H_t] (row stride from the tensor)."""
    if features.dim() != 2 or features.stride(1) != 1:
        raise ValueError("features must be 2-D with unit column stride")
    cfg = session.model.cfg
    if not features.is_cuda or features.dtype != torch_dtype(cfg) or features.shape[1] != cfg.feature_width:
        raise ValueError(f"features: CUDA {torch_dtype(cfg)} rows of width {cfg.feature_width}")
    _check(lib.dflash_committed(session.handle, _ptr(features), features.stride(0), features.shape[0], position))


def dflash_committed_taps(session: Session, taps, position: int) -> None:
    """taps: n_taps CUDA tensors [n_rows, H_t] (unit column stride, one row stride for all)."""
    cfg = session.model.cfg
    taps = list(taps)
    if len(taps) != cfg.n_taps:
        raise ValueError(f"{cfg.n_taps} taps expected")
    rows, stride = taps[0].shape[0], taps[0].stride(0)
    for t in taps:
        if t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda or t.dtype != torch_dtype(cfg) or \
                t.shape != (rows, cfg.target_hidden) or t.stride(0) != stride:
            raise ValueError(f"taps: CUDA {torch_dtype(cfg)} [{rows}, {cfg.target_hidden}] with one row stride")
    arr = (C.c_void_p * len(taps))(*[t.data_ptr() for t in taps])
    _check(lib.dflash_committed_taps(session.handle, arr, stride, rows, position))


def dflash_committed_batch(sessions, features, positions) -> None:
    """features: one CUDA tensor [n_rows_b, K*H_t] per session (one row stride
    for all); positions: the committed run's position per session.  Sessions
    that reach the flush threshold flush in one batched forward."""
    arr, b = _sessions(sessions)
    features, positions = list(features), [int(x) for x in positions]
    if len(features) != b or len(positions) != b:
        raise ValueError("one features tensor and one position per session")
    cfg = _model_of(sessions).cfg
    stride = features[0].stride(0)
    for f in features:
        if f.dim() != 2 or f.stride(1) != 1 or not f.is_cuda or f.dtype != torch_dtype(cfg) or \
                f.shape[1] != cfg.feature_width or (f.shape[0] > 1 and f.stride(0) != stride):
            raise ValueError(f"features: CUDA {torch_dtype(cfg)} rows of width {cfg.feature_width}, one row stride")
    ptrs = (C.c_void_p * b)(*[f.data_ptr() for f in features])
    rows = (C.c_int32 * b)(*[f.shape[0] for f in features])
    pos = (C.c_int64 * b)(*positions)
    _check(lib.dflash_committed_batch(arr, b, ptrs, stride, rows, pos))


def dflash_flush(sessions) -> None:
    arr, n = _sessions(sessions)
    _check(lib.dflash_flush(arr, n))


def dflash_settle(session: Session) -> None:
    _check(lib.dflash_settle(session.handle))


def dflash_commit_block(sessions) -> None:
    arr, n = _sessions(sessions)
    _check(lib.dflash_commit_block(arr, n))


def dflash_propose(sessions, current: torch.Tensor, max_tokens: int, temperature: float, seed: int, rnd: int,
                   out_tokens: torch.Tensor, out_q: torch.Tensor, out_logits: torch.Tensor | None = None) -> list:
    """Returns out_n per session (0 where the pages return nil)."""
    arr, n = _sessions(sessions)
    cfg = _model_of(sessions).cfg
    per = max(0, min(int(max_tokens), cfg.block_size - 1))
    if per and getattr(cfg, "variant", "dflash") == "dflash2":
        per = min(DFLASH2_DEPTH, cfg.block_size - 1)      # a DFlash2 proposal's fixed length
    rows = n * per
    _need(current, torch.int32, n, "current")
    _need(out_tokens, torch.int32, rows, "out_tokens")
    _need(out_q, torch.float32, rows, "out_q")
    _need(out_logits, torch.float32, rows * cfg.vocab, "out_logits")
    out_n = (C.c_int32 * n)()
    _check(lib.dflash_propose(arr, n, _ptr(current), max_tokens, float(temperature), seed, rnd, _ptr(out_tokens),
                              _ptr(out_q), _ptr(out_logits), out_n))
    return list(out_n)


def _verify_args(sessions, b, target_logits, draft_tokens, n, out_accept, out_bonus) -> None:
    V = _model_of(sessions).cfg.vocab
    n = max(0, int(n))
    _need(target_logits, (torch.float32, torch.bfloat16), b * (n + 1) * V, "target_logits [batch, n+1, V]")
    _need(draft_tokens, torch.int32, b * n, "draft_tokens [batch, n]")
    _need(out_accept, torch.int32, b, "out_accept")
    _need(out_bonus, torch.int32, b, "out_bonus")


def dflash_verify(sessions, target_logits: torch.Tensor, draft_tokens: torch.Tensor, n: int, temperature: float,
                  seed: int, rnd: int, out_accept: torch.Tensor, out_bonus: torch.Tensor) -> None:
    arr, b = _sessions(sessions)
    _verify_args(sessions, b, target_logits, draft_tokens, n, out_accept, out_bonus)
    dt = DFLASH_DTYPE_BF16 if target_logits.dtype == torch.bfloat16 else DFLASH_DTYPE_F32
    _check(lib.dflash_verify(arr, b, _ptr(target_logits), dt, _ptr(draft_tokens), n, float(temperature), seed, rnd,
                             _ptr(out_accept), _ptr(out_bonus)))


def dflash_verify_noalloc(sessions, target_logits: torch.Tensor, draft_tokens: torch.Tensor, n: int,
                          temperature: float, seed: int, rnd: int, out_accept: torch.Tensor,
                          out_bonus: torch.Tensor) -> None:
    """dflash_verify on the library's static scratch (no device allocation)."""
    arr, b = _sessions(sessions)
    _verify_args(sessions, b, target_logits, draft_tokens, n, out_accept, out_bonus)
    dt = DFLASH_DTYPE_BF16 if target_logits.dtype == torch.bfloat16 else DFLASH_DTYPE_F32
    _check(lib.dflash_verify_noalloc(arr, b, _ptr(target_logits), dt, _ptr(draft_tokens), n, float(temperature), seed,
                                     rnd, _ptr(out_accept), _ptr(out_bonus)))


def dflash_close(session: Session) -> None:
    if session.handle:
        _check(lib.dflash_close(session.handle))
        session.handle = None


def dflash_candidates(session: Session, out_ids: torch.Tensor, out_probs: torch.Tensor) -> None:
    """A DFlash2 session's last candidate distributions: ids int32 and
    probabilities fp32, each [n, sel_candidates] on the device."""
    cfg = session.model.cfg
    k, n = cfg.sel_candidates, min(DFLASH2_DEPTH, cfg.block_size - 1)
    _need(out_ids, torch.int32, n * k, "out_ids [n, sel_candidates]")
    _need(out_probs, torch.float32, n * k, "out_probs [n, sel_candidates]")
    _check(lib.dflash_candidates(session.handle, _ptr(out_ids), _ptr(out_probs)))


def dflash_set_penalties(session: Session, repeat: float = 1.0, presence: float = 0.0, frequency: float = 0.0,
                         history: torch.Tensor | None = None) -> None:
    """The sampler's penalties over a committed history (CUDA int32 [n] token ids)."""
    n = 0 if history is None else int(history.numel())
    if n and (not history.is_cuda or history.dtype != torch.int32 or not history.is_contiguous()):
        raise ValueError("history: contiguous CUDA int32 token ids")
    _check(lib.dflash_set_penalties(session.handle, float(repeat), float(presence), float(frequency),
                                    _ptr(history) if n else None, n))


def dflash_set_sampler(session: Session, top_k: int = 0, top_p: float = 1.0, min_p: float = 0.0) -> None:
    _check(lib.dflash_set_sampler(session.handle, top_k, top_p, min_p))


def dflash_stats(session: Session) -> dict:
    c = _abi.dflash_counters()
    _check(lib.dflash_stats(session.handle, C.byref(c)))
    return {k: getattr(c, k) for k, _ in c._fields_}


def dflash_session_state(session: Session) -> tuple:
    F, P, B = C.c_int64(), C.c_int32(), C.c_int32()
    _check(lib.dflash_session_state(session.handle, C.byref(F), C.byref(P), C.byref(B)))
    return F.value, P.value, bool(B.value)


def dflash_kv_export(session: Session, layer: int, first_slot: int, n_rows: int, k_out: torch.Tensor,
                     v_out: torch.Tensor) -> None:
    _check(lib.dflash_kv_export(session.handle, layer, first_slot, n_rows, _ptr(k_out), _ptr(v_out)))


def dflash_kv_import(session: Session, layer: int, first_slot: int, n_rows: int, k_in: torch.Tensor,
                     v_in: torch.Tensor) -> None:
    _check(lib.dflash_kv_import(session.handle, layer, first_slot, n_rows, _ptr(k_in), _ptr(v_in)))


def dflash_timing_enable(model: Model, on: bool) -> None:
    _check(lib.dflash_timing_enable(model.handle, 1 if on else 0))


def dflash_timing_read(model: Model) -> dict:
    """kernel class -> dict(launches, total_ms, bytes, flops); synchronises."""
    arr = (_abi.dflash_kernel_time * 16)()
    n = C.c_int32()
    _check(lib.dflash_timing_read(model.handle, arr, 16, C.byref(n)))
    return {arr[i].name.decode(): dict(launches=arr[i].launches, total_ms=arr[i].total_ms, bytes=arr[i].bytes,
                                       flops=arr[i].flops) for i in range(n.value)}


# ---------------------------------------------------------------------------
# synthetic target (fp32)
# ---------------------------------------------------------------------------
class Target:
    """Handle of a dflash_target; keeps the weight tensors alive."""

    def __init__(self, handle: int, cfg: dict, tensors: list, layer_structs):
        self.handle = handle
        self.cfg = cfg
        self._tensors = tensors
        self._layers = layer_structs

    def __del__(self):
        if getattr(self, "handle", None):
            lib.dflash_target_destroy(self.handle)
            self.handle = None


def dflash_target_create(cfg: dict, weights: dict, max_ctx: int = 4096, stream=None) -> Target:
    """cfg: hidden, n_heads, head_dim, intermediate, vocab, n_layers, rope_theta, rms_eps;
    weights: fp32 CUDA tensors embed, unembed, final_norm and layers = [dict n1, wq, wk,
    wv, wo, n2, wg, wu, wd]."""
    c = _abi.dflash_target_config(hidden=cfg["hidden"], n_heads=cfg["n_heads"], head_dim=cfg["head_dim"],
                                  intermediate=cfg["intermediate"], vocab=cfg["vocab"], n_layers=cfg["n_layers"],
                                  rope_theta=cfg["rope_theta"], rms_eps=cfg["rms_eps"])
    keep = []
    H, qd, I, V = cfg["hidden"], cfg["n_heads"] * cfg["head_dim"], cfg["intermediate"], cfg["vocab"]
    shapes = dict(n1=(H,), wq=(qd, H), wk=(qd, H), wv=(qd, H), wo=(H, qd), n2=(H,), wg=(I, H), wu=(I, H),
                  wd=(H, I))

    def dev(t, shape, name):
        t = t.contiguous()
        if not t.is_cuda or t.dtype != torch.float32:
            raise ValueError("target weights are fp32 CUDA tensors")
        if tuple(t.shape) != shape:
            raise ValueError(f"target weight {name}: shape {tuple(t.shape)}, expected {shape}")
        keep.append(t)
        return t.data_ptr()

    if len(weights["layers"]) != cfg["n_layers"]:
        raise ValueError("target weights: one dict per layer")
    layers = (_abi.dflash_target_layer * cfg["n_layers"])()
    for l, lw in enumerate(weights["layers"]):
        for name, shape in shapes.items():
            setattr(layers[l], name, dev(lw[name], shape, name))
    w = _abi.dflash_target_weights(embed=dev(weights["embed"], (V, H), "embed"),
                                   unembed=dev(weights["unembed"], (V, H), "unembed"),
                                   final_norm=dev(weights["final_norm"], (H,), "final_norm"), layers=layers)
    stream = stream if stream is not None else torch.cuda.current_stream()
    out = C.c_void_p()
    _check(lib.dflash_target_create(C.byref(c), C.byref(w), max_ctx, C.c_void_p(stream.cuda_stream), C.byref(out)))
    return Target(out.value, dict(cfg), keep, layers)


def dflash_target_destroy(target: Target) -> None:
    if target.handle:
        _check(lib.dflash_target_destroy(target.handle))
        target.handle = None


def dflash_target_forward(target: Target, tokens: torch.Tensor, start: int, logits: torch.Tensor,
                          taps: torch.Tensor | None = None) -> None:
    """tokens: int32 CUDA [rows]; logits: fp32 CUDA [rows][vocab]; taps: fp32 CUDA [rows][(2L+1)*hidden]."""
    c = target.cfg
    rows = tokens.numel()
    if tokens.dtype != torch.int32 or not tokens.is_contiguous():
        raise ValueError("tokens must be contiguous int32")
    if logits.dtype != torch.float32 or not logits.is_contiguous() or tuple(logits.shape) != (rows, c["vocab"]):
        raise ValueError("logits must be contiguous fp32 [rows, vocab]")
    if taps is not None and (taps.dtype != torch.float32 or not taps.is_contiguous() or
                             tuple(taps.shape) != (rows, (2 * c["n_layers"] + 1) * c["hidden"])):
        raise ValueError("taps must be contiguous fp32 [rows, (2 * n_layers + 1) * hidden]")
    _check(lib.dflash_target_forward(target.handle, _ptr(tokens), tokens.numel(), start, _ptr(logits), _ptr(taps)))


def dflash_target_trim(target: Target, length: int) -> None:
    _check(lib.dflash_target_trim(target.handle, length))


def dflash_target_length(target: Target) -> int:
    v = C.c_int64()
    _check(lib.dflash_target_length(target.handle, C.byref(v)))
    return v.value


def dflash_target_argmax(target: Target, logits: torch.Tensor, out: torch.Tensor) -> None:
    """logits: fp32 CUDA [rows][vocab]; out: int32 CUDA [rows], the greedy token of each row."""
    if logits.dtype != torch.float32 or not logits.is_contiguous() or logits.dim() != 2 or \
            logits.shape[1] != target.cfg["vocab"] or out.dtype != torch.int32 or out.numel() < logits.shape[0]:
        raise ValueError("logits must be contiguous fp32 [rows, vocab] and out int32 [rows]")
    _check(lib.dflash_target_argmax(target.handle, _ptr(logits), logits.shape[0], _ptr(out)))


def dflash_target_device_status(target: Target) -> None:
    _check(lib.dflash_target_device_status(target.handle))


EXACTNESS_ROW_BYTES = C.sizeof(_abi.dflash_exactness_row)


def _rows_buffer(out: torch.Tensor, rows: int) -> None:
    if out.dtype != torch.uint8 or not out.is_contiguous() or out.numel() < rows * EXACTNESS_ROW_BYTES:
        raise ValueError(f"out must be a contiguous uint8 CUDA buffer of rows * {EXACTNESS_ROW_BYTES} bytes")


def _logits_pair(a: torch.Tensor, b: torch.Tensor) -> tuple:
    if a.dtype != torch.float32 or b.dtype != torch.float32 or a.dim() != 2 or a.shape != b.shape or \
            not a.is_contiguous() or not b.is_contiguous():
        raise ValueError("block and chain logits must be contiguous fp32 [rows, vocab] of one shape")
    return a.shape[0], a.shape[1]


def dflash_logits_compare(block: torch.Tensor, chain: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """block, chain: fp32 CUDA [rows][vocab]; out: uint8 CUDA buffer of rows dflash_exactness_row records."""
    rows, V = _logits_pair(block, chain)
    _rows_buffer(out, rows)
    stream = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.dflash_logits_compare(_ptr(block), _ptr(chain), rows, V, _ptr(out), C.c_void_p(stream.cuda_stream)))


def _records(buf):
    raw = bytes(buf.cpu().numpy().tobytes()) if isinstance(buf, torch.Tensor) else bytes(buf)
    n = len(raw) // EXACTNESS_ROW_BYTES
    return (_abi.dflash_exactness_row * n).from_buffer_copy(raw[:n * EXACTNESS_ROW_BYTES])


def exactness_rows(buf) -> list:
    """Decodes row records (the uint8 buffer, copied to the host) into dicts."""
    return [dict(differing_bytes=r.differing_bytes, block_top=list(r.block_top), chain_top=list(r.chain_top),
                 block_val=list(r.block_val), chain_val=list(r.chain_val)) for r in _records(buf)]


def dflash_exactness_summarize(buf) -> dict:
    arr = _records(buf)
    s = _abi.dflash_exactness_summary()
    _check(lib.dflash_exactness_summarize(arr, len(arr), C.byref(s)))
    return {k: getattr(s, k) for k, _ in s._fields_}


def dflash_target_exactness_probe(target: Target, tokens: torch.Tensor, start: int, block_logits: torch.Tensor,
                                  chain_logits: torch.Tensor, out: torch.Tensor) -> dict:
    """Block forward and one-token forwards of `tokens` at start, compared; the
    cache is left at `start`.  Returns the summary (the call synchronises)."""
    rows, V = _logits_pair(block_logits, chain_logits)
    if tokens.dtype != torch.int32 or not tokens.is_contiguous() or tokens.numel() != rows or \
            V != target.cfg["vocab"]:
        raise ValueError("tokens must be contiguous int32 [rows] and logits [rows, vocab]")
    _rows_buffer(out, rows)
    s = _abi.dflash_exactness_summary()
    _check(lib.dflash_target_exactness_probe(target.handle, _ptr(tokens), rows, start, _ptr(block_logits),
                                             _ptr(chain_logits), _ptr(out), C.byref(s)))
    return {k: getattr(s, k) for k, _ in s._fields_}
