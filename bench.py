#!/usr/bin/env python3
"""Throughput of the DFlash draft round on GB300.

One step is one whole round of the hot path for one sequence of the
Qwen3-8B-shaped bf16 draft (5 layers, hidden 4096, 32 Q / 8 KV heads of 128,
SwiGLU 12288, vocab 151936, block 16 so n = 15, temperature 1.0):

  committed   4 new target feature rows [4, 5 x 4096] (the steady-state
              accepted + bonus rows of a round), appended at the frontier
  propose     commit_block rewind, the 4 held rows pass aux norms / fc /
              hidden norm / per-layer K/V into the cache, the 16-row block
              forward against the context, unembedding of rows 1..15 and
              one batched Gumbel-max draw
  verify      accept length and bonus token from target logits [16, 151936]

The context starts at 4096 - 4 (W + K/2) rows filled by a real flush, so the
mean context over the K timed steps is 4096.  Weights (3.4 GB) are read every
step, far more than the 129 MB L2, so no L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 (under torchrun): N independent replicas, one sequence per GPU, no
collective on the data path (weak scaling); rank 0 prints the line with the
max time over ranks.  --impl reference times the CPU oracle (this method has
no other reference implementation) on bounded samples of the same round.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft rounds/sec & proposed tok/s (bs1, bs64); flush rows/s; % HBM roofline"
UNIT = "draft rounds/s"
CFG_NAME = "qwen3_8b_bf16"
CTX = 4096
P_ROWS = 4
TEMP = 1.0
SEED = 20260201
PROFILE_RANGE = False   # --profile-range


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--small", action="store_true",
                    help="batched only: the same serving mix with one draft layer and a 32000-entry "
                         "vocabulary (about 3 GB on the device), a case small enough for a full ncu capture")
    ap.add_argument("--profile-range", action="store_true",
                    help="bracket every timed region with cudaProfilerStart/Stop, so that "
                         "`ncu --profile-from-start off` captures the timed steps only")
    ap.add_argument("--workload", choices=["round", "flush", "laguna", "batched", "spec", "truncated"],
                    default="round",
                    help="round: the bs1 Qwen3-8B-shaped round (the default line); flush: 8 sequences x 256-row "
                         "context flushes; laguna: window-512 gated draft, bs1, blocks 16 and 8; batched: 64 "
                         "sequences, contexts 1k-16k, propose + rejection-sampling verify at T=0.7; spec: greedy "
                         "speculative decoding with the tiny fp32 draft and the synthetic target, both on the GPU; "
                         "truncated: the bs1 round with a top-k 40 / top-p 0.9 sampler against the same round "
                         "with full distributions")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# ranks (replicas only: the barrier and the max over ranks are the only
# cross-rank traffic)
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [r for r in csv.reader(io.StringIO(open(self.path).read())) if len(r) >= 9]
        os.unlink(self.path)
        sm, smax, reasons, samples = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except ValueError:
                continue
            samples += 1
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": samples}


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def traffic_from_profile(kernel_src: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "k_gemm_tc_traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    digest = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    if kv.get("source_sha256_16") != digest:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def round_bytes(cfg, ctx, P):
    """Algorithmic bytes of one bs1 round: every weight read once, the context
    K/V read once per layer, the features read once, the new K/V written once,
    the logits written and read once, the target logits read once."""
    H, I, V = cfg.hidden, cfg.intermediate, cfg.vocab
    qkv = (cfg.qkv_rows + (cfg.n_q_heads if cfg.gated_attention else 0)) * H
    per_layer = qkv + H * cfg.n_q_heads * cfg.head_dim + 3 * H * I
    if cfg.window:
        ctx = min(ctx, cfg.window - 1)
    weights = 2 * (cfg.n_layers * per_layer + V * H + (H * cfg.feature_width if P else 0))
    nb = cfg.block_size
    kv_row = 2 * cfg.n_kv_heads * cfg.head_dim * 2 * cfg.n_layers
    kv = (ctx + nb) * kv_row + (P + nb) * kv_row
    feats = P * cfg.feature_width * 2
    logits = (nb - 1) * V * 4 * 2 + nb * V * 4
    return weights + kv + feats + logits


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def gpu_weights(cfg, seed, device):
    import torch

    import synthetic as S
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = {}
    for name, shape in S.weight_shapes(cfg).items():
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * 0.02
        if name.endswith("norm") or name == "aux_norms":
            x += 1.0
        out[name] = x.to(torch.bfloat16 if cfg.dtype == "bf16" else torch.float32)
    return out


def run_ours(args, rank, world, local_rank):
    import torch

    import block_diffusion_speculative_flush_gb300 as D
    import synthetic as S

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist_init(world, "nccl")
    cfg = S.CONFIGS[CFG_NAME]
    K, W = args.steps, args.warmup
    n = cfg.block_size - 1
    V = cfg.vocab
    stream = torch.cuda.Stream(device=dev)
    weights = gpu_weights(cfg, SEED + rank, dev)
    model = D.dflash_model_create(cfg, weights)
    start_ctx = CTX - P_ROWS * (W + K // 2)
    assert start_ctx > 0, "too many steps for the 4096-row mean context"
    max_ctx = start_ctx + P_ROWS * (W + K + 8)
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 1000 + rank)
    sessions = []
    with torch.cuda.stream(stream):
        for _ in range(3):   # kernel-only loop, end-to-end loop, instrumented loop
            s = D.dflash_open(model, max_ctx=max_ctx, stream=stream)
            for lo in range(0, start_ctx, 1024):
                hi = min(start_ctx, lo + 1024)
                f = torch.randn((hi - lo, cfg.feature_width), generator=g, device=dev).to(torch.bfloat16)
                D.dflash_committed(s, f, lo)
                del f
            D.dflash_flush([s])
            sessions.append(s)
        feats = torch.randn((W + K, P_ROWS, cfg.feature_width), generator=g, device=dev).to(torch.bfloat16)
        tl = (torch.randn((1, n + 1, V), generator=g, device=dev) * 3.0).contiguous()
        cur = torch.full((1,), 17, dtype=torch.int32, device=dev)
        tok = torch.empty((1, n), dtype=torch.int32, device=dev)
        q = torch.empty((1, n), dtype=torch.float32, device=dev)
        acc = torch.empty(1, dtype=torch.int32, device=dev)
        bon = torch.empty(1, dtype=torch.int32, device=dev)
    stream.synchronize()

    def step(s, i, f, logits):
        D.dflash_committed(s, f, start_ctx + P_ROWS * i)
        D.dflash_propose([s], cur, n, TEMP, SEED, i, tok, q)
        D.dflash_verify([s], logits, tok, n, TEMP, SEED, i, acc, bon)

    # ---- kernel-only timed region: inputs resident in HBM ----
    sa = sessions[0]
    with torch.cuda.stream(stream):
        for i in range(W):
            step(sa, i, feats[i], tl)
            step(sessions[2], i, feats[i], tl)
    stream.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    _profile_range(torch, True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(W, W + K):
            step(sa, i, feats[i], tl)
        e1.record(stream)
    torch.cuda.synchronize()
    _profile_range(torch, False)
    barrier(world)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, world, dev)

    # ---- the same steps again with CUDA events around every instrumented
    # launch (per-kernel-class durations for the roofline; the events break
    # the launch overlap, so this pass is not the one that gives `value`)
    sc = sessions[2]
    D.dflash_timing_enable(model, True)
    with torch.cuda.stream(stream):
        for i in range(W, W + K):
            step(sc, i, feats[i], tl)
    timing = D.dflash_timing_read(model)
    D.dflash_timing_enable(model, False)

    # ---- end to end through the public API with host buffers ----
    sb = sessions[1]
    feats_h = feats.cpu().pin_memory()
    tl_h = tl.cpu().pin_memory()
    f_dev = torch.empty((P_ROWS, cfg.feature_width), dtype=torch.bfloat16, device=dev)
    tl_dev = torch.empty_like(tl)
    tok_h = torch.empty((1, n), dtype=torch.int32).pin_memory()
    acc_h = torch.empty(1, dtype=torch.int32).pin_memory()
    bon_h = torch.empty(1, dtype=torch.int32).pin_memory()

    def e2e_step(i):
        f_dev.copy_(feats_h[i], non_blocking=True)
        tl_dev.copy_(tl_h, non_blocking=True)
        step(sb, i, f_dev, tl_dev)
        tok_h.copy_(tok, non_blocking=True)
        acc_h.copy_(acc, non_blocking=True)
        bon_h.copy_(bon, non_blocking=True)
        stream.synchronize()

    with torch.cuda.stream(stream):
        for i in range(W):
            e2e_step(i)
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(W, W + K):
            e2e_step(i)
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
    barrier(world)
    e2e_max = max_over_ranks(e2e_s, world, dev)
    D.dflash_device_status(model)
    h2d = P_ROWS * cfg.feature_width * 2 + tl.numel() * 4
    d2h = n * 4 + 4 + 4

    result = None
    if rank == 0:
        peaks, peak_kind = measured_peaks()
        gt = timing.get("gemm_tc", {})
        achieved = gt["bytes"] / (gt["total_ms"] * 1e-3) / 1e9 if gt.get("total_ms") else None
        launches = gt.get("launches", 0)
        traffic = traffic_from_profile(os.path.join(ROOT, "block_diffusion_speculative_flush_gb300", "csrc",
                                                    "gemm_tc.cu"))
        value = world * K / (ms_max * 1e-3)
        rb = round_bytes(cfg, CTX, P_ROWS)
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(ms_max / K, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init draft weights, N(0,1) features, "
                                                          "N(0,3) target logits)",
            "config": {"workload": "qwen3_8b_bf16 draft round, bs1, block 16 (n=15), mean ctx 4096, "
                                   "4 committed rows per round, T=1.0",
                       "model": "Qwen3-8B-shaped DFlash draft (5 layers, H 4096, 32/8 heads x 128, I 12288, "
                                "V 151936)",
                       "global_batch": world, "seq_len": CTX, "parallelism": f"replicas x{world}",
                       "l2": "no flush: 3.4 GB of weights streamed per step (L2 is 129 MB)"},
            "proposed_tok_s": round(value * n, 1),
            "round_roofline": {"bound": "hbm", "algorithmic_bytes": rb,
                               "achieved_gbs": round(rb / (ms_max / K * 1e-3) / 1e9, 1),
                               "peak_gbs": peaks["hbm_gbs"],
                               "frac": round(rb / (ms_max / K * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
            "roofline": {"kernel": "k_gemm_tc (tcgen05 weight-streaming GEMM)", "bound": "hbm",
                         "achieved": round(achieved, 1) if achieved else None, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4) if achieved else None,
                         "peak_kind": f"{peak_kind} HBM copy bandwidth",
                         "algorithmic_bytes_per_launch": round(gt["bytes"] / launches) if launches else None,
                         "traffic": traffic, "launches": launches},
            "kernel_classes_instrumented": {k: {"launches": v["launches"], "ms_per_step": round(v["total_ms"] / K, 4),
                                   "gbs": round(v["bytes"] / (v["total_ms"] * 1e-3) / 1e9, 1)
                                   if v["total_ms"] else None}
                               for k, v in timing.items()},
            "gpu_launches": int(timing.get("all", {}).get("launches", 0)),
            "clocks": clk,
            "e2e": {"value": round(world * K / e2e_max, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
        }
    # weights for the CPU baseline are read before the GPU state goes away
    host_w = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host_w = {k: v.float().cpu().numpy() for k, v in weights.items()}
    for s in sessions:
        D.dflash_close(s)
    del model, weights
    torch.cuda.empty_cache()
    # the metric's other two configurations, each timed the same way (own
    # warm-up, CUDA events, clocks sampled during its own timed region)
    for key, wl in (("bs64", "batched"), ("flush", "flush")):
        sub = run_workload(argparse.Namespace(**dict(vars(args), workload=wl)), rank, world, local_rank)
        torch.cuda.empty_cache()
        if result is not None:
            result[key] = {k: sub[k] for k in ("metric", "value", "unit", "ms_per_step", "roofline", "clocks",
                                               "gpu_launches", "config") if k in sub}
            for extra in ("rounds_s", "per_sequence_flush_rows_s"):
                if extra in sub:
                    result[key][extra] = sub[extra]
    if result is not None and host_w is not None:
        result["cpu_baseline"] = cpu_baseline(cfg, host_w)
    return result


# ---------------------------------------------------------------------------
# further workloads (one JSON line each; the default line is the round above)
# ---------------------------------------------------------------------------
def _profile_range(torch, on):
    if PROFILE_RANGE:
        (torch.cuda.profiler.start if on else torch.cuda.profiler.stop)()


def _timed(torch, stream, fn, K, W, local_rank, world, dev):
    with torch.cuda.stream(stream):
        for i in range(W):
            fn(i)
    stream.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    _profile_range(torch, True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(W, W + K):
            fn(i)
        e1.record(stream)
    torch.cuda.synchronize()
    _profile_range(torch, False)
    barrier(world)
    clk = clocks.stop()
    return max_over_ranks(e0.elapsed_time(e1), world, dev), clk


def _instrumented_step(D, model, stream, step, torch, i=0):
    """One more step with the library's per-class CUDA events: returns its
    kernel launches and, per kernel class, launches, milliseconds and GB/s.
    (The events break the launch overlap, so this step is not a timed one.)"""
    D.dflash_timing_enable(model, True)
    with torch.cuda.stream(stream):
        step(i)
    t = D.dflash_timing_read(model)
    D.dflash_timing_enable(model, False)
    classes = {k: {"launches": v["launches"], "ms": round(v["total_ms"], 4),
                   "gbs": round(v["bytes"] / (v["total_ms"] * 1e-3) / 1e9, 1) if v["total_ms"] else None,
                   "tflops": round(v["flops"] / (v["total_ms"] * 1e-3) / 1e12, 1) if v["total_ms"] else None}
               for k, v in t.items() if k != "all"}
    return int(t.get("all", {}).get("launches", 0)), classes


def _launches_per_step(D, model, stream, step, torch, i=0):
    """Kernel launches of one more step, counted by the library."""
    return _instrumented_step(D, model, stream, step, torch, i)[0]


def _line(metric, unit, value, world, K, W, ms, dtype, config, extra, clk):
    out = {"metric": metric, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": K, "warmup": W,
           "ms_per_step": round(ms / K, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": dtype, "data": "synthetic (random-init draft weights, N(0,1) features and K/V)",
           "config": config, "clocks": clk}
    out.update(extra)
    return out


def run_workload(args, rank, world, local_rank):
    import numpy as np
    import torch

    import block_diffusion_speculative_flush_gb300 as D
    import synthetic as S

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist_init(world, "nccl")
    K, W = args.steps, args.warmup
    stream = torch.cuda.Stream(device=dev)
    peaks, peak_kind = measured_peaks()
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 7 + rank)

    if args.workload == "flush":
        # 8 sequences at context offsets 0, 1k, ..., 7k; each step every
        # sequence commits 256 new feature rows in one dflash_committed_batch
        # call: all 8 reach the pending threshold and flush together as one
        # context-only forward of 2048 rows (the first step also rewinds the
        # outstanding blocks)
        cfg = S.CONFIGS[CFG_NAME]
        rows, nseq = 256, 8
        model = D.dflash_model_create(cfg, gpu_weights(cfg, SEED + rank, dev))
        with torch.cuda.stream(stream):
            sess = [D.dflash_open(model, restored_offset=1024 * j, max_ctx=1024 * j + rows * (2 * K + 2 * W + 8),
                                  stream=stream) for j in range(nseq)]
            feats = torch.randn((rows, cfg.feature_width), generator=g, device=dev).to(torch.bfloat16)
            n = cfg.block_size - 1
            cur = torch.full((1,), 3, dtype=torch.int32, device=dev)
            tok = torch.empty((1, n), dtype=torch.int32, device=dev)
            q = torch.empty((1, n), dtype=torch.float32, device=dev)
            for s_ in sess:      # an outstanding block that the first flush rewinds
                D.dflash_propose([s_], cur, n, 0.0, 0, 0, tok, q)
        pos = [1024 * j for j in range(nseq)]

        def step(i):
            D.dflash_committed_batch(sess, [feats] * nseq, pos)
            for j in range(nseq):
                pos[j] += rows

        ms, clk = _timed(torch, stream, step, K, W, local_rank, world, dev)
        for j, s_ in enumerate(sess):       # cursor consistency after every rewind + flush
            assert D.dflash_session_state(s_) == (1024 * j + rows * (K + W), 0, False)
        launches, classes = _instrumented_step(D, model, stream, step, torch)
        # the same rows flushed one sequence at a time (dflash_committed per
        # sequence: eight forwards of 256 rows)
        def step_1(i):
            for j, s_ in enumerate(sess):
                D.dflash_committed(s_, feats, pos[j])
                pos[j] += rows

        ms_1, _ = _timed(torch, stream, step_1, max(1, K // 2), 1, local_rank, world, dev)
        kv_params = 2 * cfg.n_kv_heads * cfg.head_dim * cfg.hidden * cfg.n_layers
        fc_params = cfg.hidden * cfg.feature_width
        flops = 2.0 * rows * nseq * (fc_params + kv_params)
        tflops = flops / (ms / K * 1e-3) / 1e12
        peak_t = peaks.get("bf16_tflops_sustained", 1700.0)
        for s_ in sess:
            D.dflash_close(s_)
        return _line("flush rows/s (8 sequences x 256 pending rows, Qwen3-8B-shaped draft)", "rows/s",
                     world * rows * nseq / (ms / K * 1e-3), world, K, W, ms, "bf16",
                     {"workload": "8 sequences at context offsets 0..7k commit 256 rows [256, 20480] each per step "
                                  "(dflash_committed_batch): one batched context-only forward of 2048 rows, the "
                                  "first after a block rewind", "l2": "252 MB of fc/K/V weights per flush; "
                                  "features 10.5 MB resident"},
                     {"roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak_t,
                                   "unit": "TFLOP/s", "frac": round(tflops / peak_t, 4),
                                   "peak_kind": f"{peak_kind} bf16 (sustained)",
                                   "algorithmic_flops_per_step": flops},
                      "per_sequence_flush_rows_s": round(world * rows * nseq / (ms_1 / max(1, K // 2) * 1e-3), 1),
                      "kernel_classes_instrumented_one_step": classes,
                      "gpu_launches": launches * K}, clk)

    if args.workload == "laguna":
        res = {}
        for bs in (16, 8):
            cfg = S.CONFIGS["laguna_bf16"].replace(block_size=bs)
            n = bs - 1
            model = D.dflash_model_create(cfg, gpu_weights(cfg, SEED + rank, dev))
            T = 32768
            with torch.cuda.stream(stream):
                s_ = D.dflash_open(model, max_ctx=T + P_ROWS * (K + W + 4) + 64, stream=stream)
                for lo in range(0, T, 4096):      # rows older than the window are dropped before the fc
                    f = torch.randn((4096, cfg.feature_width), generator=g, device=dev).to(torch.bfloat16)
                    D.dflash_committed(s_, f, lo)
                    del f
                D.dflash_flush([s_])
                feats = torch.randn((W + K + 1, P_ROWS, cfg.feature_width), generator=g,
                                    device=dev).to(torch.bfloat16)
                tl = (torch.randn((1, n + 1, cfg.vocab), generator=g, device=dev) * 3.0).contiguous()
                cur = torch.full((1,), 17, dtype=torch.int32, device=dev)
                tok = torch.empty((1, n), dtype=torch.int32, device=dev)
                q = torch.empty((1, n), dtype=torch.float32, device=dev)
                acc = torch.empty(1, dtype=torch.int32, device=dev)
                bon = torch.empty(1, dtype=torch.int32, device=dev)

            def step(i):
                D.dflash_committed(s_, feats[i], T + P_ROWS * i)
                D.dflash_propose([s_], cur, n, TEMP, SEED, i, tok, q)
                D.dflash_verify([s_], tl, tok, n, TEMP, SEED, i, acc, bon)

            ms, clk = _timed(torch, stream, step, K, W, local_rank, world, dev)
            rb = round_bytes(cfg, T, P_ROWS)
            res[bs] = (world * K / (ms * 1e-3), ms, clk, rb, _launches_per_step(D, model, stream, step, torch, K + W))
            D.dflash_close(s_)
            del model
            torch.cuda.empty_cache()
        v16, ms16, clk16, rb16, launches16 = res[16]
        gbs = rb16 / (ms16 / K * 1e-3) / 1e9
        return _line("draft rounds/s (Laguna-style gated window-512 draft, bs1, block 16)", "draft rounds/s", v16,
                     world, K, W, ms16, "bf16",
                     {"workload": "laguna_bf16: 4 layers, H 3072, 24/8 heads x 128, I 8192 (assumed), V 100352, "
                                  "window 512 over a 32768-row temporal context, 4 committed rows per round, T=1.0",
                      "l2": f"no flush: {rb16 / 1e9:.2f} GB of weights, K/V and logits per round"},
                     {"roofline": {"kernel": "whole round (weight-streaming GEMMs dominate)", "bound": "hbm",
                                   "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                   "frac": round(gbs / peaks["hbm_gbs"], 4),
                                   "peak_kind": f"{peak_kind} HBM copy bandwidth",
                                   "algorithmic_bytes_per_step": rb16, "traffic": None},
                      "gpu_launches": launches16 * K,
                      "block8_rounds_s": round(res[8][0], 2),
                      "block8_round_roofline_frac": round(res[8][3] / (res[8][1] / K * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                                          4)}, clk16)

    if args.workload == "spec":
        return _spec_decode(args, world, local_rank, dev, stream, K, W)
    if args.workload == "truncated":
        return _truncated_round(args, world, local_rank, dev, stream, K, W, peaks, peak_kind)

    # batched serving mix
    cfg = S.CONFIGS[CFG_NAME]
    if args.small:
        cfg = cfg.replace(n_layers=1, vocab=32000, mask_token=31999)
    B, n, Tb = 64, cfg.block_size - 1, 0.7
    ctxs = np.random.default_rng(0).integers(1024, 16385, size=B)
    model = D.dflash_model_create(cfg, gpu_weights(cfg, SEED + rank, dev))
    with torch.cuda.stream(stream):
        sess = []
        for b in range(B):
            c = int(ctxs[b])
            s_ = D.dflash_open(model, restored_offset=c, max_ctx=c + P_ROWS * (K + W + 4) + 64, stream=stream)
            for l in range(cfg.n_layers):      # restored context: seeded K/V rows
                kk = torch.randn((cfg.n_kv_heads, c, cfg.head_dim), generator=g, device=dev).to(torch.bfloat16)
                vv = torch.randn((cfg.n_kv_heads, c, cfg.head_dim), generator=g, device=dev).to(torch.bfloat16)
                D.dflash_kv_import(s_, l, 0, c, kk, vv)
                del kk, vv
            sess.append(s_)
        feats = torch.randn((B, P_ROWS, cfg.feature_width), generator=g, device=dev).to(torch.bfloat16)
        tl = (torch.randn((B, n + 1, cfg.vocab), generator=g, device=dev) * 3.0).contiguous()
        cur = torch.randint(0, cfg.vocab, (B,), generator=g, device=dev, dtype=torch.int32)
        tok = torch.empty((B, n), dtype=torch.int32, device=dev)
        q = torch.empty((B, n), dtype=torch.float32, device=dev)
        acc = torch.empty(B, dtype=torch.int32, device=dev)
        bon = torch.empty(B, dtype=torch.int32, device=dev)

    feat_list = [feats[b] for b in range(B)]

    def step(i):
        D.dflash_committed_batch(sess, feat_list, [int(c) + P_ROWS * i for c in ctxs])
        D.dflash_propose(sess, cur, n, Tb, SEED, i, tok, q)
        D.dflash_verify(sess, tl, tok, n, Tb, SEED, i, acc, bon)

    ms, clk = _timed(torch, stream, step, K, W, local_rank, world, dev)
    launches, classes = _instrumented_step(D, model, stream, step, torch, K + W)
    H, I, V = cfg.hidden, cfg.intermediate, cfg.vocab
    per_layer = cfg.qkv_rows * H + H * cfg.n_q_heads * cfg.head_dim + 3 * H * I
    gemm_flops = 2.0 * (B * (n + 1) * (cfg.n_layers * per_layer) + B * n * V * H +
                        B * P_ROWS * (H * cfg.feature_width + cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim * H))
    kv_bytes = float(sum(int(c) + 2 * P_ROWS * (K + W) // 2 + n + 1 for c in ctxs)) * cfg.n_layers * 2 * \
        cfg.n_kv_heads * cfg.head_dim * 2
    t_step = ms / K * 1e-3
    ideal = gemm_flops / (peaks.get("bf16_tflops_sustained", 1700.0) * 1e12) + \
        (kv_bytes + B * (n + 1) * V * 4) / (peaks["hbm_gbs"] * 1e9)
    D.dflash_device_status(model)
    for s_ in sess:
        D.dflash_close(s_)
    shape = "Qwen3-8B-shaped draft" if not args.small else "Qwen3-8B-shaped draft cut to 1 layer and V 32000 (--small)"
    return _line(f"proposed tok/s (bs64 serving mix, {shape}, block 16, ctx 1k-16k)", "proposed tok/s",
                 world * B * n / t_step, world, K, W, ms, "bf16",
                 {"workload": "64 sequences, contexts uniform 1k-16k (seeded K/V), 4 committed rows each per round, "
                              "batched propose + rejection-sampling verify at T=0.7 on N(0,3) target logits "
                              "[64,16,151936]", "l2": "no flush: 11+ GB of K/V and 3.4 GB of weights per round"},
                 {"rounds_s": round(world / t_step, 2), "gpu_launches": launches * K,
                  "kernel_classes_instrumented_one_step": classes,
                  "roofline": {"bound": "mixed (GEMMs tensor, attention and verify HBM)",
                               "ideal_ms_per_step": round(ideal * 1e3, 3), "frac": round(ideal / t_step, 4),
                               "gemm_tflop_per_step": round(gemm_flops / 1e12, 3),
                               "kv_gb_per_step": round(kv_bytes / 1e9, 2)}}, clk)


def _truncated_round(args, world, local_rank, dev, stream, K, W, peaks, peak_kind):
    """The bs1 Qwen3-8B-shaped round at T = 1 with the session's sampler
    truncating to top-k 40 / top-p 0.9 (draft rows and target rows), timed
    against the same round with full distributions, alternating on one box.
    The truncation's own cost is the cut kernel (k_trunc_cut): one CTA per row
    reads the row of logits five times (four radix passes and the gather),
    from L2."""
    import torch

    import block_diffusion_speculative_flush_gb300 as D
    import synthetic as S

    cfg = S.CONFIGS[CFG_NAME]
    n, V = cfg.block_size - 1, cfg.vocab
    model = D.dflash_model_create(cfg, gpu_weights(cfg, SEED, dev))
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 11)
    start = CTX - P_ROWS * (W + K)
    sess = {}
    with torch.cuda.stream(stream):
        for name in ("full", "trunc"):
            s_ = D.dflash_open(model, max_ctx=start + P_ROWS * (2 * (W + K) + 8), stream=stream)
            for lo in range(0, start, 1024):
                f = torch.randn((min(start, lo + 1024) - lo, cfg.feature_width), generator=g,
                                device=dev).to(torch.bfloat16)
                D.dflash_committed(s_, f, lo)
                del f
            D.dflash_flush([s_])
            sess[name] = s_
        D.dflash_set_sampler(sess["trunc"], 40, 0.9, 0.0)
        feats = torch.randn((W + K, P_ROWS, cfg.feature_width), generator=g, device=dev).to(torch.bfloat16)
        tl = (torch.randn((1, n + 1, V), generator=g, device=dev) * 3.0).contiguous()
        cur = torch.full((1,), 17, dtype=torch.int32, device=dev)
        tok = torch.empty((1, n), dtype=torch.int32, device=dev)
        q = torch.empty((1, n), dtype=torch.float32, device=dev)
        acc = torch.empty(1, dtype=torch.int32, device=dev)
        bon = torch.empty(1, dtype=torch.int32, device=dev)
    res = {}
    for name in ("full", "trunc", "full", "trunc"):          # alternate: two timed runs each
        s_ = sess[name]
        base = D.dflash_session_state(s_)[0] + D.dflash_session_state(s_)[1]

        def step(i, s_=s_, base=base):
            D.dflash_committed(s_, feats[i % (W + K)], base + P_ROWS * i)
            D.dflash_propose([s_], cur, n, TEMP, SEED, i, tok, q)
            D.dflash_verify([s_], tl, tok, n, TEMP, SEED, i, acc, bon)

        ms, clk = _timed(torch, stream, step, K // 2, W, local_rank, world, dev)
        # the W warm-up steps advanced the cursor too: base moves on for the next run
        prev = res.get(name, (0.0, 0, None))
        res[name] = (prev[0] + ms, prev[1] + K // 2, clk)
    D.dflash_device_status(model)
    for s_ in sess.values():
        D.dflash_close(s_)
    ms_t, k_t, clk = res["trunc"]
    ms_f, k_f, _ = res["full"]
    v_t, v_f = world * k_t / (ms_t * 1e-3), world * k_f / (ms_f * 1e-3)
    rows = 2 * n + 1                                            # n proposal rows + n + 1 target rows
    return _line("draft rounds/s (bs1 Qwen3-8B-shaped round, top-k 40 / top-p 0.9 sampler)", "draft rounds/s", v_t,
                 world, k_t, W, ms_t, "bf16",
                 {"workload": "qwen3_8b_bf16 draft round, bs1, block 16 (n=15), ctx ~4096, 4 committed rows per "
                              "round, T=1.0, session sampler top_k 40, top_p 0.9 on the 15 draft rows and the 16 "
                              "target rows [1,16,151936]", "l2": "no flush: 3.4 GB of weights streamed per step"},
                 {"full_distribution_rounds_s": round(v_f, 2),
                  "truncation_cost_us_per_round": round((ms_t / k_t - ms_f / k_f) * 1e3, 2),
                  "cut_rows_per_round": rows,
                  "cut_algorithmic_bytes_per_round": rows * V * 4}, clk)


def _spec_decode(args, world, local_rank, dev, stream, K, W):
    """Whole greedy speculative rounds on the GPU: the tiny fp32 draft proposes
    7 tokens, the synthetic 2-layer target runs its 8-row verify forward (logits
    and the 5 hidden taps), verify takes the accepted prefix and the bonus
    token, the target cache is trimmed to the accepted rows and their taps are
    committed to the draft.  The accept length is read on the host every round
    (trim and commit take host integers), so a step ends in one device sync."""
    import numpy as np
    import torch

    import block_diffusion_speculative_flush_gb300 as D
    import synthetic as S
    from synthetic.target import TARGET_TINY, make_target_weights

    cfg = S.CONFIGS["tiny_fp32"]
    n = cfg.block_size - 1
    ts = TARGET_TINY
    hw = make_target_weights(1, ts)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    tw = dict(embed=f32(hw["embed"]), unembed=f32(hw["unembed"]), final_norm=f32(hw["final_norm"]),
              layers=[{k: f32(v) for k, v in lw.items()} for lw in hw["layers"]])
    model = D.dflash_model_create(cfg, gpu_weights(cfg, SEED, dev))
    max_ctx = 16 + (n + 1) * (W + K + 2)
    V, NT = ts.vocab, ts.n_taps * ts.hidden
    prompt = [int(x) for x in S.rng_for(0, "prompt").integers(0, V, size=8)]
    with torch.cuda.stream(stream):
        tgt = D.dflash_target_create(ts.as_dict(), tw, max_ctx=max_ctx, stream=stream)
        sess = D.dflash_open(model, max_ctx=max_ctx, stream=stream)
        lg_p = torch.empty((len(prompt), V), dtype=torch.float32, device=dev)
        tp_p = torch.empty((len(prompt), NT), dtype=torch.float32, device=dev)
        D.dflash_target_forward(tgt, torch.tensor(prompt, dtype=torch.int32, device=dev), 0, lg_p, tp_p)
        cur = torch.empty(1, dtype=torch.int32, device=dev)
        D.dflash_target_argmax(tgt, lg_p[-1:], cur)
        D.dflash_committed(sess, tp_p, 0)
        blk = torch.empty(n + 1, dtype=torch.int32, device=dev)
        lg = torch.empty((n + 1, V), dtype=torch.float32, device=dev)
        tp = torch.empty((n + 1, NT), dtype=torch.float32, device=dev)
        tok = blk[1:].view(1, n)
        q = torch.empty((1, n), dtype=torch.float32, device=dev)
        acc = torch.empty(1, dtype=torch.int32, device=dev)
        bon = torch.empty(1, dtype=torch.int32, device=dev)
        host = torch.empty(2, dtype=torch.int32, pin_memory=True)
    st = {"pos": len(prompt), "tokens": 0, "accepted": 0}

    def step(i):
        if i == W:          # first timed step: count tokens from here
            st["mark_tokens"], st["mark_accepted"] = st["tokens"], st["accepted"]
        blk[:1].copy_(cur)
        D.dflash_propose([sess], cur, n, 0.0, 0, i, tok, q)
        D.dflash_target_forward(tgt, blk, st["pos"], lg, tp)
        D.dflash_verify([sess], lg[None], tok, n, 0.0, 0, i, acc, bon)
        host[:1].copy_(acc, non_blocking=True)
        stream.synchronize()
        a = int(host[0])
        D.dflash_target_trim(tgt, st["pos"] + a + 1)
        D.dflash_committed(sess, tp[:a + 1], st["pos"])
        cur.copy_(bon)
        st["pos"] += a + 1
        st["tokens"] += a + 1
        st["accepted"] += a

    ms, clk = _timed(torch, stream, step, K, W, local_rank, world, dev)
    timed_tokens = st["tokens"] - st["mark_tokens"]
    timed_accepted = st["accepted"] - st["mark_accepted"]
    # the target's verify forward alone (8 rows at the cached frontier, trimmed back each time)
    fw = torch.cuda.Event(enable_timing=True)
    fe = torch.cuda.Event(enable_timing=True)
    base = st["pos"]
    with torch.cuda.stream(stream):
        for _ in range(3):
            D.dflash_target_forward(tgt, blk, base, lg, tp)
            D.dflash_target_trim(tgt, base)
        fw.record(stream)
        for _ in range(50):
            D.dflash_target_forward(tgt, blk, base, lg, tp)
            D.dflash_target_trim(tgt, base)
        fe.record(stream)
    torch.cuda.synchronize()
    fwd_us = fw.elapsed_time(fe) / 50 * 1e3
    D.dflash_target_device_status(tgt)
    D.dflash_device_status(model)
    D.dflash_close(sess)
    launches_fwd = 2 + 14 * ts.n_layers + 2 + 1
    return _line("generated tok/s (greedy speculative decoding, tiny fp32 draft + synthetic target, on GPU)",
                 "generated tok/s", world * timed_tokens / (ms * 1e-3), world, K, W, ms, "f32",
                 {"workload": "tiny_fp32 draft (2 layers, H 256, block 8, n=7) + a 2-layer H-256 fp32 target, "
                              "8-token prompt, greedy rounds: propose, 8-row target verify forward with 5 taps, "
                              "verify, trim, commit", "l2": "all weights (6 MB) L2-resident: latency-bound"},
                 {"rounds_s": round(world * K / (ms * 1e-3), 2),
                  "mean_accepted": round(timed_accepted / K, 3),
                  "target_forward_us": round(fwd_us, 2), "target_forward_launches": launches_fwd,
                  "total_tokens": timed_tokens}, clk)


# ---------------------------------------------------------------------------
# the CPU oracle: baseline leg and reference arm
# ---------------------------------------------------------------------------
def _oracle_setup(cfg, host_w):
    import numpy as np

    import synthetic as S
    from oracle import dflash_oracle as O
    d = O.OracleDraft(cfg, host_w)
    Kc = S.make_kv(cfg, CTX, SEED, "ctx_k").astype(np.float64)
    Vc = S.make_kv(cfg, CTX, SEED, "ctx_v").astype(np.float64)
    cache = {s: (Kc[:, :, s, :], Vc[:, :, s, :]) for s in range(CTX)}
    feats = S.make_features(cfg, P_ROWS, seed=SEED)
    n = cfg.block_size - 1
    tl = np.random.default_rng(SEED).standard_normal((n + 1, cfg.vocab)) * 3.0
    return O, d, cache, feats, tl


def _threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count() or 1])
    except ImportError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu on Arm hosts, /proc/cpuinfo elsewhere)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_sample_child():
    """One bounded sample of the round on the oracle, in a fresh process whose
    BLAS runs one thread: the context path of the 4 held rows, one draft layer
    (its K/V of the new rows and the 16-row block layer at ctx 4096), 1/16 of
    the unembedding, and the draw + verify over the whole vocabulary.  Prints
    the times as JSON, with the round time extrapolated as
    start + L * layer + 16 * unembed slice + finish."""
    import numpy as np

    import synthetic as S
    from oracle import dflash_oracle as O
    cfg = S.CONFIGS[CFG_NAME]
    L, n, V, H = cfg.n_layers, cfg.block_size - 1, cfg.vocab, cfg.hidden
    J = 16
    names = ["aux_norms", "w_fc", "hidden_norm", "final_norm"] + \
        [k for k in S.weight_shapes(cfg) if k.startswith("layers.0.")]
    w = S.make_weights(cfg, seed=SEED, names=names)
    # the embedding is only gathered (two rows) and 1/16 of the unembedding is
    # read: untouched zero pages stand for the rest
    w["embed"] = np.zeros((V, H), dtype=np.float32)
    w["unembed"] = np.zeros((V, H), dtype=np.float32)
    w["unembed"][: V // J] = S.normal(SEED, "unembed", (V // J, H), std=0.02, dtype="bf16")
    d = O.OracleDraft(cfg, w)
    feats = S.make_features(cfg, P_ROWS, seed=SEED)
    Kc = S.make_kv(cfg, CTX - P_ROWS, SEED, "ctx_k")[0].transpose(1, 0, 2).astype(np.float64)
    Vc = S.make_kv(cfg, CTX - P_ROWS, SEED, "ctx_v")[0].transpose(1, 0, 2).astype(np.float64)
    tl = np.random.default_rng(SEED).standard_normal((n + 1, V)) * 3.0
    t = {}
    t0 = time.perf_counter()
    hid = d.context_hidden(feats)
    h = d.w.rows("embed", [17] + [cfg.mask_token] * n)
    t["start"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    ck, cv = d.context_layer_kv(0, hid, np.arange(CTX - P_ROWS, CTX))
    h = d.block_layer(0, h, CTX + np.arange(n + 1, dtype=np.float64), np.concatenate([Kc, ck]),
                      np.concatenate([Vc, cv]), np.arange(CTX, dtype=np.float64))
    t["layer"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    lg = np.zeros((n, V))
    lg[:, : V // J] = d.unembed(h[1:], 0, V // J)
    t["unembed_slice"] = time.perf_counter() - t0
    t0 = time.perf_counter()
    toks, _, _ = O.sample_rows(lg, TEMP, SEED, 0, 0)
    O.verify(tl, toks, lg, toks, TEMP, TEMP, SEED, 0, 0)
    t["finish"] = time.perf_counter() - t0
    t["round_s"] = t["start"] + L * t["layer"] + J * t["unembed_slice"] + t["finish"]
    print(json.dumps(t), flush=True)


def _oracle_samples(nproc: int):
    """Runs _oracle_sample_child in nproc fresh single-threaded processes at
    once; returns their results and the wall time."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    cmd = [sys.executable, "-c", "import bench; bench._oracle_sample_child()"]
    t0 = time.perf_counter()
    procs = [subprocess.Popen(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for _ in range(nproc)]
    outs = []
    for pr in procs:
        out, _ = pr.communicate(timeout=600)
        if pr.returncode == 0 and out.strip():
            outs.append(json.loads(out.strip().splitlines()[-1]))
    return outs, time.perf_counter() - t0


def cpu_baseline(cfg, host_w):
    """One whole round of the oracle on the host with every BLAS thread: 4
    held rows through the context path, the 16-row block at ctx 4096 (context
    K/V seeded directly), the unembedding, the draw, and the verify.  Then a
    bounded single-thread sample of the round (extrapolated to a round), and
    the same sample in one single-threaded process per host core at once
    (independent sequences)."""
    O, d, cache, feats, tl = _oracle_setup(cfg, host_w)
    n = cfg.block_size - 1
    s = O.OracleSession(d, restored_offset=CTX - P_ROWS, restored_cache={k: v for k, v in cache.items()
                                                                          if k < CTX - P_ROWS})
    s.committed(feats, CTX - P_ROWS)
    t0 = time.perf_counter()
    out = s.propose(17, n, TEMP, SEED, 0)
    s.verify(tl, out["tokens"], TEMP, SEED, 0)
    dt = time.perf_counter() - t0
    del d, cache, s
    res = {"value": round(1.0 / dt, 5), "unit": UNIT, "cores": _threads(), "kind": "oracle",
           "sample": f"one whole round on the host ({dt:.1f} s): 4 held rows, 16-row block at ctx 4096 "
                     "(context K/V seeded directly), unembedding, draw and verify; float64 numpy",
           "cpu_model": cpu_model(), "nproc": os.cpu_count()}
    one, _ = _oracle_samples(1)
    if one:
        res["single_thread"] = {"rounds_s": round(1.0 / one[0]["round_s"], 5), "round_s": round(one[0]["round_s"], 2),
                                "sample": "context path + 1 of 5 layers + 1/16 of the unembedding + draw and "
                                          "verify, one BLAS thread, extrapolated to a round", "times_s": one[0]}
    N = os.cpu_count() or 1
    many, wall = _oracle_samples(N)
    if many:
        res["n_process"] = {"processes": len(many),
                            "rounds_s": round(sum(1.0 / m["round_s"] for m in many), 5),
                            "sample": "the single-thread sample in one process per core at once, one sequence "
                                      "each; rounds/s summed over the processes", "wall_s": round(wall, 1)}
    return res


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host's cores.  The round is cut
    into its oracle calls in order (context hidden rows, then per layer the
    new rows' K/V and the block layer, then vocabulary slices of the
    unembedding, then the draw and the verify); the K timed steps share those
    calls out in order, so together they run exactly one round and
    value = 1 / (sum of the K step times) rounds/s.  The W warm-up steps run
    one more round the same way.  The whole run costs about two rounds."""
    if rank != 0:
        return None
    import numpy as np

    import synthetic as S
    cfg = S.CONFIGS[CFG_NAME]
    rng = np.random.default_rng(SEED)
    host_w = {}
    for name, shape in S.weight_shapes(cfg).items():
        x = rng.standard_normal(shape, dtype=np.float32) * np.float32(0.02)
        if name.endswith("norm") or name == "aux_norms":
            x += np.float32(1.0)
        host_w[name] = S.to_dtype_values(x, "bf16")
    O, d, cache, feats, tl = _oracle_setup(cfg, host_w)
    L, n, V = cfg.n_layers, cfg.block_size - 1, cfg.vocab
    F0 = CTX - P_ROWS
    ctx_pos = np.arange(CTX, dtype=np.float64)
    slots = np.arange(F0, CTX)
    tokens = [17] + [cfg.mask_token] * n
    pos = CTX + np.arange(n + 1, dtype=np.float64)
    ctx_k = [np.stack([cache[s][0][l] for s in range(F0)]) for l in range(L)]
    ctx_v = [np.stack([cache[s][1][l] for s in range(F0)]) for l in range(L)]
    st = {}

    def start(rnd):
        st["rnd"] = rnd
        st["hid"] = d.context_hidden(feats)
        st["h"] = d.w.rows("embed", tokens)
        st["logits"] = np.zeros((n, V))

    def layer(l):
        ck, cv = d.context_layer_kv(l, st["hid"], slots)
        st["h"] = d.block_layer(l, st["h"], pos, np.concatenate([ctx_k[l], ck]), np.concatenate([ctx_v[l], cv]),
                                ctx_pos)

    def unembed(j, J):
        lo, hi = j * V // J, (j + 1) * V // J
        st["logits"][:, lo:hi] = d.unembed(st["h"][1:], lo, hi)

    def finish():
        toks, _, _ = O.sample_rows(st["logits"], TEMP, SEED, st["rnd"], 0)
        O.verify(tl, toks, st["logits"], toks, TEMP, TEMP, SEED, st["rnd"], 0)

    J = 8
    calls = [start] + [(lambda l=l: layer(l)) for l in range(L)] + [(lambda j=j: unembed(j, J)) for j in range(J)] \
        + [finish]

    def run_round(rnd, steps):
        """Runs one round as `steps` steps; returns each step's seconds."""
        st["rnd_arg"] = rnd
        times = []
        c = 0
        for k in range(steps):
            hi = (k + 1) * len(calls) // steps
            t0 = time.perf_counter()
            while c < hi:
                f = calls[c]
                f(rnd) if f is start else f()
                c += 1
            times.append(time.perf_counter() - t0)
        return times

    run_round(0, max(1, args.warmup))
    times = run_round(1, args.steps)
    per_round = sum(times)
    value = 1.0 / per_round
    sample = (f"the {args.steps} timed steps together run one whole round ({per_round:.1f} s): 4 held rows, "
              f"16-row block at ctx 4096 (context K/V seeded directly), unembedding, draw and verify, "
              f"each step a contiguous slice of the round's oracle calls; float64 numpy")
    return {
        "metric": METRIC, "value": round(value, 5), "unit": UNIT, "impl": "reference", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_round * 1e3 / args.steps, 2),
        "ms_per_round": round(per_round * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (random-init draft weights, N(0,1) features, N(0,3) target logits)",
        "config": {"workload": "qwen3_8b_bf16 draft round, bs1, block 16 (n=15), ctx 4096, "
                               "4 committed rows per round, T=1.0", "l2": "host run"},
        "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": _threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    global PROFILE_RANGE
    args = parse_args(argv)
    PROFILE_RANGE = args.profile_range
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    elif args.workload != "round":
        out = run_workload(args, rank, world, local_rank)
    else:
        out = run_ours(args, rank, world, local_rank)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
