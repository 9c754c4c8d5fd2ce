#!/usr/bin/env python3
"""Benchmark of the KIVI hot path on GB300 (libkivi through its C ABI).

One step = one pass of the whole path over one batch of the workload:
prefix encode of keys and values (quantize + pack + residual copy),
materialize both back to fp16, append one decoded token per sequence, and
fused-dequant decode attention (q.K_hat^T, softmax, p.V_hat).  The default
workload is the Llama-2-7B-shaped layer: K, V fp16 [8, 32, 4096, 128],
int2 keys and values, G = 32, R = 128, q [8, 32, 1, 128].

Metric: fp16-equivalent KV gigabytes per second over the step (the fp16 bytes
of K and V the step encodes, materializes and attends over, divided by the
step time), with decode tokens/s and per-kernel HBM roofline fractions.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Under torchrun each rank runs an independent replica on its own GPU (the path
has no cross-GPU exchange); the timed region is bracketed by barriers and the
slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV quant/dequant GB/s (fp16-equiv) & decode-attn tok/s; % of HBM roofline"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20     # GB300 L2
ROTATE_MIN_BYTES = 2 * L2_BYTES  # decode-only working sets rotate over at least this much


# ------------------------------------------------------------------ setup --

def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="kivi", choices=["kivi", "reference"])
    p.add_argument("--workload", default="llama2_7b_layer")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-c2c", action="store_true")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other workloads' per-kernel lines (run before the headline timing)")
    p.add_argument("--workload-steps", type=int, default=200)
    p.add_argument("--decode", default="fused", choices=["fused", "split"],
                   help="decode through kivi_decode_attention (fused) or kivi_decode_qk + kivi_decode_pv")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "kivi_bit_kv_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel
    sources are unchanged since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[workload][kernel]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


def queue_ahead(torch, ms: float = 2.0) -> None:
    """A device-side busy wait of about `ms` (at up to 2.07 GHz) on the current
    stream, issued just before the start event of a timed region: while it
    runs, the host enqueues the first timed steps, so the events time the
    device's work and not the host's launch of the first call (with the queue
    empty at the start event, the first step's first call measured about
    40 us too long)."""
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(int(ms * 2.07e6))


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[2:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, flags in rows:
            for n, v in zip(names, flags[1:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------- byte accounting --

# How each workload is stepped: "full" = encode + materialize + append +
# decode of one batch; "store" = encode + materialize (the exact-prefix store
# round trip); "decode" / "stream" = append + decode on a cache encoded once
# before the timed region (the cache grows by one token per step).
KINDS = {"tiny": "full", "llama2_7b_layer": "full", "prefix_store_int4": "store",
         "prefix_store_int8": "store", "mistral_gqa": "decode", "streaming": "stream"}
STEP_CALLS = {
    "full": ["quant_keys", "quant_values", "dequant_keys", "dequant_values", "append", "decode"],
    "store": ["quant_keys", "quant_values", "dequant_keys", "dequant_values"],
    "decode": ["append", "decode"],
    "stream": ["append", "decode"],
}
# "decode" is the fused kivi_decode_attention (--decode fused, the default) or
# kivi_decode_qk followed by kivi_decode_pv (--decode split).
DECODE_CALLS = {"fused": ["decode_attn"], "split": ["decode_qk", "decode_pv"]}
LAUNCHES = {"quant_keys": 1, "quant_values": 1, "dequant_keys": 1, "dequant_values": 1,
            "append": 2, "decode_qk": 1, "decode_pv": 2, "decode_attn": 2}  # + combine kernels


def step_calls(w, kind: str, decode: str) -> list:
    mode = decode
    out = []
    for c in STEP_CALLS[kind]:
        out += DECODE_CALLS[mode] if c == "decode" else [c]
    return out


def _split(n, G, R):
    tq = max(0, (int(n) - R) // G * G)
    return tq, int(n) - tq


def slice_bytes(w, n: int, which: int) -> int:
    """Stored bytes of one (b, h) slice holding n tokens: codes + fp32
    scale/zero + fp16 residual (keys: which = 0, values: which = 1)."""
    tq, res = _split(n, w.G, w.R)
    bits = w.bits_k if which == 0 else w.bits_v
    stats = (tq // w.G) * w.D * 8 if which == 0 else tq * (w.D // w.G) * 8
    return tq * w.D * bits // 8 + stats + res * w.D * 2


def call_bytes(w, enc_lens, dec_lens) -> dict:
    """Algorithmic HBM bytes (read + write) of each call of one step.

    enc_lens[b]: tokens of sequence b encoded / materialized; dec_lens[b]:
    tokens the decode attends over (after the append)."""
    H, Hq, D = w.H, w.Hq, w.D
    fp16 = sum(H * int(n) * D * 2 for n in enc_lens)
    kst = sum(H * slice_bytes(w, n, 0) for n in enc_lens)
    vst = sum(H * slice_bytes(w, n, 1) for n in enc_lens)
    kdec = sum(H * slice_bytes(w, n, 0) for n in dec_lens)
    vdec = sum(H * slice_bytes(w, n, 1) for n in dec_lens)
    logits = sum(Hq * int(n) * 4 for n in dec_lens)
    B = len(dec_lens)
    return {
        "quant_keys": fp16 + kst, "quant_values": fp16 + vst,
        "dequant_keys": kst + fp16, "dequant_values": vst + fp16,
        "append": B * H * D * 2 * 4,
        "decode_qk": kdec + B * Hq * D * 2 + logits,
        "decode_pv": vdec + logits + B * Hq * D * 4,
        "decode_attn": kdec + vdec + B * Hq * D * 2 + B * Hq * D * 4,
    }


def fp16_equiv_bytes(w, kind: str, enc_lens, dec_lens) -> int:
    """fp16 K+V bytes the step encodes, materializes and attends over."""
    H, D = w.H, w.D
    enc = sum(2 * H * int(n) * D * 2 for n in enc_lens)
    dec = sum(2 * H * int(n) * D * 2 for n in dec_lens)
    app = 2 * len(dec_lens) * H * D * 2
    return {"full": 2 * enc + dec + app, "store": 2 * enc}.get(kind, dec + app)


def reduce_max(value: float, device="cpu") -> float:
    """Max of `value` over the ranks of the default process group (identity
    when there is none): the slowest replica defines the job time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(bytes_per_rank: float, world: int, ms_per_step: float) -> float:
    """Job throughput in GB/s: every replica moves the same bytes per step,
    and the step lasts as long as the slowest replica."""
    return bytes_per_rank * world / (ms_per_step * 1e-3) / 1e9


# --------------------------------------------------------------- GPU arm --

def cache_copies(w, lens, Tmax) -> int:
    """Caches a decode-only workload rotates over, so that one step's packed
    cache is gone from L2 when it comes round again (the copies together
    hold at least twice the L2)."""
    per = sum(w.H * (slice_bytes(w, int(n), 0) + slice_bytes(w, int(n), 1)) for n in lens)
    return max(1, -(-ROTATE_MIN_BYTES // max(1, per)))


def l2_note(kind: str, copies: int, per_copy: int) -> str:
    if kind in ("full", "store"):
        return "fp16 K/V and packed cache of a step larger than 2x L2 (no flush needed)"
    if copies == 1:
        return f"packed cache {per_copy / 2**20:.0f} MB, larger than 2x L2 (no rotation needed)"
    return (f"{copies} caches of {per_copy / 2**20:.0f} MB rotated step by step "
            f"({copies * per_copy / 2**20:.0f} MB, at least 2x L2)")


def run_secondary(name, steps, warmup, dev, decode="fused") -> dict:
    """Per-call times, algorithmic bytes and roofline fractions of another
    workload, measured the same way as the headline one (bounded steps)."""
    import numpy as np
    import torch
    from kivi_bit_kv_gb300 import KiviCache, abi
    from kivi_bit_kv_gb300 import workloads as W
    w = W.WORKLOADS[name]
    kind = KINDS[name]
    calls = step_calls(w, kind, decode)
    grows = kind in ("decode", "stream")
    lens0 = W.make_lengths(w).numpy().astype(np.int64)
    n_app = warmup + steps if grows else 1
    Tmax = (int(lens0.max()) + n_app + w.G) // w.G * w.G + w.G
    seq_lens = None if w.ragged is None else torch.as_tensor(lens0.astype(np.int32), device=dev)
    K, V = W.make_kv(w, device=dev)
    ncp = cache_copies(w, lens0, Tmax) if grows else 1
    caches = [KiviCache(w.B, w.H, w.D, w.bits_k, w.bits_v, w.G, w.R, Tmax, device=dev) for _ in range(ncp)]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    ld = (Tmax + 3) // 4 * 4
    logits = torch.empty((w.B, w.Hq, ld), dtype=torch.float32, device=dev) if decode == "split" else None
    wss = [c.workspace(w.Hq) for c in caches]
    if grows:
        for c in caches:
            abi.kivi_quant_keys(c, K, seq_lens)
            abi.kivi_quant_values(c, V, seq_lens)
        torch.cuda.synchronize(dev)
        del K, V
        torch.cuda.empty_cache()
        kh = vh = None
    else:
        kh = torch.empty((w.B, w.H, w.T, w.D), dtype=torch.float16, device=dev)
        vh = torch.empty_like(kh)
    kn, vn = W.make_step_tokens(w, n_app, device=dev)
    qs = torch.stack([W.make_q(w, dev, step=s) for s in range(n_app)]) if grows else W.make_q(w, dev)[None]
    stream = torch.cuda.current_stream(dev)

    def step(i, ev=None):
        c = caches[i % ncp]
        j = i if grows else 0
        fns = {
            "quant_keys": lambda: abi.kivi_quant_keys(c, K, seq_lens),
            "quant_values": lambda: abi.kivi_quant_values(c, V, seq_lens),
            "dequant_keys": lambda: abi.kivi_dequant(c, 0, kh),
            "dequant_values": lambda: abi.kivi_dequant(c, 1, vh),
            "append": lambda: abi.kivi_append_token(c, kn[j], vn[j], status),
            "decode_qk": lambda: abi.kivi_decode_qk(c, qs[j], logits),
            "decode_pv": lambda: abi.kivi_decode_pv(c, logits, out, wss[i % ncp]),
            "decode_attn": lambda: abi.kivi_decode_attention(c, qs[j], out, wss[i % ncp]),
        }
        for c_i, nm in enumerate(calls):
            if ev is not None:
                ev[2 * c_i].record(stream)
            fns[nm]()
            if ev is not None:
                ev[2 * c_i + 1].record(stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(calls))] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    queue_ahead(torch)
    t0.record(stream)
    for s_ in range(steps):
        step(warmup + s_, evs[s_])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0, "a sequence ran out of capacity"
    if "decode_attn" in calls:
        for ws_ in wss:
            assert int(ws_[:1].view(torch.int32).item()) == 0, "decode status word"
    per_call = {c: sum(evs[s_][2 * i].elapsed_time(evs[s_][2 * i + 1]) for s_ in range(steps)) / steps
                for i, c in enumerate(calls)}
    ms_step = t0.elapsed_time(t1) / steps
    if grows:
        timed = [lens0 + (warmup + s_) // ncp + 1 for s_ in range(steps)]
        pick = timed[:: max(1, len(timed) // 16)]
        ab_list = [call_bytes(w, d, d) for d in pick]
        ab = {k: sum(a[k] for a in ab_list) / len(ab_list) for k in ab_list[0]}
    else:
        ab = call_bytes(w, lens0, lens0 + 1)
    hbm, _ = peaks()
    kernels = {}
    for c in calls:
        gbs = ab[c] / (per_call[c] * 1e-3) / 1e9
        kernels[c] = {"ms": round(per_call[c], 5), "alg_bytes": int(ab[c]), "gbs": round(gbs, 1),
                      "frac": round(gbs / hbm, 3)}
    per_copy = sum(w.H * (slice_bytes(w, int(n), 0) + slice_bytes(w, int(n), 1)) for n in lens0)
    res = {"step": kind, "shape": [w.B, w.H, w.T, w.D], "Hq": w.Hq, "bits_k": w.bits_k, "bits_v": w.bits_v,
           "steps": steps, "warmup": warmup, "ms_per_step": round(ms_step, 5), "kernels": kernels,
           "l2": l2_note(kind, ncp, per_copy)}
    if kind != "store":
        dec_ms = sum(per_call[c] for c in calls if c.startswith("decode"))
        res["decode_tok_s"] = round(w.B / (dec_ms * 1e-3), 1)
    del caches, wss
    torch.cuda.empty_cache()
    return res


def run_kivi(args, rank, world, local):
    import numpy as np
    import torch
    from kivi_bit_kv_gb300 import KiviCache, abi
    from kivi_bit_kv_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if dist.is_nccl_available() else "gloo")
    w = W.WORKLOADS[args.workload]
    kind = KINDS[w.name]
    # the other workloads first, one after another on this GPU (their lines
    # go into "workloads"); they also bring the clocks to their loaded state
    others = {}
    if world == 1 and not args.no_workloads:
        for name in ("prefix_store_int4", "prefix_store_int8", "mistral_gqa", "streaming"):
            if name != w.name:
                others[name] = run_secondary(name, args.workload_steps, max(3, args.warmup // 4), dev,
                                             args.decode)
    calls = step_calls(w, kind, args.decode)
    grows = kind in ("decode", "stream")
    n_app = (args.warmup + args.steps) if grows else 1
    lens0 = W.make_lengths(w).numpy().astype(np.int64)
    Tmax = (int(lens0.max()) + n_app + w.G) // w.G * w.G + w.G
    K, V = W.make_kv(w, device=dev)
    ncp = cache_copies(w, lens0, Tmax) if grows else 1
    caches = [KiviCache(w.B, w.H, w.D, w.bits_k, w.bits_v, w.G, w.R, Tmax, device=dev) for _ in range(ncp)]
    cache = caches[0]
    seq_lens = None if w.ragged is None else torch.as_tensor(lens0.astype(np.int32), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ld = (Tmax + 3) // 4 * 4
    logits = torch.empty((w.B, w.Hq, ld), dtype=torch.float32, device=dev)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device=dev)
    wss = [c.workspace(w.Hq) for c in caches]
    ws = wss[0]
    kn, vn = W.make_step_tokens(w, n_app, device=dev)
    qs = torch.stack([W.make_q(w, dev, step=s) for s in range(n_app)]) if grows else W.make_q(w, dev)[None]
    if kind in ("full", "store"):
        kh = torch.empty((w.B, w.H, w.T, w.D), dtype=torch.float16, device=dev)
        vh = torch.empty_like(kh)
    else:  # encode the prefix once; the timed steps only append and decode
        for c in caches:
            abi.kivi_quant_keys(c, K, seq_lens)
            abi.kivi_quant_values(c, V, seq_lens)
        torch.cuda.synchronize(dev)
        del K, V
        torch.cuda.empty_cache()
    stream = torch.cuda.current_stream(dev)

    def step(i, ev=None):
        j = i if grows else 0
        c, wsc = caches[i % ncp], wss[i % ncp]
        fns = {
            "quant_keys": lambda: abi.kivi_quant_keys(c, K, seq_lens),
            "quant_values": lambda: abi.kivi_quant_values(c, V, seq_lens),
            "dequant_keys": lambda: abi.kivi_dequant(c, 0, kh),
            "dequant_values": lambda: abi.kivi_dequant(c, 1, vh),
            "append": lambda: abi.kivi_append_token(c, kn[j], vn[j], status),
            "decode_qk": lambda: abi.kivi_decode_qk(c, qs[j], logits),
            "decode_pv": lambda: abi.kivi_decode_pv(c, logits, out, wsc),
            "decode_attn": lambda: abi.kivi_decode_attention(c, qs[j], out, wsc),
        }
        for c_i, name in enumerate(calls):
            if ev is not None:
                ev[2 * c_i].record(stream)
            fns[name]()
            if ev is not None:
                ev[2 * c_i + 1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(calls))] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        queue_ahead(torch)
        t0.record(stream)
        for s in range(args.steps):
            step(args.warmup + s, evs[s])
        t1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    assert int(status.item()) == 0, "a sequence ran out of capacity"
    if "decode_attn" in calls:
        for wsc in wss:
            assert int(wsc[:1].view(torch.int32).item()) == 0, "decode status word"
    per_call = {c: sum(evs[s][2 * i].elapsed_time(evs[s][2 * i + 1]) for s in range(args.steps)) / args.steps
                for i, c in enumerate(calls)}
    ms_step = reduce_max(t0.elapsed_time(t1), dev) / args.steps

    # bytes per step, averaged over the timed steps (decode caches grow)
    if grows:
        timed = [lens0 + (args.warmup + s) // ncp + 1 for s in range(args.steps)]
        pick = timed[:: max(1, len(timed) // 16)]
        ab_list = [call_bytes(w, d, d) for d in pick]
        ab = {k: sum(a[k] for a in ab_list) / len(ab_list) for k in ab_list[0]}
        eq = sum(fp16_equiv_bytes(w, kind, d, d) for d in pick) / len(pick)
    else:
        dec = lens0 + 1
        ab = call_bytes(w, lens0, dec)
        eq = fp16_equiv_bytes(w, kind, lens0, dec)
    value = whole_job_value(eq, world, ms_step)
    hbm, src = peaks()
    kernels = {}
    for c in calls:
        gbs = ab[c] / (per_call[c] * 1e-3) / 1e9
        kernels[c] = {"ms": round(per_call[c], 5), "alg_bytes": int(ab[c]), "gbs": round(gbs, 1),
                      "frac": round(gbs / hbm, 3)}
    dominant = max(calls, key=lambda c: per_call[c])
    dk = kernels[dominant]
    breakdown = {"kernels": kernels}
    H, D = w.H, w.D
    if kind in ("full", "store"):
        enc = sum(2 * H * int(n) * D * 2 for n in lens0)
        qms = per_call["quant_keys"] + per_call["quant_values"]
        dms = per_call["dequant_keys"] + per_call["dequant_values"]
        breakdown["quant_gbs_fp16eq"] = round(enc / (qms * 1e-3) / 1e9, 1)
        breakdown["dequant_gbs_fp16eq"] = round(enc / (dms * 1e-3) / 1e9, 1)
    if kind != "store":
        dec_ms = sum(per_call[c] for c in calls if c.startswith("decode"))
        breakdown["decode_tok_s"] = round(w.B * world / (dec_ms * 1e-3), 1)
        breakdown["step_tok_s"] = round(w.B * world / (ms_step * 1e-3), 1)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"u{w.bits_k}/u{w.bits_v} codes, f32 stats, f16 KV, f32 accumulate",
        "data": "synthetic (seeded N(0,1) fp16, outlier key channels)",
        "config": {"workload": w.name, "step": kind, "shape": [w.B, w.H, w.T, w.D], "Hq": w.Hq,
                   "bits_k": w.bits_k, "bits_v": w.bits_v, "G": w.G, "R": w.R,
                   "ragged": list(w.ragged) if w.ragged else None,
                   "parallelism": f"replicas x{world}",
                   "l2": l2_note(kind, ncp, sum(w.H * (slice_bytes(w, int(n), 0) + slice_bytes(w, int(n), 1))
                                                for n in lens0))},
        "breakdown": breakdown,
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": dk["gbs"], "peak": hbm,
                     "peak_source": src, "unit": "GB/s", "frac": dk["frac"],
                     "traffic": recorded_traffic(dominant, w.name)},
        "gpu_launches": sum(LAUNCHES[c] for c in calls) * args.steps,
        "clocks": clk.summary(),
    }
    if others:
        line["workloads"] = others
    if kind == "full" and not args.no_e2e:
        line["e2e"] = run_e2e(args, w, cache, kh, vh, logits, out, ws, status, dev, world, eq, calls)
    if kind == "full" and not args.no_c2c:
        line["c2c"] = run_c2c(cache, dev)
    if rank == 0 and world == 1 and kind == "full" and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, K, V, qs[0], kn[0], vn[0])
    if world > 1:
        torch.distributed.destroy_process_group()
    return line if rank == 0 else None


def run_c2c(cache, dev, reps: int = 5) -> dict:
    """Compact-payload round trip through pinned host memory (kivi_export,
    kivi_import): payload bytes over the CUDA-event time of each call.  The
    kernels load and store host memory directly, so this is the CPU-GPU link's
    rate, reported apart from the HBM roofline."""
    import torch
    from kivi_bit_kv_gb300 import abi
    lens = cache.lens.cpu().tolist()
    n = abi.kivi_payload_bytes(cache.desc, lens)
    host = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    for name, fn in (("export", lambda: abi.kivi_export(cache, host, status)),
                     ("import", lambda: abi.kivi_import(cache, host, status))):
        fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = e0.elapsed_time(e1) / reps
    assert int(status.item()) == 0
    return {"payload_bytes": n, "export_ms": round(res["export"], 4), "import_ms": round(res["import"], 4),
            "export_gbs": round(n / (res["export"] * 1e-3) / 1e9, 1),
            "import_gbs": round(n / (res["import"] * 1e-3) / 1e9, 1),
            "memory": "pinned host (kernel loads / stores over the CPU-GPU link)"}


def run_e2e(args, w, cache, kh, vh, logits, out, ws, status, dev, world, eq, calls):
    """Same step through the public API from pinned host buffers: H2D of the
    step's K, V, q and new token, the step, D2H of the attention output.
    Double-buffered the way a serving loop would run it: a copy stream moves
    step i+1's inputs into the other pair of device buffers while step i
    computes, so every step's copy is inside the timed region and the compute
    hides behind it."""
    import torch
    from kivi_bit_kv_gb300 import abi
    from kivi_bit_kv_gb300 import workloads as W
    Kh, Vh = (t.pin_memory() for t in W.make_kv(w, device="cpu"))
    qh = W.make_q(w, "cpu").pin_memory()
    knh, vnh = (t[0].contiguous().pin_memory() for t in W.make_step_tokens(w, 1, "cpu"))
    hosts = (Kh, Vh, qh, knh, vnh)
    bufs = [tuple(torch.empty_like(h, device=dev) for h in hosts) for _ in range(2)]
    outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    stream = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]  # inputs of the buffer copied
    free = [torch.cuda.Event() for _ in range(2)]   # the buffer's last step done
    n = max(20, args.steps // 10)

    def issue_copy(i):
        b = i % 2
        copy.wait_event(free[b])
        with torch.cuda.stream(copy):
            for d, h in zip(bufs[b], hosts):
                d.copy_(h, non_blocking=True)
        ready[b].record(copy)

    def compute(i):
        b = i % 2
        stream.wait_event(ready[b])
        Kd, Vd, qd, knd, vnd = bufs[b]
        abi.kivi_quant_keys(cache, Kd)
        abi.kivi_quant_values(cache, Vd)
        abi.kivi_dequant(cache, 0, kh)
        abi.kivi_dequant(cache, 1, vh)
        abi.kivi_append_token(cache, knd, vnd, status)
        if "decode_attn" in calls:
            abi.kivi_decode_attention(cache, qd, out, ws)
        else:
            abi.kivi_decode_qk(cache, qd, logits)
            abi.kivi_decode_pv(cache, logits, out, ws)
        free[b].record(stream)
        outh.copy_(out, non_blocking=True)

    def run(steps, start=None):
        if start is not None:
            copy.wait_event(start)
        issue_copy(0)
        for i in range(steps):
            if i + 1 < steps:
                issue_copy(i + 1)
            compute(i)

    run(2)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    t0.record(stream)
    run(n, start=t0)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = reduce_max(t0.elapsed_time(t1), dev)
    bi = sum(t.numel() * t.element_size() for t in hosts)
    bo = outh.numel() * outh.element_size()
    return {"value": round(whole_job_value(eq, world, ms / n), 1), "unit": UNIT,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": n,
            "pipeline": "inputs of step i+1 copied on a second stream while step i computes"}


# ------------------------------------------------------ CPU oracle legs --

def _oracle_pass(R, w, Ks, Vs, qs, kn, vn, threads):
    """The whole step on the oracle for a sample of (b, h) slices, each
    treated as its own single-head sequence."""
    n, T, D = Ks.shape[0], Ks.shape[2], w.D
    Tmax = (T + 1 + w.G - 1) // w.G * w.G + w.G
    rc = R.RefCache(n, 1, D, w.bits_k, w.bits_v, w.G, w.R, Tmax)
    rc.encode(Ks, Vs, threads=threads)
    rc.decode(0, threads=threads)
    rc.decode(1, threads=threads)
    rc.append(kn, vn)
    rc.attention(qs, threads=threads)


def _sample(w, K, V, q, kn, vn, n, T):
    import numpy as np
    import torch
    idx = [(i * 7) % (w.B * w.H) for i in range(n)]
    bs = torch.tensor([i // w.H for i in idx])
    hs = torch.tensor([i % w.H for i in idx])
    Ks = K[bs, hs, :T].unsqueeze(1).cpu().numpy().view(np.uint16)
    Vs = V[bs, hs, :T].unsqueeze(1).cpu().numpy().view(np.uint16)
    qs = q[bs, hs * (w.Hq // w.H)].unsqueeze(1).cpu().numpy().view(np.uint16)
    ks = kn[bs, hs].unsqueeze(1).cpu().numpy().view(np.uint16)
    vs = vn[bs, hs].unsqueeze(1).cpu().numpy().view(np.uint16)
    return Ks, Vs, qs, ks, vs


def _slice_fp16eq(w, T):
    return 2 * T * w.D * 2 * 3 + 2 * w.D * 2


def _oracle_rate(R, w, K, V, q, kn, vn, threads: int, budget_s: float):
    """fp16-equivalent GB/s of the oracle on `threads` host threads, over
    rounds of `threads` (b, h) slices until budget_s has passed."""
    Ks, Vs, qs, ks, vs = _sample(w, K, V, q, kn, vn, threads, w.T)
    done, t_start = 0, time.perf_counter()
    while True:
        _oracle_pass(R, w, Ks, Vs, qs, ks, vs, threads)
        done += 1
        el = time.perf_counter() - t_start
        if el >= budget_s:
            break
    return done * threads * _slice_fp16eq(w, w.T) / el / 1e9, done, el


def cpu_baseline(w, K, V, q, kn, vn, budget_s: float = 10.0):
    """The oracle as it stands on a bounded sample (about 10 s of CPU work
    each): on every host core (the baseline of record) and on one thread."""
    from oracle import ref as R
    cores = R.host_threads()
    value, done, el = _oracle_rate(R, w, K, V, q, kn, vn, cores, budget_s)
    v1, done1, el1 = _oracle_rate(R, w, K, V, q, kn, vn, 1, budget_s)
    return {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done} rounds x {cores} (b,h) slices of {w.name} ({w.T} tokens each, full step "
                      f"per slice: encode, materialize K and V, append, decode), {el:.1f} s",
            "single_thread": {"value": round(v1, 4), "unit": UNIT, "cores": 1,
                              "sample": f"{done1} rounds x 1 slice, {el1:.1f} s"},
            "of_record": "all cores"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: every step is a bounded sample of the
    workload, sized so the whole run stays within a few minutes."""
    if rank != 0:
        return None
    import torch
    from kivi_bit_kv_gb300 import workloads as W
    from oracle import ref as R
    w = W.WORKLOADS[args.workload]
    cores = R.host_threads()
    K, V = W.make_kv(w, "cpu")
    q = W.make_q(w, "cpu")
    kn, vn = (t[0] for t in W.make_step_tokens(w, 1, "cpu"))
    # calibrate one full slice on one thread
    Ks, Vs, qs, ks, vs = _sample(w, K, V, q, kn, vn, 1, w.T)
    t = time.perf_counter()
    _oracle_pass(R, w, Ks, Vs, qs, ks, vs, 1)
    t1 = time.perf_counter() - t
    per_step = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    Tw = int(min(w.T, max(w.R + w.G, w.T * per_step / t1)))
    Tw = max(w.R + w.G, Tw // w.G * w.G)
    Ks, Vs, qs, ks, vs = _sample(w, K, V, q, kn, vn, cores, Tw)
    for _ in range(args.warmup):
        _oracle_pass(R, w, Ks, Vs, qs, ks, vs, cores)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_pass(R, w, Ks, Vs, qs, ks, vs, cores)
    el = time.perf_counter() - t
    ms_step = el / args.steps * 1e3
    value = cores * _slice_fp16eq(w, Tw) / (ms_step * 1e-3) / 1e9
    sample = f"per step {cores} (b,h) slices of {w.name} truncated to {Tw} tokens"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64 (CPU oracle)",
        "data": "synthetic (seeded N(0,1) fp16, outlier key channels)",
        "config": {"workload": w.name, "shape": [w.B, w.H, w.T, w.D], "Hq": w.Hq, "bits_k": w.bits_k,
                   "bits_v": w.bits_v, "G": w.G, "R": w.R, "parallelism": "host threads"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_kivi(args, rank, world, local)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
