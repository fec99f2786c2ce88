#!/usr/bin/env python3
"""Benchmark of the attention-forward hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch of synthetic input:
  1. prefill FMHA on gqa_prefill_3314  (B=1, Hq=28, Hkv=4, S=3314, d=128, causal, O bf16)
  2. split-KV decode with its merge on gqa_decode_1641 (B=1, Hq=28, Hkv=4, KV 1641,
     8 splits), one launch: the last split of each query-head group merges
  3. the same on ragged_gqa_decode_b64 (B=64, Hq=32, Hkv=8, KV ~ U[512,8192])
Beside the step, each further workload is timed alone and reported on its own
line object: chunked (varlen) prefill, the sliding window with sinks, the
128-head multi-query decode, the non-causal head-dim sweep (B=2, H=16,
S=4096, d = 64, 128, 256, and 512), and, for context, the 1641-key decode of
the 28 layers of a model in one CUDA graph.
L2 is flushed (a 256 MiB device write, then a 256 MiB read so that no dirty lines
are left behind) before every step, outside the kernel
events.  `value` is the prefill throughput in TFLOP/s (algorithmic FLOPs:
4*d per admissible (query, key) pair); the decode throughput (algorithmic K+V
bytes, every cached row of every KV head read once) is reported beside it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With --gpus N > 1 the script expects torchrun (one process per GPU); every rank
runs an independent replica (the path has no exchange step) and rank 0 prints
one JSON line with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s (% BF16 TC peak); decode KV GB/s (% HBM peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu_index = gpu_index
        self.interval_ms = interval_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)  # let the sampler start before the timed region
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = []
        for rec in csv.reader(io.StringIO(getattr(self, "out", "") or "")):
            if len(rec) < 9:
                continue
            try:
                rows.append({"sm": float(rec[1]), "max": float(rec[2]), "power": float(rec[3]),
                             "hw": rec[5].strip(), "hw_thermal": rec[6].strip(),
                             "sw_thermal": rec[7].strip(), "sw_power": rec[8].strip()})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [r for r in rows if r["power"] > 0] or rows
        reasons = set()
        for r in busy:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["max"] for r in busy), "reasons": sorted(reasons),
                "samples": len(busy), "power_w_max": max(r["power"] for r in busy)}


# --------------------------------------------------------------------------- ours
class L2Flush:
    """Empties L2 of the timed kernels' data between timed launches: a write of a
    buffer larger than L2 (256 MiB), then a read of a second one, so that L2 holds
    clean lines of the second buffer rather than dirty lines of the first (which
    the next kernel's reads would otherwise have to write back to HBM first)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.s = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.s)


def max_over_ranks(values, world):
    """Element-wise maximum of per-rank timings over all ranks (the slowest replica
    sets the job's time); the identity with one process."""
    if world <= 1:
        return [float(x) for x in values]
    import torch
    import torch.distributed as dist
    tt = torch.tensor([float(x) for x in values], dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return [float(x) for x in tt]


def run_line(args):
    """One extra workload line alone (--line), for profiling its kernel."""
    import torch

    import attention_forward_tcgen05_gb300 as attn
    from attention_forward_tcgen05_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    attn.load()
    peaks, peak_src = load_peaks()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    if args.line.startswith("sweep"):
        return time_sweep(args, attn, W, dev, stream, flush, peaks, peak_src, int(args.line[5:]))
    fn = {"varlen": time_varlen, "window": time_window, "mqa": time_mqa_decode}[args.line]
    return fn(args, attn, W, dev, stream, flush, peaks, peak_src)


def run_ours(args, rank, world, local_rank):
    import torch

    import attention_forward_tcgen05_gb300 as attn
    from attention_forward_tcgen05_gb300 import workloads as W

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    attn.load()  # fails loudly if the CUDA library is missing
    peaks, peak_src = load_peaks()

    P = prefill_workload(args.prefill_workload)
    D3 = W.GQA_DECODE
    D5 = W.RAGGED_DECODE
    # inputs resident in HBM before the timed region
    q, k, v = [t.to(dev) for t in W.prefill_inputs_for(P)]
    o = torch.empty((P.B, P.Sq, P.Hq, P.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((P.B, P.Hq, P.Sq), dtype=torch.float32, device=dev)
    dec = {}
    for sh in (D3, D5):
        qd, kc, vc, lens = W.decode_inputs_for(sh)
        dec[sh.name] = dict(
            shape=sh, host=(qd, kc, vc, lens), dev=[t.to(dev) for t in (qd, kc, vc, lens)],
            part=(torch.empty((sh.B, sh.Hq, sh.n_splits, sh.d), dtype=torch.float32, device=dev),
                  torch.empty((sh.B, sh.Hq, sh.n_splits), dtype=torch.float32, device=dev)),
            out=(torch.empty((sh.B, sh.Hq, sh.d), dtype=torch.bfloat16, device=dev),
                 torch.empty((sh.B, sh.Hq), dtype=torch.float32, device=dev)),
            # completion counters of the combine fused into the split launch (zero between calls)
            counters=torch.zeros(sh.B * sh.Hq, dtype=torch.int32, device=dev),
            kv_bytes=W.decode_kv_bytes(lens, sh.Hkv, sh.d))
    flush = L2Flush(dev)
    flops = W.prefill_flops(P.B, P.Hq, P.Sq, P.Skv, P.d, P.causal)
    stream = torch.cuda.current_stream()

    do_prefill = args.only in (None, "prefill")
    do_decode = args.only in (None, "decode")

    def step(ev=None):
        flush()  # evict L2 (outside the kernel events)
        if ev is not None:
            ev[0].record(stream)
        if do_prefill:
            attn.prefill(q, k, v, causal=P.causal, scale=P.scale, out=(o, lse))
        if ev is not None:
            ev[1].record(stream)
        i = 2
        for name in ((D3.name, D5.name) if do_decode else ()):
            dd = dec[name]
            sh = dd["shape"]
            qd, kc, vc, lens = dd["dev"]
            # split partials and their combine in one launch (attn_decode)
            attn.decode(qd, kc, vc, lens, sh.n_splits, sh.min_rows_per_split, sh.scale,
                        torch.bfloat16, out=dd["out"], parts=dd["part"], counters=dd["counters"])
            if ev is not None:
                ev[i].record(stream)
            i += 1
        if not do_decode and ev is not None:
            for e in ev[2:]:
                e.record(stream)

    # warm-up
    for _ in range(args.warmup):
        step()
    attn.sync_check()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as sampler:
        barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for s in range(args.steps):
            step(evs[s])
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
    attn.sync_check()
    clocks = sampler.summary()

    # per-kernel device times (ms), averaged over the K timed steps
    def avg(a, b):
        return sum(evs[s][a].elapsed_time(evs[s][b]) for s in range(args.steps)) / args.steps

    t_prefill = avg(0, 1)
    t_dec3 = avg(1, 2)
    t_dec5 = avg(2, 3)
    ms_step = t_prefill + t_dec3 + t_dec5
    wall_ms = t_start.elapsed_time(t_end)

    ms_step, t_prefill_max, t_dec5_max, wall_ms = max_over_ranks(
        [ms_step, t_prefill, t_dec5, wall_ms], world)

    # ---- packed variable-length prefill (chunked prefill against a KV cache) ----
    varlen = None if args.only else time_varlen(args, attn, W, dev, stream, flush, peaks, peak_src)
    # ---- causal sliding window with attention sinks ----
    window = None if args.only else time_window(args, attn, W, dev, stream, flush, peaks, peak_src)
    # ---- multi-query decode on the tensor cores (heads packed into the tile rows) ----
    mqa = None if args.only else time_mqa_decode(args, attn, W, dev, stream, flush, peaks, peak_src)
    # ---- the 1641-key decode of all 28 layers of a model, in one CUDA graph ----
    layers28 = None if args.only else time_decode_layers_graph(args, attn, W, dev, stream, flush, peaks, peak_src)
    # ---- non-causal head-dim sweep (B = 2, H = 16, S = 4096; d = 64, 128, 256) ----
    sweep = None if args.only else [time_sweep(args, attn, W, dev, stream, flush, peaks, peak_src, d)
                                    for d in (64, 128, 256, 512)]

    # ---- end to end through the public API with host buffers ----
    e2e = None if (args.no_e2e or args.only) else run_e2e(args, attn, W, dev, stream, P, dec, flops)

    if rank != 0:
        return None
    prefill_tflops = world * flops / (max(t_prefill_max, 1e-9) * 1e-3) / 1e12
    kv5 = dec[D5.name]["kv_bytes"]
    kv3 = dec[D3.name]["kv_bytes"]
    dec_gbs = world * kv5 / (max(t_dec5_max, 1e-9) * 1e-3) / 1e9
    split_gbs = kv5 / (max(t_dec5, 1e-9) * 1e-3) / 1e9
    peak_tc = float(peaks["bf16_tflops"])
    peak_hbm = float(peaks["hbm_gbs"])
    traffic = load_traffic()
    # one roofline per hot kernel; the top-level one is the kernel that takes the
    # largest share of the step's device time
    pkern = prefill_kernel_name(P.d, P.causal, P.Sq)
    prefill_mufu = mufu_roofline(flops / (4 * P.d), t_prefill)
    prefill_roof = {"bound": "tensor", "kernel": pkern, "workload": P.name,
                    "achieved": round(prefill_tflops / world, 2), "peak": peak_tc,
                    "unit": "TFLOP/s", "frac": round(prefill_tflops / world / peak_tc, 4),
                    "traffic": traffic.get(f"{pkern} {P.name}"),
                    "step_share": round(t_prefill / ms_step, 4),
                    "peak_source": f"bf16_tflops (burst) of {peak_src}"}
    decode_roof = {"bound": "hbm", "kernel": "decode_split_kernel<128,4>", "workload": D5.name,
                   "achieved": round(split_gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                   "frac": round(split_gbs / peak_hbm, 4),
                   # keyed by split policy too: a capture holds for the grid it was taken on
                   "traffic": traffic.get(f"decode_split_kernel<128,4> fused {D5.name} "
                                          f"{D5.n_splits}x{D5.min_rows_per_split}"),
                   "step_share": round(t_dec5 / ms_step, 4),
                   "peak_source": f"hbm_gbs of {peak_src}"}
    if not do_decode:
        dominant_roof = prefill_roof
    elif not do_prefill:
        dominant_roof = decode_roof
    else:
        dominant_roof = prefill_roof if t_prefill >= t_dec5 else decode_roof
    line = {
        "metric": METRIC,
        "value": round(prefill_tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{P.name} + {D3.name} + {D5.name}",
                   "prefill": {"B": P.B, "Hq": P.Hq, "Hkv": P.Hkv, "Sq": P.Sq, "Skv": P.Skv,
                               "d": P.d, "causal": P.causal, "o_dtype": "bf16"},
                   "decode_1641": {"B": D3.B, "Hq": D3.Hq, "Hkv": D3.Hkv, "kv_len": D3.fixed_len,
                                   "d": D3.d, "n_splits": D3.n_splits},
                   "decode_ragged": {"B": D5.B, "Hq": D5.Hq, "Hkv": D5.Hkv, "d": D5.d,
                                     "kv_len_range": list(D5.len_range), "n_splits": D5.n_splits,
                                     "min_rows_per_split": D5.min_rows_per_split},
                   "l2": "flushed before every step (256 MiB device write, then a 256 MiB read)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": dominant_roof,
        "rooflines": {"prefill": prefill_roof, "decode_split": decode_roof, "prefill_mufu": prefill_mufu},
        "decode": {"value": round(dec_gbs, 1), "unit": "GB/s", "workload": D5.name,
                   "kv_bytes": kv5, "decode_us": round(t_dec5 * 1e3, 2),
                   "launches": "one: split partials and their combine (attn_decode)",
                   "roofline": decode_roof,
                   "gqa_decode_1641": {"decode_us": round(t_dec3 * 1e3, 2),
                                       "kv_bytes": kv3,
                                       "traffic": traffic.get(f"decode_split_kernel<128,4> fused {D3.name} "
                                                              f"{D3.n_splits}x{D3.min_rows_per_split}"),
                                       "GB_per_s": round(kv3 / (max(t_dec3, 1e-9) * 1e-3) / 1e9, 1)}},
        "prefill_us": round(t_prefill * 1e3, 2),
        "wall_ms_timed_region": round(wall_ms, 3),
        "gpu_launches": (int(do_prefill) + 2 * int(do_decode)) * args.steps,
        "e2e": e2e,
        "prefill_varlen": varlen,
        "prefill_window": window,
        "decode_packed": mqa,
        "decode_1641_layers_graph": layers28,
        "prefill_headdim_sweep": sweep,
        "clocks": clocks,
    }
    return line


def time_varlen(args, attn, W, dev, stream, flush, peaks, peak_src):
    """Chunked prefill (packed sequences against a KV cache): average launch time
    of attn_prefill_varlen over the timed iterations, L2 flushed before each."""
    import torch

    V = W.CHUNKED_PREFILL
    q, kc, vc, cu, kv = W.varlen_inputs_for(V)
    flops = W.varlen_flops(cu, kv, V.Hq, V.d, V.causal)
    max_sq = int((cu[1:] - cu[:-1]).max())
    qd, kcd, vcd, cud, kvd = (t.to(dev) for t in (q, kc, vc, cu, kv))
    o = torch.empty((q.shape[0], V.Hq, V.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((V.Hq, q.shape[0]), dtype=torch.float32, device=dev)

    def call():
        attn.prefill_varlen(qd, kcd, vcd, cud, kvd, max_sq, causal=V.causal, scale=V.scale, out=(o, lse))

    for _ in range(args.warmup):
        call()
    n = max(1, min(args.steps, 50))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        flush()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    attn.sync_check()
    ms = sum(a.elapsed_time(b) for a, b in evs) / n
    tf = flops / (ms * 1e-3) / 1e12
    peak_tc = float(peaks["bf16_tflops"])
    return {"workload": V.name, "B": V.B, "Hq": V.Hq, "Hkv": V.Hkv, "d": V.d, "causal": V.causal,
            "total_q": int(q.shape[0]), "kv_tokens": int(kv.sum()), "gflop": round(flops / 1e9, 3),
            "us": round(ms * 1e3, 2), "value": round(tf, 2), "unit": "TFLOP/s", "steps": n,
            "roofline": {"bound": "tensor", "kernel": "fmha_fwd_kernel<128>", "achieved": round(tf, 2),
                         "peak": peak_tc, "unit": "TFLOP/s", "frac": round(tf / peak_tc, 4),
                         "traffic": load_traffic().get(f"fmha_fwd_kernel<128> varlen {V.name}"),
                         "peak_source": f"bf16_tflops (burst) of {peak_src}"}}


def time_window(args, attn, W, dev, stream, flush, peaks, peak_src):
    """Causal sliding-window prefill with attention sinks: average launch time of
    attn_prefill_window over the timed iterations, L2 flushed before each.  The
    FLOPs count only admissible (query, key) pairs."""
    import torch

    S = W.WINDOW_PREFILL
    P = S.base
    q, k, v = (t.to(dev) for t in W.prefill_inputs_for(P))
    flops = W.window_flops(S)
    o = torch.empty((P.B, P.Sq, P.Hq, P.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((P.B, P.Hq, P.Sq), dtype=torch.float32, device=dev)

    def call():
        attn.prefill_window(q, k, v, S.window, S.n_sink, scale=P.scale, out=(o, lse))

    for _ in range(args.warmup):
        call()
    n = max(1, min(args.steps, 50))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        flush()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    attn.sync_check()
    ms = sum(a.elapsed_time(b) for a, b in evs) / n
    tf = flops / (ms * 1e-3) / 1e12
    peak_tc = float(peaks["bf16_tflops"])
    kern = prefill_kernel_name(P.d, False, P.Sq)
    return {"workload": S.name, "B": P.B, "Hq": P.Hq, "Hkv": P.Hkv, "S": P.Sq, "d": P.d,
            "window": S.window, "n_sink": S.n_sink, "gflop": round(flops / 1e9, 3),
            "us": round(ms * 1e3, 2), "value": round(tf, 2), "unit": "TFLOP/s", "steps": n,
            "roofline": {"bound": "tensor", "kernel": kern, "achieved": round(tf, 2),
                         "peak": peak_tc, "unit": "TFLOP/s", "frac": round(tf / peak_tc, 4),
                         "traffic": load_traffic().get(f"{kern} window {S.name}"),
                         "peak_source": f"bf16_tflops (burst) of {peak_src}"}}


def time_sweep(args, attn, W, dev, stream, flush, peaks, peak_src, d):
    """Non-causal MHA prefill of the head-dim sweep (B = 2, H = 16, S = 4096, bf16 O)
    at head dim d: average launch time of attn_prefill_fwd over the timed
    iterations, L2 flushed before each."""
    import torch

    P = W.mha_sweep(d)
    q, k, v = (t.to(dev) for t in W.prefill_inputs_for(P))
    flops = W.prefill_flops(P.B, P.Hq, P.Sq, P.Skv, P.d, P.causal)
    o = torch.empty((P.B, P.Sq, P.Hq, P.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((P.B, P.Hq, P.Sq), dtype=torch.float32, device=dev)

    def call():
        attn.prefill(q, k, v, causal=P.causal, scale=P.scale, out=(o, lse))

    for _ in range(args.warmup):
        call()
    n = max(1, min(args.steps, 50))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        flush()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    attn.sync_check()
    ms = sum(a.elapsed_time(b) for a, b in evs) / n
    tf = flops / (ms * 1e-3) / 1e12
    peak_tc = float(peaks["bf16_tflops"])
    kern = prefill_kernel_name(P.d, P.causal, P.Sq)
    line = {"workload": P.name, "B": P.B, "Hq": P.Hq, "Hkv": P.Hkv, "S": P.Sq, "d": P.d,
            "causal": P.causal, "gflop": round(flops / 1e9, 3), "us": round(ms * 1e3, 2),
            "value": round(tf, 2), "unit": "TFLOP/s", "steps": n,
            "roofline": {"bound": "tensor", "kernel": kern, "achieved": round(tf, 2), "peak": peak_tc,
                         "unit": "TFLOP/s", "frac": round(tf / peak_tc, 4),
                         "traffic": load_traffic().get(f"{kern} {P.name}"),
                         "peak_source": f"bf16_tflops (burst) of {peak_src}"}}
    if P.d == 512:
        # O is computed in two column halves and S = QK^T once per half: the tensor
        # cores execute 6*d FLOPs per pair, 1.5x the algorithmic 4*d counted above
        line["executed_gflop"] = round(1.5 * flops / 1e9, 3)
        line["executed_tflops"] = round(1.5 * tf, 2)
    line["roofline_mufu"] = mufu_roofline(flops / (4 * P.d), ms)
    return line


# MUFU ex2 rate: 32 lanes per clock per SM (a probe on this GPU; 8 per sub-partition)
MUFU_EX2_PER_CLK_SM = 32


def mufu_roofline(exps: float, ms: float) -> dict:
    """The secondary bound of the prefill: one exp2 per admissible (query, key) pair on
    the MUFU, against the GPU's rate at its maximum SM clock."""
    import torch
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    clk_ghz = 2.07  # maximum SM clock of the GB300s this runs on (nvidia-smi clocks.max.sm)
    peak = MUFU_EX2_PER_CLK_SM * props.multi_processor_count * clk_ghz  # G exp2 / s
    achieved = exps / (ms * 1e-3) / 1e9
    return {"bound": "alu", "unit": "Gexp2/s", "achieved": round(achieved, 1), "peak": round(peak, 1),
            "frac": round(achieved / peak, 4),
            "peak_source": f"{MUFU_EX2_PER_CLK_SM} ex2 per clock per SM x {props.multi_processor_count} SMs "
                           f"x {clk_ghz} GHz"}


def prefill_kernel_name(d: int, causal: bool = False, Sq: int = 4096) -> str:
    """The kernel that runs a fixed-length prefill of head dim d (causal launches of
    head dims 64 and 128 run on the persistent kernel; head dim 512 runs on CTA pairs
    once the queries span more than one 128-row tile)."""
    if d == 512:
        return "fmha_d512_pair_kernel"
    if d == 256:
        return f"fmha_pair_kernel<{d}>"
    return f"fmha_persistent_kernel<{d}>" if causal else f"fmha_fwd_kernel<{d}>"


def time_mqa_decode(args, attn, W, dev, stream, flush, peaks, peak_src):
    """One-token decode with 128 query heads per KV head through attn_decode_packed:
    average launch time over the timed iterations, L2 flushed before each.  Both
    rooflines are reported: FLOPs on the tensor cores and K/V bytes from HBM."""
    import torch

    S = W.MQA_DECODE
    q, kc, vc, lens = W.decode_inputs_for(S)
    flops = W.decode_flops(lens, S.Hq, S.d)
    kvb = W.decode_kv_bytes(lens, S.Hkv, S.d)
    qd, kd, vd, ld = (t.to(dev) for t in (q, kc, vc, lens))
    o = torch.empty((S.B, S.Hq, S.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((S.B, S.Hq), dtype=torch.float32, device=dev)

    def call():
        attn.decode_packed(qd, kd, vd, ld, S.scale, out=(o, lse))

    for _ in range(args.warmup):
        call()
    n = max(1, min(args.steps, 50))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        flush()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    attn.sync_check()
    ms = sum(a.elapsed_time(b) for a, b in evs) / n
    tf = flops / (ms * 1e-3) / 1e12
    gbs = kvb / (ms * 1e-3) / 1e9
    peak_tc, peak_hbm = float(peaks["bf16_tflops"]), float(peaks["hbm_gbs"])
    kern = f"fmha_fwd_kernel<{S.d}>"
    traffic = load_traffic().get(f"{kern} packed {S.name}")  # DRAM bytes of the launch, both rooflines
    return {"workload": S.name, "B": S.B, "Hq": S.Hq, "Hkv": S.Hkv, "d": S.d,
            "kv_tokens": int(lens.sum()), "gflop": round(flops / 1e9, 3), "kv_mb": round(kvb / 1e6, 1),
            "us": round(ms * 1e3, 2), "value": round(tf, 2), "unit": "TFLOP/s", "gbs": round(gbs, 1),
            "steps": n,
            "roofline": {"bound": "tensor", "kernel": kern, "achieved": round(tf, 2),
                         "peak": peak_tc, "unit": "TFLOP/s", "frac": round(tf / peak_tc, 4), "traffic": traffic,
                         "peak_source": f"bf16_tflops (burst) of {peak_src}"},
            "roofline_hbm": {"bound": "hbm", "kernel": kern, "achieved": round(gbs, 1), "peak": peak_hbm,
                             "unit": "GB/s", "frac": round(gbs / peak_hbm, 4), "traffic": traffic,
                             "peak_source": f"hbm_gbs of {peak_src}"}}


def time_decode_layers_graph(args, attn, W, dev, stream, flush, peaks, peak_src, layers=28):
    """Context for the latency-bound 1641-key GQA decode: one decode per layer of a
    28-layer model (each layer its own KV cache, the same shape), the 28 calls (split
    and merge in one launch each) captured in one CUDA graph and replayed, L2 flushed
    before each replay.  Reports the time per layer, with the graph and with plain
    launches, and the K/V bandwidth over the whole replay."""
    import torch

    S = W.GQA_DECODE
    lens = torch.full((S.B,), S.fixed_len, dtype=torch.int32)
    caches = []
    for layer in range(layers):
        q, kc, vc = W.decode_inputs(S.B, S.Hq, S.Hkv, S.d, lens, S.seed + 100 + layer)
        caches.append([t.to(dev) for t in (q, kc, vc, lens)])
    kvb = W.decode_kv_bytes(lens, S.Hkv, S.d) * layers
    o = torch.empty((layers, S.B, S.Hq, S.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((layers, S.B, S.Hq), dtype=torch.float32, device=dev)
    # the layers run one after another on one stream: they can share the partials
    # and the completion counters
    po = torch.empty((S.B, S.Hq, S.n_splits, S.d), dtype=torch.float32, device=dev)
    pl = torch.empty((S.B, S.Hq, S.n_splits), dtype=torch.float32, device=dev)
    ctr = torch.zeros(S.B * S.Hq, dtype=torch.int32, device=dev)

    def run():
        for layer, (q, kc, vc, ln) in enumerate(caches):
            attn.decode(q, kc, vc, ln, S.n_splits, S.min_rows_per_split, S.scale, torch.bfloat16,
                        out=(o[layer], lse[layer]), parts=(po, pl), counters=ctr)

    run()
    torch.cuda.synchronize()
    attn.sync_check()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    n = max(1, min(args.steps, 50))

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in evs:
            flush()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        attn.sync_check()
        return sum(a.elapsed_time(b) for a, b in evs) / n

    ms_graph = timed(graph.replay)
    ms_plain = timed(run)
    return {"workload": f"{S.name} x {layers} layers", "layers": layers, "B": S.B, "Hq": S.Hq, "Hkv": S.Hkv,
            "d": S.d, "kv_len": S.fixed_len, "n_splits": S.n_splits,
            "us_per_layer_graph": round(ms_graph * 1e3 / layers, 2),
            "us_per_layer_launches": round(ms_plain * 1e3 / layers, 2),
            "gbs_graph": round(kvb / (ms_graph * 1e-3) / 1e9, 1),
            "gpu_launches_per_replay": layers, "steps": n,
            "note": "context line: the 28 layers' decodes run in sequence, as in a model's decode step; "
                    "L2 flushed before each replay, not between the layers"}


def _pipelined_ms(n, h2d, compute, d2h, dev):
    """Milliseconds per step of n steps run as a three-stage pipeline on three
    streams: a step's host-to-device copies, its kernels, its device-to-host copies.
    h2d(b) and d2h(b) name the (dst, src) tensor pairs of device buffer b;
    compute(b, stream) launches the kernels.  The copies of steps s + 1 and s - 1
    overlap the kernels of step s.  Device inputs and outputs are double-buffered
    (buffer s % 2): a step's input copies wait until the kernels of step s - 2 are
    done with its buffer, and its kernels wait until step s - 2's outputs have left
    their buffer.  Timed from before the first copy to after the last one, on the
    device.  (Cutting each direction's copies over 2, 4 or 8 streams measured
    slower: one stream per direction already moves what the host link carries.)"""
    import torch

    s_in, s_c, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev_in, ev_c, ev_out = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(s_in)
    for i in range(n):
        b = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_c[i - 2])
            for d_, h in h2d(b):
                d_.copy_(h, non_blocking=True)
            ev_in[i].record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(ev_in[i])
            if i >= 2:
                s_c.wait_event(ev_out[i - 2])
            compute(b, s_c)
            ev_c[i].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[i])
            for h, d_ in d2h(b):
                h.copy_(d_, non_blocking=True)
            ev_out[i].record(s_out)
    end.record(s_out)  # after the last step's output copy, which follows all other work
    torch.cuda.synchronize()
    return start.elapsed_time(end) / n


def _staged(specs, dev):
    """One flat byte buffer (pinned host memory when dev is None) and a contiguous
    view of it for each (shape, dtype) in specs, every view 256-byte aligned."""
    import torch

    offs, n = [], 0
    for shape, dtype in specs:
        offs.append(n)
        nbytes = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        n += (nbytes + 255) // 256 * 256
    buf = torch.empty(n, dtype=torch.uint8, device=dev) if dev is not None else \
        torch.empty(n, dtype=torch.uint8).pin_memory()
    views = []
    for (shape, dtype), o in zip(specs, offs):
        nbytes = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        views.append(buf[o:o + nbytes].view(dtype).view(shape))
    return buf, views


def run_e2e(args, attn, W, dev, stream, P, dec, flops):
    """The step's work through the public API from pinned host buffers: every step
    copies its inputs host-to-device, runs the kernels and copies O and LSE back,
    all inside the timed region.  The steps run as a pipeline on three streams
    (copies of neighbouring steps overlap a step's kernels, device buffers doubled),
    the way a serving loop would; `value` is the prefill's rate so measured.  The
    same work done one step at a time on one stream is reported as the latency."""
    import torch

    # a step's inputs sit in one pinned staging buffer and its outputs in one device
    # buffer, so that each direction is one copy per step (three input copies and
    # two output copies measured slower: each copy has a cost of its own)
    q0, k0, v0 = W.prefill_inputs_for(P)
    o_shape, l_shape = (P.B, P.Sq, P.Hq, P.d), (P.B, P.Hq, P.Sq)
    hin, (qh, kh, vh) = _staged([(q0.shape, q0.dtype), (k0.shape, k0.dtype), (v0.shape, v0.dtype)], None)
    for h, t in zip((qh, kh, vh), (q0, k0, v0)):
        h.copy_(t)
    hout, (oh, lh) = _staged([(o_shape, torch.bfloat16), (l_shape, torch.float32)], None)
    din, dq = zip(*(_staged([(q0.shape, q0.dtype), (k0.shape, k0.dtype), (v0.shape, v0.dtype)], dev)
                    for _ in range(2)))
    dout, dol = zip(*(_staged([(o_shape, torch.bfloat16), (l_shape, torch.float32)], dev) for _ in range(2)))
    h2d = hin.numel()
    d2h = hout.numel()

    def pre_in(b):  # (device, host) pairs of buffer b's inputs: one copy
        return [(din[b], hin)]

    def pre_run(b, st):
        q_, k_, v_ = dq[b]
        attn.prefill(q_, k_, v_, causal=P.causal, scale=P.scale, out=dol[b], stream=st)

    def pre_out(b):  # (host, device) pairs of buffer b's outputs: one copy
        return [(hout, dout[b])]

    # the ragged decode (the step's second workload) the same way
    name = list(dec)[1]
    dd = dec[name]
    sh = dd["shape"]
    dh = [t.pin_memory() for t in dd["host"]]
    ddev = [[torch.empty_like(t, device=dev) for t in dh] for _ in range(2)]
    dod = [torch.empty((sh.B, sh.Hq, sh.d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    dld = [torch.empty((sh.B, sh.Hq), dtype=torch.float32, device=dev) for _ in range(2)]
    doh = torch.empty((sh.B, sh.Hq, sh.d), dtype=torch.bfloat16).pin_memory()
    dlh = torch.empty((sh.B, sh.Hq), dtype=torch.float32).pin_memory()
    parts = (torch.empty((sh.B, sh.Hq, sh.n_splits, sh.d), dtype=torch.float32, device=dev),
             torch.empty((sh.B, sh.Hq, sh.n_splits), dtype=torch.float32, device=dev))
    counters = torch.zeros(sh.B * sh.Hq, dtype=torch.int32, device=dev)
    dec_h2d = sum(t.numel() * t.element_size() for t in dh)
    dec_d2h = doh.numel() * 2 + dlh.numel() * 4

    def dec_in(b):
        return list(zip(ddev[b], dh))

    def dec_run(b, st):
        x = ddev[b]
        attn.decode(x[0], x[1], x[2], x[3], sh.n_splits, sh.min_rows_per_split, sh.scale, stream=st,
                    out=(dod[b], dld[b]), parts=parts, counters=counters)

    def dec_out(b):
        return [(doh, dod[b]), (dlh, dld[b])]

    # latency: one step at a time on one stream
    def serial(h2d_fn, run_fn, d2h_fn, n):
        def one():
            for d_, h in h2d_fn(0):
                d_.copy_(h, non_blocking=True)
            run_fn(0, stream)
            for h, d_ in d2h_fn(0):
                h.copy_(d_, non_blocking=True)

        for _ in range(max(1, min(args.warmup, 3))):
            one()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b_ in evs:
            a.record(stream)
            one()
            b_.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b_) for a, b_ in evs) / n

    n = max(1, min(args.steps, 20))
    with torch.cuda.stream(stream):
        lat_pre = serial(pre_in, pre_run, pre_out, n)
        lat_dec = serial(dec_in, dec_run, dec_out, max(1, min(n, 5)))
    _pipelined_ms(max(2, min(args.warmup, 3)), pre_in, pre_run, pre_out, dev)  # warm-up
    t_pre = _pipelined_ms(n, pre_in, pre_run, pre_out, dev)
    nd = max(2, min(n, 5))
    t_dec = _pipelined_ms(nd, dec_in, dec_run, dec_out, dev)
    attn.sync_check()
    # the pipelined steps computed what the kernels compute: compare the last copy-out
    o_ref, l_ref = attn.prefill(*dq[0], causal=P.causal, scale=P.scale)
    torch.cuda.synchronize()
    assert torch.equal(oh, o_ref.cpu()) and torch.equal(lh, l_ref.cpu()), "pipelined e2e output differs"
    kv = dd["kv_bytes"]
    return {"value": round(flops / (t_pre * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": n, "prefill_ms": round(t_pre, 4),
            "prefill_latency_ms": round(lat_pre, 4),
            "decode_ragged": {"GB_per_s": round(kv / (t_dec * 1e-3) / 1e9, 1), "ms": round(t_dec, 4),
                              "latency_ms": round(lat_dec, 4), "steps": nd,
                              "h2d_bytes_per_step": int(dec_h2d), "d2h_bytes_per_step": int(dec_d2h)},
            "note": "pinned host buffers; every step copies its inputs in and O and LSE out inside the "
                    "timed region; steps pipelined on three streams (copies in / kernels / copies out, "
                    "device buffers doubled); latency = one step at a time on one stream"}


def prefill_workload(name: str):
    """The prefill workload of the step: gqa_prefill_3314 by default; the head-dim
    sweep shapes are selectable for profiling their kernels."""
    from attention_forward_tcgen05_gb300 import workloads as W
    shapes = {W.GQA_PREFILL.name: W.GQA_PREFILL}
    for d in (64, 128, 256, 512):
        shapes[W.mha_sweep(d).name] = W.mha_sweep(d)
    if name not in shapes:
        raise SystemExit(f"unknown prefill workload {name!r}; one of {sorted(shapes)}")
    return shapes[name]


def load_traffic():
    """DRAM bytes per launch from the committed ncu summary, if present."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)
    return {}


# --------------------------------------------------------------------------- CPU baseline
def _oracle_sampler():
    """The fp64 oracle as it stands, timed on the host cores over bounded samples of
    the prefill workload (every key of a strided subset of query rows of all heads).
    Inputs are prepared and the oracle's row rate calibrated once; the returned
    function times one sample sized to a time budget and returns
    (GFLOP/s, threads, seconds, rows, stride)."""
    import numpy as np
    import torch

    import oracle
    from attention_forward_tcgen05_gb300 import workloads as W

    P = W.GQA_PREFILL
    q, k, v = W.prefill_inputs_for(P)
    qn, kn, vn = (t.to(torch.float64).numpy() for t in (q, k, v))
    cores = oracle.num_cores()
    stride = 64
    rows = [(0, h, i) for h in range(P.Hq) for i in range(stride // 2, P.Sq, stride)]
    t0 = time.perf_counter()
    oracle.sdpa_rows(qn, kn, vn, P.causal, P.scale, rows, nthreads=cores)
    rate = len(rows) / max(time.perf_counter() - t0, 1e-3)  # rows per second

    def run(budget_s: float, seed: int):
        target = max(1, int(rate * budget_s))
        stride2 = max(1, int(P.Sq * P.Hq / target))
        rng = np.random.default_rng(seed)
        sample = [(0, h, i) for h in range(P.Hq) for i in range(int(rng.integers(stride2)), P.Sq, stride2)]
        t1 = time.perf_counter()
        oracle.sdpa_rows(qn, kn, vn, P.causal, P.scale, sample, nthreads=cores)
        dt = time.perf_counter() - t1
        fl = sum(4 * P.d * (i + 1) for _, _, i in sample)
        return fl / dt / 1e9, cores, dt, len(sample), stride2

    return run


def cpu_baseline(budget_s: float = 12.0, seed: int = 0):
    """One bounded sample of the oracle on the prefill workload (see _oracle_sampler)."""
    return _oracle_sampler()(budget_s, seed)


# wall-clock budget of the reference arm's timed samples, spread over its steps
REFERENCE_BUDGET_S = 150.0


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle as it stands, on the same workload;
    each step is one bounded sample, sized so that the whole run stays within a
    few minutes whatever --steps and --warmup are."""
    if rank != 0:
        return None
    from attention_forward_tcgen05_gb300 import workloads as W
    P = W.GQA_PREFILL
    sampler = _oracle_sampler()
    step_budget = max(0.05, REFERENCE_BUDGET_S / (args.steps + 0.25 * args.warmup))
    per_step = []
    info = None
    for s in range(args.warmup + args.steps):
        budget = 0.25 * step_budget if s < args.warmup else step_budget
        g, cores, dt, n_rows, stride = sampler(budget, s)
        if s >= args.warmup:
            per_step.append(g)
            info = (cores, n_rows, stride)
    val = statistics.median(per_step) / 1e3  # TFLOP/s
    cores, n_rows, stride = info
    sample = (f"per step {n_rows} query rows (every {stride}th row of each of the {P.Hq} heads, "
              f"random offset) of {P.name}; 4*d FLOPs per admissible (query, key) pair")
    return {"metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": P.name, "B": P.B, "Hq": P.Hq, "Hkv": P.Hkv, "Sq": P.Sq,
                       "d": P.d, "causal": P.causal},
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=("prefill", "decode"), default=None,
                    help="time only one part of the step (profiling runs)")
    ap.add_argument("--line", choices=("varlen", "window", "mqa", "sweep64", "sweep128", "sweep256", "sweep512"),
                    default=None,
                    help="time only one of the extra workload lines and print it (profiling runs)")
    ap.add_argument("--prefill-workload", default="gqa_prefill_3314",
                    help="prefill workload of the step (the head-dim sweep shapes are for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        if args.gpus > 1:
            sys.exit(f"--gpus {args.gpus} needs torchrun with {args.gpus} processes")
    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        line = run_reference(args, rank, world)
        print(json.dumps(line))
        return
    if args.line:
        if rank == 0:
            print(json.dumps(run_line(args)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0 and line is not None:
        if not args.no_cpu_baseline and not args.only:
            g, cores, dt, n_rows, stride = cpu_baseline()
            line["cpu_baseline"] = {
                "value": round(g / 1e3, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                "seconds": round(dt, 2),
                "sample": f"{n_rows} query rows (every {stride}th row of each head) of "
                          f"{W_name()}; fp64, all host threads"}
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def W_name():
    from attention_forward_tcgen05_gb300 import workloads as W
    return W.GQA_PREFILL.name


if __name__ == "__main__":
    main()
