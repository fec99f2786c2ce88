"""Parity and timing report for every configuration (run on a GPU; not collected by pytest).

For each workload it runs the library through its public API, compares every
output element with the fp64 oracle (full outputs, not samples), and times
both: the GPU with CUDA events (median of the timed repetitions, L2 flushed
before each), the oracle with wall time on all host cores.  Prints one
markdown table row per configuration.

    python tests/parity_report.py
"""
import json
import os
import statistics
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from attn_forward_tcgen05_gb300 import decode, prefill, prefill_window, sync_check  # noqa: E402
from attn_forward_tcgen05_gb300 import workloads as W  # noqa: E402

REPS = 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured"
    return 1900.0, 6800.0, "fallback"


def gpu_time_ms(fn):
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(REPS):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    sync_check()
    return statistics.median(ts)


def max_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    both = np.isneginf(got) & np.isneginf(ref)
    d = np.abs(np.where(both, 0.0, got) - np.where(both, 0.0, ref))
    return float(d.max()) if d.size else 0.0


def prefill_row(label, s, peak_tc):
    q, k, v = W.prefill_inputs_for(s)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    odt = torch.float32 if s.out_dtype == "f32" else torch.bfloat16
    o, lse = prefill(qd, kd, vd, causal=s.causal, scale=s.scale, out_dtype=odt)
    ms = gpu_time_ms(lambda: prefill(qd, kd, vd, causal=s.causal, scale=s.scale, out=(o, lse)))
    t0 = time.perf_counter()
    ro, rl = oracle.sdpa(q, k, v, s.causal, s.scale)
    cpu_s = time.perf_counter() - t0
    fl = W.prefill_flops(s.B, s.Hq, s.Sq, s.Skv, s.d, s.causal)
    tf = fl / (ms * 1e-3) / 1e12
    eo = max_err(o.float().cpu().numpy(), ro)
    el = max_err(lse.cpu().numpy(), rl)
    # the same kernel with the other output type: fp32 O shows the arithmetic error
    # alone (limit 5e-3); bf16 O adds the output's own rounding (limit 5e-3 + ulp/2)
    other = torch.bfloat16 if odt == torch.float32 else torch.float32
    o2, _ = prefill(qd, kd, vd, causal=s.causal, scale=s.scale, out_dtype=other)
    sync_check()
    e2 = max_err(o2.float().cpu().numpy(), ro)
    e32, e16 = (eo, e2) if odt == torch.float32 else (e2, eo)
    return (f"| {label} | {ms * 1e3:.1f} µs | {tf:.1f} TFLOP/s | {tf / peak_tc:.3f} of {peak_tc:.1f} TFLOP/s "
            f"| {e32:.2e} (fp32 O); {e16:.2e} (bf16 O) | {el:.2e} | {cpu_s:.2f} s ({oracle.num_cores()} cores) |")


def window_row(label, s, peak_tc):
    b = s.base
    q, k, v = W.prefill_inputs_for(b)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    # timed with bf16 O (the bench line's output type); errors for both output types
    o, lse = prefill_window(qd, kd, vd, s.window, s.n_sink, scale=b.scale, out_dtype=torch.bfloat16)
    ms = gpu_time_ms(lambda: prefill_window(qd, kd, vd, s.window, s.n_sink, scale=b.scale, out=(o, lse)))
    o32, _ = prefill_window(qd, kd, vd, s.window, s.n_sink, scale=b.scale, out_dtype=torch.float32)
    sync_check()
    t0 = time.perf_counter()
    ro, rl = oracle.sdpa_window(q, k, v, s.window, s.n_sink, b.scale)
    cpu_s = time.perf_counter() - t0
    tf = W.window_flops(s) / (ms * 1e-3) / 1e12
    e16 = max_err(o.float().cpu().numpy(), ro)
    eo = max_err(o32.cpu().numpy(), ro)
    el = max_err(lse.cpu().numpy(), rl)
    return (f"| {label} | {ms * 1e3:.1f} µs | {tf:.1f} TFLOP/s | {tf / peak_tc:.3f} of {peak_tc:.1f} TFLOP/s "
            f"| {eo:.2e} (fp32 O); {e16:.2e} (bf16 O) | {el:.2e} | {cpu_s:.2f} s ({oracle.num_cores()} cores) |")


def decode_row(label, s, peak_hbm):
    q, kc, vc, lens = W.decode_inputs_for(s)
    qd, kd, vd, ld = q.cuda(), kc.cuda(), vc.cuda(), lens.cuda()
    o, lse = decode(qd, kd, vd, ld, s.n_splits, s.min_rows_per_split, s.scale)
    ms = gpu_time_ms(lambda: decode(qd, kd, vd, ld, s.n_splits, s.min_rows_per_split, s.scale))
    t0 = time.perf_counter()
    ro, rl = oracle.decode(q, kc, vc, lens, s.scale)
    cpu_s = time.perf_counter() - t0
    nbytes = W.decode_kv_bytes(lens, s.Hkv, s.d)
    gbs = nbytes / (ms * 1e-3) / 1e9
    eo = max_err(o.float().cpu().numpy(), ro)
    el = max_err(lse.cpu().numpy(), rl)
    return (f"| {label} | {ms * 1e3:.1f} µs (split + merge) | {gbs:.0f} GB/s | {gbs / peak_hbm:.3f} of "
            f"{peak_hbm:.0f} GB/s | {eo:.2e} (bf16 O) | {el:.2e} | {cpu_s:.2f} s ({oracle.num_cores()} cores) |")


def main():
    peak_tc, peak_hbm, src = peaks()
    print(f"peaks: {peak_tc} TFLOP/s bf16, {peak_hbm} GB/s ({src})")
    print("| config | GPU time | throughput | % of roofline (peak used) | max\\|ΔO\\| | max\\|ΔLSE\\| | CPU oracle time (cores) |")
    print("|---|---|---|---|---|---|---|")
    print(prefill_row("C1 tiny MHA causal prefill, d = 64", W.TINY, peak_tc), flush=True)
    print(prefill_row("C2 GQA causal prefill, S = 3314, d = 128", W.GQA_PREFILL, peak_tc), flush=True)
    print(decode_row("C3 GQA decode, L = 1641, 8 splits + merge", W.GQA_DECODE, peak_hbm), flush=True)
    for d in (64, 128, 256):
        print(prefill_row(f"C4 non-causal MHA, S = 4096, d = {d}", W.mha_sweep(d), peak_tc), flush=True)
    print(decode_row("C5 ragged GQA decode, B = 64", W.RAGGED_DECODE, peak_hbm), flush=True)
    print(window_row("GQA prefill S = 3314, window 1024 + 4 sinks", W.WINDOW_PREFILL, peak_tc), flush=True)


if __name__ == "__main__":
    main()
