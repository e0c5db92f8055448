"""Benchmark of the fused-attention hot path on GB300.

A step is one pass of the whole path over one batch of synthetic inputs:
  1. attn_fwd   -- MHA prefill B4 H32 S2048 D128 bf16, causal (137.5 GFLOP);
  2. attn_decode -- flash-decoding B64 Hq32 Hkv8 D128 bf16 over a cache
     [64, 8, 32768, 128] with seq_lens uniform in [512, 32768], 64 splits
     (chunk 512; about 4.36 GB of K/V prefixes read).
The metric is the step's share of the GPU roofline: the time the step would
take at the measured peaks (prefill flops at the dense bf16 tensor peak, plus
decode bytes at the HBM copy bandwidth) divided by the measured time, in
percent, summed over GPUs for N > 1.  Per-leg TFLOP/s and GB/s are reported
beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

Timing: CUDA events on the launching stream around exactly K steps, with a
barrier and a device synchronize on both sides; inputs are larger than L2
(the decode leg streams ~4.4 GB between prefill calls, so no step starts with
a warm L2).  Inputs are resident in HBM when the timed region starts; the
e2e figure repeats the step from pinned host buffers with the copies inside
its timed region: the prefill's Q, K, V, the decode queries, the valid prefix
(seq_lens rows) of every (sequence, KV head) of the K and V caches, and
seq_lens in; O, LSE and the decode output back.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal fwd attn TFLOP/s + decode KV GB/s on 1×GB300, % of roofline"
UNIT = "% of GB300 roofline (summed over GPUs)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured (MEASURED_PEAKS.json)"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback (no MEASURED_PEAKS.json)"


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "exact_attention_43_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kind):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[kind]
        src = {"decode": ("decode.cu", "ptx.cuh"), "fwd": ("fwd.cu", "ptx.cuh")}[kind]
        if d["source_sha"] == source_sha(*src):
            return float(d["bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU is busy."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = []
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s, r in zip(sm, rows) if num(r[3]) and num(r[3]) > 200.0] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(seconds, device=None):
    """The slowest rank's time (every rank gets it); the local value when not distributed."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return seconds
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def whole_job_value(roofline_s_per_step, steps, world, max_seconds):
    """Percent of one GPU's roofline, summed over the replicas (every rank runs the full step)."""
    return 100.0 * world * roofline_s_per_step * steps / max_seconds


def roofline_time(fwd_flops, dec_bytes, peaks):
    return fwd_flops / (peaks["bf16_tflops"] * 1e12) + dec_bytes / (peaks["hbm_gbs"] * 1e9)


# ---------------------------------------------------------------------------- oracle (CPU)

def oracle_sample(n_heads, n_seqs, seed_shift=0):
    """Time the float64 oracle on a bounded sample of the same workload.

    Sample: the first `n_heads` (batch 0) query heads of the MHA prefill at full
    length (2048 causal rows each) and the first `n_seqs` sequences of the decode
    batch (all 32 query heads, full prefixes).  Returns (seconds, flops, bytes).
    """
    import numpy as np  # noqa: F401
    import torch

    import oracle
    from exact_attention_43_gb300 import workloads as wl

    w = wl.MHA
    g = wl.SEED_BASE + w.index + seed_shift
    q = wl.normal((1, n_heads, w.Sq, w.D), seed=g, dtype=w.dtype)
    k = wl.normal((1, n_heads, w.Skv, w.D), seed=g + 1, dtype=w.dtype)
    v = wl.normal((1, n_heads, w.Skv, w.D), seed=g + 2, dtype=w.dtype)
    d = wl.DECODE
    lens_all = wl.seq_lens(d.B, d.len_lo, d.len_hi, seed=wl.SEED_BASE + d.index)
    lens = lens_all[:n_seqs]
    Lmax = int(lens.max())
    dq = wl.normal((n_seqs, d.Hq, d.D), seed=wl.SEED_BASE + d.index + 10, dtype=d.dtype)
    dk = wl.normal((n_seqs, d.Hkv, Lmax, d.D), seed=wl.SEED_BASE + d.index + 11, dtype=d.dtype)
    dv = wl.normal((n_seqs, d.Hkv, Lmax, d.D), seed=wl.SEED_BASE + d.index + 12, dtype=d.dtype)
    t0 = time.perf_counter()
    oracle.sdpa(q, k, v, causal=True, scale=w.scale)
    oracle.decode(dq, dk, dv, lens, scale=d.scale)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.D * n_heads * wl.visible_pairs(w.Sq, w.Skv, True)
    nbytes = int(lens.to(torch.int64).sum()) * d.Hkv * d.D * 4 + 2 * n_seqs * d.Hq * d.D * 2
    return dt, flops, nbytes


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, peaks, peaks_src):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    n_heads, n_seqs = 2, 1
    for _ in range(args.warmup):
        oracle_sample(n_heads, n_seqs)
    tot_t, tot_f, tot_b = 0.0, 0.0, 0
    for _ in range(args.steps):
        dt, f, b = oracle_sample(n_heads, n_seqs)
        tot_t += dt
        tot_f += f
        tot_b += b
    value = 100.0 * roofline_time(tot_f, tot_b, peaks) / tot_t
    sample = (f"per step: float64 oracle on {n_heads} MHA heads (S2048 D128 causal, full rows) "
              f"+ {n_seqs} decode sequence(s) of the decode batch (32 heads, full prefix)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "MHA prefill B4 H32 S2048 D128 causal + flash-decoding B64 Hq32 "
                               "Hkv8 D128 cache 32768 chunk 512 (bounded sample per step)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample,
                         "gflops": tot_f / tot_t / 1e9, "gbs": tot_b / tot_t / 1e9},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "peaks": peaks_src,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- GPU arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=3, help="0 skips the end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-soak", type=float, default=1.5,
                    help="seconds of untimed steps before the warm-up, for clock sampling")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    peaks, peaks_src = load_peaks()
    if args.impl == "reference":
        return run_reference(args, peaks, peaks_src)

    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from exact_attention_43_gb300 import build as _build

    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    import exact_attention_43_gb300 as ea
    from exact_attention_43_gb300 import workloads as wl

    ea.load()
    fw, dw = wl.MHA, wl.DECODE
    q, k, v = wl.workload_fwd_inputs(fw, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((fw.B, fw.Hq, fw.Sq), dtype=torch.float32, device=dev)
    dq, dk, dv, lens = wl.workload_decode_inputs(dw, device=dev)
    lens_d = lens.to(dev)
    do = torch.empty_like(dq)
    fwd_flops = fw.flops()
    dec_bytes = dw.io_bytes(lens)
    stream = torch.cuda.current_stream()

    def step():
        ea.attn_fwd(q, k, v, causal=True, scale=fw.scale, out=o, lse=lse, stream=stream)
        ea.attn_decode(dq, dk, dv, lens_d, num_splits=dw.num_splits, out=do, stream=stream)

    uuid = torch.cuda.get_device_properties(dev).uuid
    sampler = ClockSampler(str(uuid) if uuid else None)
    sampler.start()
    # untimed load before the warm-up so the 100 ms clock samples see the GPU busy
    soak_steps, t_end = 0, time.time() + args.clock_soak
    while time.time() < t_end:
        for _ in range(20):
            step()
        soak_steps += 20
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ea.check_device_status() != 0:
        raise RuntimeError("device status error during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        ea.attn_fwd(q, k, v, causal=True, scale=fw.scale, out=o, lse=lse, stream=stream)
        ev[i][1].record(stream)
        ea.attn_decode(dq, dk, dv, lens_d, num_splits=dw.num_splits, out=do, stream=stream)
        ev[i][2].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_s = start.elapsed_time(stop) / 1e3
    t_fwd = statistics.mean(a.elapsed_time(b) for a, b, _ in ev) / 1e3
    t_dec = statistics.mean(b.elapsed_time(c) for _, b, c in ev) / 1e3
    if ea.check_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    total_s = max_over_ranks(total_s, dev)

    # ------------------------------------------------ end to end from pinned host buffers
    e2e = None
    if args.e2e_steps > 0:
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        hdq, hdk, hdv = (x.cpu().pin_memory() for x in (dq, dk, dv))
        hlens = lens.clone().pin_memory()
        ho = torch.empty_like(hq).pin_memory()
        hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        hdo = torch.empty_like(hdq).pin_memory()
        # The decode step reads only the first seq_lens[b] rows of each (sequence, KV
        # head) of the cache, so those prefixes are what goes over each step (one
        # contiguous copy per (sequence, head) and tensor); rows past seq_lens are
        # never read.
        lens_l = [int(x) for x in lens]
        kv_prefix = [(b, h, n) for b, n in enumerate(lens_l) for h in range(hdk.shape[1]) if n > 0]
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdq, hlens))
        h2d += 2 * sum(n for _, _, n in kv_prefix) * hdk.shape[3] * hdk.element_size()
        d2h = sum(x.numel() * x.element_size() for x in (ho, hlse, hdo))

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            dq.copy_(hdq, non_blocking=True)
            for b, h, n in kv_prefix:
                dk[b, h, :n].copy_(hdk[b, h, :n], non_blocking=True)
                dv[b, h, :n].copy_(hdv[b, h, :n], non_blocking=True)
            lens_d.copy_(hlens, non_blocking=True)
            ea.attn_fwd(q, k, v, causal=True, scale=fw.scale, out=o, lse=lse, stream=stream)
            ea.attn_decode(dq, dk, dv, lens_d, num_splits=dw.num_splits, out=do, stream=stream)
            ho.copy_(o, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)
            hdo.copy_(do, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_s = e0.elapsed_time(e1) / 1e3
        e2e_s = max_over_ranks(e2e_s, dev)
        e2e = {"value": whole_job_value(roofline_time(fwd_flops, dec_bytes, peaks),
                                        args.e2e_steps, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": args.e2e_steps, "ms_per_step": 1e3 * e2e_s / args.e2e_steps}

    rt = roofline_time(fwd_flops, dec_bytes, peaks)
    value = whole_job_value(rt, args.steps, world, total_s)

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            n_heads, n_seqs = 16, 4
            dt, f, b = oracle_sample(n_heads, n_seqs)
            cpu = {"value": 100.0 * roofline_time(f, b, peaks) / dt, "unit": UNIT,
                   "cores": cpu_cores(), "kind": "oracle",
                   "sample": f"float64 oracle on {n_heads} MHA heads (S2048 D128 causal, all "
                             f"rows) + the first {n_seqs} decode sequences (32 heads, full "
                             f"prefixes); {dt:.1f} s",
                   "seconds": dt, "gflops": f / dt / 1e9, "gbs": b / dt / 1e9}
        dec_gbs = dec_bytes / t_dec / 1e9
        fwd_tflops = fwd_flops / t_fwd / 1e12
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "MHA prefill B4 H32 S2048 D128 bf16 causal + flash-decoding "
                                   "B64 Hq32 Hkv8 D128 bf16, cache [64,8,32768,128], seq_lens "
                                   "U[512,32768] (sum %d), 64 splits (chunk 512)" % int(lens.sum()),
                       "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (decode streams ~4.4 GB between prefill calls)"},
            "legs": {
                "fwd": {"ms": 1e3 * t_fwd, "tflops": fwd_tflops, "gflop": fwd_flops / 1e9,
                        "frac": fwd_tflops / peaks["bf16_tflops"]},
                "decode": {"ms": 1e3 * t_dec, "gbs": dec_gbs, "gbytes": dec_bytes / 1e9,
                           "frac": dec_gbs / peaks["hbm_gbs"]},
            },
            "roofline": {"kernel": "attn_decode (decode_split_kernel + decode_reduce_kernel)",
                         "bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
                         "traffic": traffic_for("decode"),
                         "algorithmic_bytes_per_launch": dec_bytes},
            "roofline_fwd": {"kernel": "attn_fwd_kernel<128, bf16>", "bound": "tensor",
                             "achieved": fwd_tflops, "peak": peaks["bf16_tflops"],
                             "unit": "TFLOP/s", "frac": fwd_tflops / peaks["bf16_tflops"],
                             "traffic": traffic_for("fwd"),
                             "algorithmic_flops_per_launch": fwd_flops},
            "peaks": peaks_src,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 3 * args.steps,
            "clocks": dict(clocks, window="untimed soak (%d steps) + warm-up + timed region"
                           % soak_steps),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
