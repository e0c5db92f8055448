"""Benchmark of the fused-attention hot path on GB300.

A step is one pass of the whole path over one batch of synthetic inputs, the
three prefill workloads and the decode batch:
  1. attn_fwd    -- MHA prefill B4 H32 S2048 D128 bf16, causal (137.5 GFLOP);
  2. attn_fwd    -- GQA prefill B2 Hq32 Hkv8 S8192 D128 bf16, causal, Q ~ N(0, 9)
                    (1.0996 TFLOP);
  3. attn_fwd    -- long-context prefill B1 H32 S32768 D128 bf16, causal
                    (8.796 TFLOP);
  4. attn_decode -- flash-decoding B64 Hq32 Hkv8 D128 bf16 over a cache
                    [64, 8, 32768, 128] with seq_lens uniform in [512, 32768],
                    64 splits (chunk 512; about 4.33 GB of K/V prefixes read).
The metric is the step's share of the GPU roofline: the time the step would
take at the measured peaks (prefill flops at the dense bf16 tensor peak, plus
decode bytes at the HBM copy bandwidth) divided by the measured time, in
percent, summed over GPUs for N > 1.  Per-leg TFLOP/s and GB/s, each with its
fraction of the peak, are reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

Timing: CUDA events on the launching stream around exactly K steps, with a
barrier and a device synchronize on both sides, and around every leg of every
step; inputs are larger than L2 (the long prefill reads 0.8 GB and the decode
leg streams ~4.3 GB between the other legs, so no leg starts with a warm L2).
Inputs are resident in HBM when the timed region starts; the e2e figure
repeats the step from pinned host buffers with the copies inside its timed
region: every prefill's Q, K, V, the decode queries, the valid prefix
(seq_lens rows) of every (sequence, KV head) of the K and V caches, and
seq_lens in; every O, LSE and the decode output back.  The copies overlap the
computation as a serving loop would: a leg's inputs go over on a copy stream while
the legs before it compute, and its results come back on another stream while the
legs after it compute; a step ends when its last result is on the host.  The
backward (attn_bwd)
of the three prefill workloads is timed after the step, in a loop of its own,
and reported under "backward"; it is not part of the metric.
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
WORKLOAD = ("prefill MHA B4 H32 S2048 + GQA B2 Hq32 Hkv8 S8192 (Q ~ N(0,9)) + long-context "
            "B1 H32 S32768, D128 bf16 causal; flash-decoding B64 Hq32 Hkv8 D128 bf16, cache "
            "[64,8,32768,128], seq_lens U[512,32768], 64 splits (chunk 512)")
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
        src = ("decode.cu", "ptx.cuh") if kind == "decode" else ("fwd.cu", "ptx.cuh")
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
    """Seconds the work would take at the peaks: flops at the dense bf16 tensor peak plus
    bytes at the HBM copy bandwidth."""
    return fwd_flops / (peaks["bf16_tflops"] * 1e12) + dec_bytes / (peaks["hbm_gbs"] * 1e9)


# ---------------------------------------------------------------------------- oracle (CPU)

def oracle_sample(mha_heads, gqa_heads, gqa_rows, long_heads, long_rows, n_seqs):
    """Time the float64 oracle on a bounded sample of the step's workloads.

    Sample: the first `mha_heads` (batch 0) query heads of the MHA prefill at full
    length (2048 causal rows each); `gqa_rows` seeded rows (None: all 8192) of each
    of the first `gqa_heads` GQA query heads; `long_rows` seeded rows of each of
    the first `long_heads` long-context heads, against their full causal key
    prefixes; and the first `n_seqs` sequences of the decode batch (all 32 query
    heads, full prefixes).  Returns (seconds, flops, bytes) of the sample.
    """
    import numpy as np
    import torch

    import oracle
    from exact_attention_43_gb300 import workloads as wl

    parts = []  # (q, k, v, scale, rows, flops)
    for w, heads, nrows in ((wl.MHA, mha_heads, None), (wl.GQA, gqa_heads, gqa_rows),
                            (wl.LONG, long_heads, long_rows)):
        if heads == 0:
            continue
        g = wl.SEED_BASE + w.index
        G = w.Hq // w.Hkv
        if heads > G and heads % G:
            raise ValueError("sample whole GQA groups, or heads of one group")
        hk = -(-heads // G)  # KV heads the sampled query heads read (h -> h // G)
        q = wl.normal((1, heads, w.Sq, w.D), seed=g, std=w.q_std, dtype=w.dtype)
        k = wl.normal((1, hk, w.Skv, w.D), seed=g + 1, dtype=w.dtype)
        v = wl.normal((1, hk, w.Skv, w.D), seed=g + 2, dtype=w.dtype)
        rows = None
        if nrows is None:
            flops = 4.0 * w.D * q.shape[1] * wl.visible_pairs(w.Sq, w.Skv, True)
        else:
            rows = wl.sample_rows(w.Sq, nrows, seed=g + 7).numpy()
            flops = 4.0 * w.D * q.shape[1] * float(np.sum(rows + 1))
        parts.append((q, k, v, w.scale, rows, flops))
    d = wl.DECODE
    lens_all = wl.seq_lens(d.B, d.len_lo, d.len_hi, seed=wl.SEED_BASE + d.index)
    lens = lens_all[:n_seqs]
    Lmax = int(lens.max())
    dq = wl.normal((n_seqs, d.Hq, d.D), seed=wl.SEED_BASE + d.index + 10, dtype=d.dtype)
    dk = wl.normal((n_seqs, d.Hkv, Lmax, d.D), seed=wl.SEED_BASE + d.index + 11, dtype=d.dtype)
    dv = wl.normal((n_seqs, d.Hkv, Lmax, d.D), seed=wl.SEED_BASE + d.index + 12, dtype=d.dtype)
    t0 = time.perf_counter()
    for q, k, v, scale, rows, _ in parts:
        oracle.sdpa(q, k, v, causal=True, scale=scale, rows=rows)
    oracle.decode(dq, dk, dv, lens, scale=d.scale)
    dt = time.perf_counter() - t0
    flops = sum(p[5] for p in parts)
    nbytes = int(lens.to(torch.int64).sum()) * d.Hkv * d.D * 4 + 2 * n_seqs * d.Hq * d.D * 2
    return dt, flops, nbytes


def sample_text(mha_heads, gqa_heads, gqa_rows, long_heads, long_rows, n_seqs):
    return (f"float64 oracle on {mha_heads} MHA heads (S2048, all rows), {gqa_heads} GQA heads "
            f"({'all' if gqa_rows is None else gqa_rows} of 8192 rows), {long_heads} long-context "
            f"heads ({long_rows} seeded rows of 32768, full causal prefixes) and {n_seqs} decode "
            f"sequence(s) (32 heads, full prefixes)")


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


REF_SAMPLE = (1, 1, 64, 1, 64, 1)    # per step of --impl reference
CPU_SAMPLE = (32, 4, None, 2, 512, 8)  # cpu_baseline of the GPU arm (~10 s of CPU work)


def run_reference(args, peaks, peaks_src):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_sample(*REF_SAMPLE)
    tot_t, tot_f, tot_b = 0.0, 0.0, 0
    for _ in range(args.steps):
        dt, f, b = oracle_sample(*REF_SAMPLE)
        tot_t += dt
        tot_f += f
        tot_b += b
    value = 100.0 * roofline_time(tot_f, tot_b, peaks) / tot_t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD + " (bounded sample per step)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": "per step: " + sample_text(*REF_SAMPLE),
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
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=2, help="0 skips the end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bwd-steps", type=int, default=5,
                    help="timed backward steps after the main loop (0 skips them)")
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
    stream = torch.cuda.current_stream()

    # ------------------------------------------------ resident inputs and outputs
    fwd_legs = []  # (name, workload, q, k, v, o, lse)
    for name, w in (("fwd_mha", wl.MHA), ("fwd_gqa", wl.GQA), ("fwd_long", wl.LONG)):
        q, k, v = wl.workload_fwd_inputs(w, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
        fwd_legs.append((name, w, q, k, v, o, lse))
    dw = wl.DECODE
    dq, dk, dv, lens = wl.workload_decode_inputs(dw, device=dev)
    lens_d = lens.to(dev)
    do = torch.empty_like(dq)
    dec_bytes = dw.io_bytes(lens)
    fwd_flops = {name: w.flops() for name, w, *_ in fwd_legs}
    total_flops = sum(fwd_flops.values())
    n_legs = len(fwd_legs) + 1

    def run_leg(i):
        if i < len(fwd_legs):
            _, w, q, k, v, o, lse = fwd_legs[i]
            ea.attn_fwd(q, k, v, causal=True, scale=w.scale, out=o, lse=lse, stream=stream)
        else:
            ea.attn_decode(dq, dk, dv, lens_d, num_splits=dw.num_splits, out=do, stream=stream)

    def step():
        for i in range(n_legs):
            run_leg(i)

    uuid = torch.cuda.get_device_properties(dev).uuid
    sampler = ClockSampler(str(uuid) if uuid else None)
    sampler.start()
    # untimed load before the warm-up so the 100 ms clock samples see the GPU busy
    soak_steps, t_end = 0, time.time() + args.clock_soak
    while time.time() < t_end:
        for _ in range(5):
            step()
        soak_steps += 5
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ea.check_device_status() != 0:
        raise RuntimeError("device status error during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_legs + 1)]
          for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        for j in range(n_legs):
            run_leg(j)
            ev[i][j + 1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    total_s = start.elapsed_time(stop) / 1e3
    leg_s = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev) / 1e3 for j in range(n_legs)]
    if ea.check_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    total_s = max_over_ranks(total_s, dev)

    # ------------------------------------------------ end to end from pinned host buffers
    e2e = None
    if args.e2e_steps > 0:
        host_fwd = []
        h2d = d2h = 0
        for _, _, q, k, v, o, lse in fwd_legs:
            hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
            ho = torch.empty_like(hq).pin_memory()
            hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
            host_fwd.append((hq, hk, hv, ho, hl))
            h2d += sum(x.numel() * x.element_size() for x in (hq, hk, hv))
            d2h += sum(x.numel() * x.element_size() for x in (ho, hl))
        hdq, hdk, hdv = (x.cpu().pin_memory() for x in (dq, dk, dv))
        hlens = lens.clone().pin_memory()
        hdo = torch.empty_like(hdq).pin_memory()
        # The decode step reads only the first seq_lens[b] rows of each (sequence, KV
        # head) of the cache, so those prefixes are what goes over each step (one
        # contiguous copy per (sequence, head) and tensor); rows past seq_lens are
        # never read.
        lens_l = [int(x) for x in lens]
        kv_prefix = [(b, h, n) for b, n in enumerate(lens_l) for h in range(hdk.shape[1]) if n > 0]
        h2d += sum(x.numel() * x.element_size() for x in (hdq, hlens))
        h2d += 2 * sum(n for _, _, n in kv_prefix) * hdk.shape[3] * hdk.element_size()
        d2h += hdo.numel() * hdo.element_size()

        # Copies overlap compute: each leg's inputs go over on a copy stream as soon as
        # that leg's previous computation has read its buffers, the legs compute in order
        # on the compute stream once their inputs are in, and each leg's results come
        # back on a third stream; a step ends when its last results are on the host.
        h2d_stream = torch.cuda.Stream(device=dev)
        d2h_stream = torch.cuda.Stream(device=dev)
        freed = [torch.cuda.Event() for _ in range(n_legs)]  # leg i read its inputs

        def leg_h2d(i):
            if i < len(fwd_legs):
                _, _, q, k, v, _, _ = fwd_legs[i]
                hq, hk, hv, _, _ = host_fwd[i]
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
            else:
                dq.copy_(hdq, non_blocking=True)
                for b, h, n in kv_prefix:
                    dk[b, h, :n].copy_(hdk[b, h, :n], non_blocking=True)
                    dv[b, h, :n].copy_(hdv[b, h, :n], non_blocking=True)
                lens_d.copy_(hlens, non_blocking=True)

        def leg_d2h(i):
            if i < len(fwd_legs):
                _, _, _, _, _, o, lse = fwd_legs[i]
                _, _, _, ho, hl = host_fwd[i]
                ho.copy_(o, non_blocking=True)
                hl.copy_(lse, non_blocking=True)
            else:
                hdo.copy_(do, non_blocking=True)

        def e2e_step():
            h2d_stream.wait_stream(stream)  # nothing of this step starts before it
            ready = []
            with torch.cuda.stream(h2d_stream):
                for i in range(n_legs):
                    h2d_stream.wait_event(freed[i])
                    leg_h2d(i)
                    ev_i = torch.cuda.Event()
                    ev_i.record(h2d_stream)
                    ready.append(ev_i)
            for i in range(n_legs):
                stream.wait_event(ready[i])
                run_leg(i)
                freed[i].record(stream)
                d2h_stream.wait_event(freed[i])
                with torch.cuda.stream(d2h_stream):
                    leg_d2h(i)
            stream.wait_stream(d2h_stream)

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
        e2e = {"value": whole_job_value(roofline_time(total_flops, dec_bytes, peaks),
                                        args.e2e_steps, world, e2e_s), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": args.e2e_steps, "ms_per_step": 1e3 * e2e_s / args.e2e_steps}

    # ------------------------------------------------ backward of the three prefill workloads
    # (reported beside the step, timed in a loop of its own after it; not in the metric)
    bwd_legs = None
    if args.bwd_steps > 0:
        grads = []
        for name, w, q, k, v, o, lse in fwd_legs:
            do_ = wl.normal(tuple(q.shape), seed=wl.SEED_BASE + 50 + w.index, dtype=q.dtype, device=dev)
            grads.append((name, w, q, k, v, o, lse, do_, torch.empty_like(q), torch.empty_like(k),
                          torch.empty_like(v)))

        def run_bwd(g):
            name, w, q, k, v, o, lse, do_, gq, gk, gv = g
            ea.attn_bwd(q, k, v, o, lse, do_, causal=True, scale=w.scale, dq=gq, dk=gk, dv=gv,
                        stream=stream)

        for g in grads:
            run_bwd(g)
        torch.cuda.synchronize()
        bev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(grads) + 1)]
               for _ in range(args.bwd_steps)]
        for i in range(args.bwd_steps):
            bev[i][0].record(stream)
            for j, g in enumerate(grads):
                run_bwd(g)
                bev[i][j + 1].record(stream)
        torch.cuda.synchronize()
        if ea.check_device_status() != 0:
            raise RuntimeError("device status error in the backward loop")
        bwd_legs = {}
        for j, (name, w, *_r) in enumerate(grads):
            t = statistics.mean(e[j].elapsed_time(e[j + 1]) for e in bev) / 1e3
            fl = 2.5 * w.flops()  # dQ, dK, dV: five products per visible pair against the forward's two
            bwd_legs[name.replace("fwd", "bwd")] = {
                "ms": 1e3 * t, "tflops": fl / t / 1e12, "gflop": fl / 1e9,
                "frac": fl / t / 1e12 / peaks["bf16_tflops"], "frac_of": "measured dense bf16 peak (burst)",
                "note": "flops counted as 2.5x the forward's; the kernels execute 3.5x (dS, dP recomputed "
                        "for dQ)"}
        del grads

    rt = roofline_time(total_flops, dec_bytes, peaks)
    value = whole_job_value(rt, args.steps, world, total_s)

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            dt, f, b = oracle_sample(*CPU_SAMPLE)
            cpu = {"value": 100.0 * roofline_time(f, b, peaks) / dt, "unit": UNIT,
                   "cores": cpu_cores(), "kind": "oracle",
                   "sample": sample_text(*CPU_SAMPLE) + f"; {dt:.1f} s",
                   "seconds": dt, "gflops": f / dt / 1e9, "gbs": b / dt / 1e9}
        pk_t, pk_b = peaks["bf16_tflops"], peaks["hbm_gbs"]
        legs, rooflines = {}, {}
        for j, (name, w, *_rest) in enumerate(fwd_legs):
            tf = fwd_flops[name] / leg_s[j] / 1e12
            legs[name] = {"ms": 1e3 * leg_s[j], "tflops": tf, "gflop": fwd_flops[name] / 1e9,
                          "frac": tf / pk_t, "frac_of": "measured dense bf16 peak (burst)"}
            rooflines[name] = {"kernel": "attn_fwd_kernel<128, bf16>", "bound": "tensor",
                               "achieved": tf, "peak": pk_t, "unit": "TFLOP/s", "frac": tf / pk_t,
                               "traffic": traffic_for(name),
                               "algorithmic_flops_per_launch": fwd_flops[name]}
        dec_gbs = dec_bytes / leg_s[-1] / 1e9
        legs["decode"] = {"ms": 1e3 * leg_s[-1], "gbs": dec_gbs, "gbytes": dec_bytes / 1e9,
                          "frac": dec_gbs / pk_b, "frac_of": "measured HBM copy bandwidth"}
        fwd_s = sum(leg_s[:len(fwd_legs)])
        fwd_tf = total_flops / fwd_s / 1e12
        tr = [traffic_for(name) for name, *_ in fwd_legs]
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD + " (sum seq_lens %d)" % int(lens.sum()),
                       "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (the long prefill reads 0.8 GB and the decode "
                             "leg streams ~4.3 GB between the other legs)"},
            "legs": legs,
            "backward": bwd_legs,
            # the dominant kernel: the prefill kernel over the step's three launches
            # (flops and DRAM bytes per launch averaged over them)
            "roofline": {"kernel": "attn_fwd_kernel<128, bf16> (MHA, GQA and long-context "
                                   "launches of the step)",
                         "bound": "tensor", "achieved": fwd_tf, "peak": pk_t, "unit": "TFLOP/s",
                         "frac": fwd_tf / pk_t,
                         "traffic": (sum(tr) / len(tr)) if all(t is not None for t in tr) else None,
                         "algorithmic_flops_per_launch": total_flops / len(fwd_legs),
                         "peak_of": "measured dense bf16 (burst)"},
            "roofline_legs": dict(rooflines, decode={
                "kernel": "attn_decode (decode_split_kernel + decode_reduce_kernel)",
                "bound": "hbm", "achieved": dec_gbs, "peak": pk_b, "unit": "GB/s",
                "frac": dec_gbs / pk_b, "traffic": traffic_for("decode"),
                "algorithmic_bytes_per_launch": dec_bytes}),
            "peaks": peaks_src,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": (len(fwd_legs) + 2) * args.steps,
            "clocks": dict(clocks, window="untimed soak (%d steps) + warm-up + timed region"
                           % soak_steps),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
