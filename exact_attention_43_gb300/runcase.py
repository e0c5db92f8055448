"""Run one synthetic attention case a few times (for profiling and timing).

    python -m exact_attention_43_gb300.runcase fwd --workload mha [--iters 3]
    python -m exact_attention_43_gb300.runcase fwd --B 1 --H 8 --S 4096 --causal 1
    python -m exact_attention_43_gb300.runcase fwd --workload mha --layout qkvpacked [--window 256]
    python -m exact_attention_43_gb300.runcase bwd --workload mha
    python -m exact_attention_43_gb300.runcase decode [--B 8] [--iters 3] [--page-size 64 | --fused]

Inputs are drawn on the GPU from the seeded generators in workloads.py.
Prints one JSON line with the mean CUDA-event time per call.
"""

from __future__ import annotations

import argparse
import json

import torch

from . import binding as ea
from . import workloads as wl


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["fwd", "bwd", "decode"])
    ap.add_argument("--workload", default=None, help="tiny | mha | gqa | long (fwd)")
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--Hkv", type=int, default=None)
    ap.add_argument("--S", type=int, default=2048)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--causal", type=int, default=1)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--page-size", type=int, default=0, help="decode over a paged cache")
    ap.add_argument("--fused", action="store_true", help="single-launch decode (attn_decode_fused)")
    ap.add_argument("--layout", default="dense", choices=["dense", "varlen", "qkvpacked"],
                    help="fwd: [B,H,S,D] arrays, packed sequences, or one [B,S,3,H,D] projection")
    ap.add_argument("--window", type=int, default=-1, help="fwd token-major layouts: left window")
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    ea.load()
    if a.op in ("fwd", "bwd"):
        if a.workload:
            w = wl.FWD_WORKLOADS[a.workload]
        else:
            w = wl.FwdWorkload("custom", 9, a.B or 1, a.H, a.Hkv or a.H, a.S, a.S, a.D,
                               torch.bfloat16, bool(a.causal))
        q, k, v = wl.workload_fwd_inputs(w, device=dev)
        units, unit = w.flops(), "TFLOP/s"
        desc = f"{w.name} B{w.B} Hq{w.Hq} Hkv{w.Hkv} S{w.Sq} D{w.D} causal={w.causal}"
        if a.op == "bwd":
            # five products per (query, key) pair against the forward's two
            units = 2.5 * w.flops()
            desc += " backward"
            do = wl.normal(tuple(q.shape), seed=wl.SEED_BASE + 50, dtype=q.dtype, device=dev)
            o, lse = ea.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)

            def call():
                return ea.attn_bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
        elif a.layout == "dense":
            def call():
                return ea.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
        else:
            win = (a.window, -1)
            if a.window >= 0:  # flops of the keys the window keeps, counted row by row
                diag = torch.arange(w.Sq, dtype=torch.int64) + (w.Skv - w.Sq)
                hi = torch.clamp(diag if w.causal else torch.full_like(diag, w.Skv - 1), max=w.Skv - 1)
                lo = torch.clamp(diag - a.window, min=0)
                units = 4.0 * w.B * w.Hq * w.D * float(torch.clamp(hi - lo + 1, min=0).sum())
                desc += f" window={a.window}"
            desc += f" {a.layout}"
            if a.layout == "qkvpacked":
                assert w.Hq == w.Hkv and w.Sq == w.Skv
                qkv = torch.stack([x.transpose(1, 2) for x in (q, k, v)], dim=2).contiguous()
                del q, k, v

                def call():
                    return ea.attn_fwd_qkvpacked(qkv, causal=w.causal, window=win, scale=w.scale)
            else:
                tq, tk, tv = (x.transpose(1, 2).reshape(-1, x.shape[1], x.shape[3]).contiguous()
                              for x in (q, k, v))
                del q, k, v
                cq = torch.arange(0, (w.B + 1) * w.Sq, w.Sq, dtype=torch.int32, device=dev)
                ck = torch.arange(0, (w.B + 1) * w.Skv, w.Skv, dtype=torch.int32, device=dev)

                def call():
                    return ea.attn_fwd_varlen(tq, tk, tv, cq, ck, w.Sq, w.Skv, causal=w.causal,
                                              window=win, scale=w.scale)
    else:
        d = wl.DECODE
        B = a.B or d.B
        lens = wl.seq_lens(d.B, d.len_lo, d.len_hi, seed=wl.SEED_BASE + d.index)[:B]
        q, k, v, lens = wl.decode_inputs(B, d.Hq, d.Hkv, d.max_S, d.D, lens, dtype=d.dtype,
                                         seed=wl.SEED_BASE + d.index, device=dev)
        lens_d = lens.to(dev)
        desc = f"decode B{B} Hq{d.Hq} Hkv{d.Hkv} max_S{d.max_S} D{d.D} sumL={int(lens.sum())}"
        if a.page_size > 0:
            kp, vp, table = wl.paged_cache(k, v, [int(x) for x in lens], a.page_size,
                                           seed=wl.SEED_BASE + d.index + 100)
            del k, v
            kp, vp, table = kp.to(dev), vp.to(dev), table.to(dev)
            desc += f" paged {a.page_size}"

            def call():
                return ea.attn_decode_paged(q, kp, vp, table, lens_d, num_splits=d.num_splits)
        elif a.fused:
            desc += " fused"

            def call():
                return ea.attn_decode_fused(q, k, v, lens_d, num_splits=d.num_splits)
        else:
            def call():
                return ea.attn_decode(q, k, v, lens_d, num_splits=d.num_splits)

        units, unit = d.io_bytes(lens), "GB/s"
    for _ in range(a.warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        call()
    e1.record()
    torch.cuda.synchronize()
    st = ea.check_device_status()
    ms = e0.elapsed_time(e1) / a.iters
    rate = units / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
    print(json.dumps({"case": desc, "ms": ms, unit: rate, "status": st}))
    return 0 if st == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
