"""Attention backward (attn_bwd) through the C ABI against the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import check_guards, guarded

pytestmark = pytest.mark.gpu

# The bar for gradients, from the arithmetic: the kernel rounds each gradient to
# the input's 16-bit type at the end (at most half an ulp, 2^-8 relative for bf16)
# and P and dS to 16 bits before three of the five products (the same relative
# size per term, accumulated in fp32), while the oracle is float64.  So the
# largest error may reach a few half-ulps of the largest gradient element, and the
# mean error about half an ulp of the gradient's RMS:
#   max |err| <= 4 * 2^-8 * max |ref|,   mean |err| <= 2^-8 * rms(ref).
# (Measured on the cases below: at most 0.54 % of max |ref| and 1.7e-3 rms(ref).)
G_MAX_REL = 4 * 2.0 ** -8
G_MEAN_REL = 2.0 ** -8


def compare_grad(got, want, what):
    g = got.detach().double().cpu().numpy()
    assert g.shape == want.shape, (what, g.shape, want.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    if want.size == 0:
        return
    err = np.abs(g - want)
    mx, mean = float(err.max()), float(err.mean())
    amax, rms = float(np.abs(want).max()), float(np.sqrt((want ** 2).mean()))
    assert mx <= G_MAX_REL * max(amax, 1e-3), f"{what}: max abs err {mx:.3e} (max |ref| {amax:.3e})"
    assert mean <= G_MEAN_REL * max(rms, 1e-3), f"{what}: mean abs err {mean:.3e} (rms {rms:.3e})"


def run_bwd(q, k, v, do, causal, scale):
    import exact_attention_43_gb300 as ea

    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    o, lse = ea.attn_fwd(qc, kc, vc, causal=causal, scale=scale)
    dq_f, dq = guarded(tuple(q.shape), q.dtype)
    dk_f, dk = guarded(tuple(k.shape), k.dtype)
    dv_f, dv = guarded(tuple(v.shape), v.dtype)
    ea.attn_bwd(qc, kc, vc, o, lse, doc, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    for f in (dq_f, dk_f, dv_f):
        check_guards(f)
    return dq, dk, dv


CASES = [
    # B, Hq, Hkv, Sq, Skv, D, dtype, causal
    (1, 2, 2, 256, 256, 64, torch.float16, True),
    (2, 4, 2, 300, 300, 128, torch.bfloat16, True),      # ragged tail, GQA 2
    (1, 2, 1, 200, 333, 128, torch.bfloat16, False),     # Sq != Skv, GQA 2
    (1, 2, 2, 300, 130, 128, torch.bfloat16, True),      # rows that see no key
    (1, 2, 2, 100, 400, 64, torch.bfloat16, True),       # keys before the first query's diagonal
    (1, 8, 1, 129, 257, 128, torch.bfloat16, True),      # GQA 8, one-row tails
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}x{}q{}k{}D{}{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[7] else "f"))
def test_bwd_cases(case):
    B, Hq, Hkv, Sq, Skv, D, dtype, causal = case
    q, k, v = wl.fwd_inputs(B, Hq, Hkv, Sq, Skv, D, dtype=dtype, seed=4000 + Sq + Skv)
    do = wl.normal((B, Hq, Sq, D), seed=4100 + Sq, dtype=dtype)
    scale = D ** -0.5
    dq, dk, dv = run_bwd(q, k, v, do, causal, scale)
    want = oracle.sdpa_backward(q, k, v, do, causal=causal, scale=scale)
    for name, got, w in zip(("dQ", "dK", "dV"), (dq, dk, dv), want):
        compare_grad(got, w, f"{name} {case}")


def test_bwd_mha_workload_sampled_heads():
    """B4 H32 S2048 D128 bf16 causal (the MHA workload) end to end; every gradient of
    a seeded sample of (batch, head) pairs spread over the launch -- the first and
    the last included -- against the oracle, and all gradients finite."""
    import exact_attention_43_gb300 as ea

    w = wl.MHA
    q, k, v = wl.workload_fwd_inputs(w, device="cuda")
    do = wl.normal(tuple(q.shape), seed=4200, dtype=q.dtype, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    g = torch.Generator().manual_seed(4201)
    pick = torch.randperm(w.B * w.Hq, generator=g)[:4].tolist()
    pairs = sorted({(0, 0), (w.B - 1, w.Hq - 1)} | {(i // w.Hq, i % w.Hq) for i in pick})
    for b, h in pairs:
        sl = slice(h, h + 1)
        want = oracle.sdpa_backward(q[b:b + 1, sl].cpu(), k[b:b + 1, sl].cpu(), v[b:b + 1, sl].cpu(),
                                    do[b:b + 1, sl].cpu(), causal=True, scale=w.scale)
        for name, got, wgt in zip(("dQ", "dK", "dV"), (dq[b:b + 1, sl], dk[b:b + 1, sl], dv[b:b + 1, sl]),
                                  want):
            compare_grad(got, wgt, f"{name} MHA batch {b} head {h}")


def test_bwd_gqa_workload_sampled_heads():
    """B2 Hq32 Hkv8 S8192 (the GQA workload, peaked rows): the gradients of one whole
    GQA group in each batch against the oracle (dK, dV summed over the group's four
    query heads)."""
    import exact_attention_43_gb300 as ea

    w = wl.GQA
    q, k, v = wl.workload_fwd_inputs(w, device="cuda")
    do = wl.normal(tuple(q.shape), seed=4202, dtype=q.dtype, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    G = w.Hq // w.Hkv
    for b, g in ((0, 0), (w.B - 1, w.Hkv - 1)):
        qs, ks = slice(g * G, (g + 1) * G), slice(g, g + 1)
        want = oracle.sdpa_backward(q[b:b + 1, qs].cpu(), k[b:b + 1, ks].cpu(), v[b:b + 1, ks].cpu(),
                                    do[b:b + 1, qs].cpu(), causal=True, scale=w.scale)
        for name, got, wgt in zip(("dQ", "dK", "dV"), (dq[b:b + 1, qs], dk[b:b + 1, ks], dv[b:b + 1, ks]),
                                  want):
            compare_grad(got, wgt, f"{name} GQA batch {b} group {g}")


def test_bwd_deterministic():
    """No gradient is accumulated with atomics: two calls agree bit for bit."""
    import exact_attention_43_gb300 as ea

    q, k, v = wl.fwd_inputs(1, 8, 2, 512, 512, 128, seed=4300, device="cuda")
    do = wl.normal((1, 8, 512, 128), seed=4301, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=True)
    a = ea.attn_bwd(q, k, v, o, lse, do, causal=True)
    b = ea.attn_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_bwd_gradients_only_16_byte_aligned():
    """The C ABI promises 16-byte alignment only: gradients that are not 32-byte aligned
    take 16-byte row stores (the check is on the host, per call) and must hold the same
    bits as 32-byte-aligned ones; nothing outside them is written."""
    import exact_attention_43_gb300 as ea

    q, k, v = wl.fwd_inputs(1, 4, 2, 300, 300, 128, seed=4400, device="cuda")
    do = wl.normal((1, 4, 300, 128), seed=4401, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=True)
    ref = ea.attn_bwd(q, k, v, o, lse, do, causal=True)

    def offset_view(like):
        n = like.numel()
        buf = torch.full((n + 16,), float("nan"), dtype=like.dtype, device="cuda")
        view = buf[8:8 + n].view(tuple(like.shape))
        assert view.data_ptr() % 32 == 16
        return buf, view

    (bq, dq), (bk, dk), (bv, dv) = offset_view(q), offset_view(k), offset_view(v)
    ea.attn_bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    for buf, got, want, n in ((bq, dq, ref[0], q.numel()), (bk, dk, ref[1], k.numel()),
                              (bv, dv, ref[2], v.numel())):
        assert bool(torch.isnan(buf[:8].float()).all()) and bool(torch.isnan(buf[8 + n:].float()).all())
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
