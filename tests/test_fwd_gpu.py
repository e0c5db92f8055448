"""Prefill parity: the CUDA path (through the C ABI) against the float64 oracle."""

import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import check_guards, compare_lse, compare_o, guarded

pytestmark = pytest.mark.gpu


def run_fwd(q, k, v, causal, scale):
    import exact_attention_43_gb300 as ea

    B, Hq, Sq, D = q.shape
    o_full, o = guarded((B, Hq, Sq, D), q.dtype)
    l_full, lse = guarded((B, Hq, Sq), torch.float32)
    ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, out=o, lse=lse)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    check_guards(o_full)
    check_guards(l_full)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_workload(causal):
    w = wl.TINY
    q, k, v = wl.workload_fwd_inputs(w)
    o, lse = run_fwd(q, k, v, causal, w.scale)
    ro, rl = oracle.sdpa(q, k, v, causal=causal, scale=w.scale)
    compare_o(o, ro, "tiny O")
    compare_lse(lse, rl, "tiny LSE")


SHAPES = [
    # B, Hq, Hkv, Sq, Skv, D, dtype, causal
    (1, 2, 2, 1, 1, 64, torch.float16, True),
    (1, 2, 2, 63, 63, 128, torch.bfloat16, True),
    (2, 2, 1, 64, 64, 64, torch.bfloat16, False),
    (1, 3, 3, 127, 127, 128, torch.float16, True),
    (1, 2, 2, 129, 129, 128, torch.bfloat16, True),
    (1, 4, 2, 257, 257, 64, torch.float16, False),
    (1, 4, 1, 1000, 1000, 128, torch.bfloat16, True),
    (2, 8, 1, 300, 300, 128, torch.bfloat16, True),       # G = 8
    (1, 8, 2, 512, 512, 128, torch.float16, False),       # G = 4
    (1, 2, 2, 100, 700, 128, torch.bfloat16, True),       # Sq < Skv, bottom-right
    (1, 2, 2, 700, 100, 64, torch.bfloat16, True),        # Sq > Skv: leading rows see nothing
    (1, 2, 2, 130, 5, 128, torch.float16, False),         # fewer keys than a tile
    (1, 1, 1, 384, 384, 128, torch.bfloat16, True),       # exact multiple of the tile
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}H{}x{}S{}x{}D{}{}{}".format(
    s[0], s[1], s[2], s[3], s[4], s[5], "f16" if s[6] == torch.float16 else "bf16",
    "c" if s[7] else "n"))
def test_ragged_shapes(shape):
    B, Hq, Hkv, Sq, Skv, D, dtype, causal = shape
    q, k, v = wl.fwd_inputs(B, Hq, Hkv, Sq, Skv, D, dtype=dtype, seed=1000 + Sq + Skv + D)
    scale = 1.0 / np.sqrt(D)
    o, lse = run_fwd(q, k, v, causal, scale)
    ro, rl = oracle.sdpa(q, k, v, causal=causal, scale=scale)
    compare_o(o, ro, f"{shape} O")
    compare_lse(lse, rl, f"{shape} LSE")


@pytest.mark.parametrize("scale", [0.0, -0.2, 0.5])
def test_unusual_scales(scale):
    q, k, v = wl.fwd_inputs(1, 2, 2, 200, 200, 64, dtype=torch.bfloat16, seed=77)
    o, lse = run_fwd(q, k, v, True, scale)
    ro, rl = oracle.sdpa(q, k, v, causal=True, scale=scale)
    compare_o(o, ro, f"scale {scale} O")
    compare_lse(lse, rl, f"scale {scale} LSE")


def test_peaked_rows_need_rescaling():
    # Q ~ N(0, 3^2) (as the GQA workload) makes the running max jump between tiles
    q, k, v = wl.fwd_inputs(1, 4, 1, 1024, 1024, 128, dtype=torch.bfloat16, seed=5, q_std=3.0)
    o, lse = run_fwd(q, k, v, True, 1 / np.sqrt(128))
    ro, rl = oracle.sdpa(q, k, v, causal=True, scale=1 / np.sqrt(128))
    compare_o(o, ro, "peaked O")
    compare_lse(lse, rl, "peaked LSE")


def test_empty_keys_and_lse_optional():
    import exact_attention_43_gb300 as ea

    q, k, v = wl.fwd_inputs(1, 2, 2, 10, 0, 64, dtype=torch.float16, seed=3)
    o, lse = run_fwd(q, k, v, False, 0.125)
    assert bool((o == 0).all()) and bool(torch.isneginf(lse).all())
    q, k, v = wl.fwd_inputs(1, 2, 2, 70, 70, 64, dtype=torch.float16, seed=4)
    o2, none = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, return_lse=False)
    assert none is None
    ro, _ = oracle.sdpa(q, k, v, causal=True, scale=0.125)
    compare_o(o2, ro, "no-LSE O")


def test_deterministic():
    import exact_attention_43_gb300 as ea

    q, k, v = wl.fwd_inputs(2, 4, 2, 700, 700, 128, dtype=torch.bfloat16, seed=9, device="cuda")
    a = ea.attn_fwd(q, k, v, causal=True)
    b = ea.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])


def _full_size(w, rows_per_head=None, seed=0):
    """Run a workload at full size (the launch the bench times) and check it against
    the oracle, head by head: every row when rows_per_head is None, else
    rows_per_head seeded rows of [1, S-1) per head plus rows 0 and S-1.  The
    oracle runs per (batch, head) in a few threads (numpy releases the GIL), so
    host memory stays at a few score matrices."""
    import exact_attention_43_gb300 as ea

    q, k, v = wl.workload_fwd_inputs(w, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    S, G = w.Sq, w.Hq // w.Hkv
    qc, kc, vc, oc, lc = q.cpu(), k.cpu(), v.cpu(), o.cpu(), lse.cpu()

    def check(bh):
        b, h = bh
        rows = None
        if rows_per_head is not None:
            rows = np.sort(np.concatenate([
                wl.sample_rows(S - 2, rows_per_head, seed=seed + h).numpy() + 1, [0, S - 1]]))
        g = h // G
        ro, rl = oracle.sdpa(qc[b:b + 1, h:h + 1], kc[b:b + 1, g:g + 1], vc[b:b + 1, g:g + 1],
                             causal=w.causal, scale=w.scale, rows=rows)
        idx = slice(None) if rows is None else torch.as_tensor(rows)
        compare_o(oc[b, h, idx][None, None], ro, f"{w.name} b={b} h={h} O")
        compare_lse(lc[b, h, idx][None, None], rl, f"{w.name} b={b} h={h} LSE")

    pairs = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(6, os.cpu_count() or 1))) as ex:
        list(ex.map(check, pairs))
    return o, lse


def test_mha_workload_full_size():
    # every row of every head (B4 H32 S2048: 137 GFLOP of float64)
    _full_size(wl.MHA)


def test_gqa_workload_full_size():
    # every row of every head (B2 Hq32 Hkv8 S8192, peaked rows: 1.1 TFLOP of float64)
    _full_size(wl.GQA)


def test_long_workload_full_size():
    # 512 seeded-random query rows per head plus rows 0 and S-1, full-length keys
    _full_size(wl.LONG, 512, seed=wl.SEED_BASE + 3)


def test_output_only_16_byte_aligned():
    # the C ABI promises 16-byte alignment only: an O that is not 32-byte aligned takes
    # 16-byte stores (the check is on the host, per call)
    import exact_attention_43_gb300 as ea

    q, k, v = wl.fwd_inputs(1, 2, 2, 300, 300, 128, dtype=torch.bfloat16, seed=31)
    shape = tuple(q.shape)
    n = int(np.prod(shape))
    buf = torch.full((n + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = buf[8:].view(shape)
    assert o.data_ptr() % 32 == 16
    ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=128 ** -0.5, out=o)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    assert bool(torch.isnan(buf[:8].float()).all())
    ro, _ = oracle.sdpa(q, k, v, causal=True, scale=128 ** -0.5)
    compare_o(o, ro, "16-byte aligned O")
