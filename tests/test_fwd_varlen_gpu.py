"""Token-major prefill (attn_fwd_varlen, attn_fwd_qkvpacked): packed sequences of
different lengths, sliding windows and a packed QKV projection, through the C ABI,
against the float64 oracle; equal-length batches against the dense attn_fwd."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import CANARY16, check_guards, compare_lse, compare_o, guarded

pytestmark = pytest.mark.gpu

CASES = [
    # name, query lengths, key lengths, Hq, Hkv, D, dtype, causal, (window_left, window_right)
    ("ragged_causal", [1, 127, 128, 129, 300, 513], None, 4, 2, 128, torch.bfloat16, True, (-1, -1)),
    ("ragged_full_kv_longer", [100, 257, 0, 64], [300, 257, 50, 1], 4, 4, 64, torch.float16,
     False, (-1, -1)),
    ("window_causal", [600, 300], None, 2, 1, 128, torch.bfloat16, True, (128, -1)),
    ("window_two_sided", [500, 130], [700, 200], 4, 2, 128, torch.bfloat16, False, (100, 50)),
    ("window_diagonal", [300], None, 2, 2, 64, torch.float16, True, (0, -1)),
    ("window_narrow_long", [1000], None, 2, 2, 128, torch.bfloat16, True, (5, -1)),
    ("window_right_only", [260, 390], None, 2, 2, 128, torch.bfloat16, False, (-1, 70)),
    ("queries_past_keys", [400, 200, 3], [100, 0, 300], 2, 1, 128, torch.bfloat16, True, (-1, -1)),
    ("gqa8_window", [777], [1200], 16, 2, 128, torch.bfloat16, True, (300, -1)),
]


def run_varlen(q, k, v, cu_q, cu_k, lens_q, lens_k, causal, window, pad):
    import exact_attention_43_gb300 as ea

    Hq = q.shape[1]
    o_full, o = guarded(tuple(q.shape), q.dtype)
    l_full, lse = guarded((Hq, q.shape[0]), torch.float32)
    ea.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), max(lens_q),
                       max(lens_k), causal=causal, window=window, out=o, lse=lse)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    check_guards(o_full)
    check_guards(l_full)
    n = int(cu_q[-1])
    # rows outside every sequence keep their canary
    assert bool((o[n:].contiguous().view(torch.int16) == CANARY16).all())
    return o[:n], lse[:, :n]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_varlen_cases(case):
    name, lq, lk, Hq, Hkv, D, dtype, causal, window = case
    lk = lq if lk is None else lk
    q, k, v, cu_q, cu_k = wl.varlen_inputs(lq, lk, Hq, Hkv, D, dtype=dtype, seed=3000 + len(name),
                                           pad_q=5)
    o, lse = run_varlen(q, k, v, cu_q, cu_k, lq, lk, causal, window, pad=5)
    n = int(cu_q[-1])
    want_o, want_l = oracle.sdpa_varlen(q[:n], k, v, cu_q, cu_k, causal=causal, scale=D ** -0.5,
                                        window_left=window[0], window_right=window[1])
    compare_o(o, want_o, name)
    compare_lse(lse, want_l, name)


def test_no_keys_at_all():
    import exact_attention_43_gb300 as ea

    lq = [70, 0, 200]
    q, _, _, cu_q, _ = wl.varlen_inputs(lq, [0, 0, 0], 2, 2, 128, seed=3100)
    cu_k = torch.zeros(4, dtype=torch.int32)
    empty = torch.empty((0, 2, 128), dtype=q.dtype, device="cuda")
    o, lse = ea.attn_fwd_varlen(q.cuda(), empty, empty, cu_q.cuda(), cu_k.cuda(), 200, 0)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    assert bool((o == 0).all()) and bool(torch.isneginf(lse).all())


def test_bad_offsets_are_clamped_and_reported():
    import exact_attention_43_gb300 as ea

    q, k, v, _, _ = wl.varlen_inputs([100, 60], [100, 60], 2, 2, 64, dtype=torch.float16, seed=3200)
    cu_q = torch.tensor([0, 100, 90], dtype=torch.int32)     # decreasing
    cu_k = torch.tensor([0, 100, 400], dtype=torch.int32)    # past total_k = 160
    o = torch.zeros_like(q, device="cuda")
    ea.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(), 100, 300, out=o)
    assert ea.check_device_status() == 1                     # ATTN_ERR_INVALID_ARG
    assert bool(torch.isfinite(o.float()).all())
    assert ea.check_device_status() == 0


@pytest.mark.parametrize("causal,window,S,D", [(True, (-1, -1), 1000, 128), (True, (200, -1), 700, 64),
                                               (False, (64, 64), 520, 128)])
def test_qkvpacked(causal, window, S, D):
    import exact_attention_43_gb300 as ea

    B, H = 2, 4
    qkv = wl.normal((B, S, 3, H, D), seed=3300 + S, dtype=torch.bfloat16)
    o, lse = ea.attn_fwd_qkvpacked(qkv.cuda(), causal=causal, window=window)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    q, k, v = (qkv[:, :, i].permute(0, 2, 1, 3) for i in range(3))
    want_o, want_l = oracle.sdpa(q, k, v, causal=causal, scale=D ** -0.5, window_left=window[0],
                                 window_right=window[1])
    compare_o(o, want_o.transpose(0, 2, 1, 3), f"qkvpacked S{S}")
    compare_lse(lse, want_l.transpose(1, 0, 2), f"qkvpacked S{S}")


@pytest.mark.parametrize("S", [1024, 1000])
def test_equal_lengths_match_dense_bitwise(S):
    """Same arithmetic in the same order: the token-major kernel reproduces the dense
    one bit for bit on an equal-length batch (also when S ends inside a Q tile)."""
    import exact_attention_43_gb300 as ea

    B, H, D = 2, 4, 128
    q, k, v = wl.fwd_inputs(B, H, H, S, S, D, seed=3400, device="cuda")
    o_d, l_d = ea.attn_fwd(q, k, v, causal=True)
    tm = [x.transpose(1, 2).reshape(B * S, H, D).contiguous() for x in (q, k, v)]
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device="cuda")
    o_v, l_v = ea.attn_fwd_varlen(*tm, cu, cu, S, S, causal=True)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    assert torch.equal(o_v.view(B, S, H, D).transpose(1, 2).contiguous().view(torch.int16),
                       o_d.view(torch.int16))
    assert torch.equal(l_v.view(H, B, S).transpose(0, 1), l_d)


def test_mha_workload_packed_qkv_full_size():
    """B4 H32 S2048 D128 bf16 causal as one [B, S, 3, H, D] projection: equal to the dense
    kernel bit for bit, and sampled rows against the oracle."""
    import exact_attention_43_gb300 as ea

    w = wl.MHA
    q, k, v = wl.workload_fwd_inputs(w, device="cuda")
    qkv = torch.stack([x.transpose(1, 2) for x in (q, k, v)], dim=2).contiguous()
    o_p, l_p = ea.attn_fwd_qkvpacked(qkv, causal=True)
    o_d, l_d = ea.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    assert torch.equal(o_p.transpose(1, 2).contiguous().view(torch.int16), o_d.view(torch.int16))
    assert torch.equal(l_p.transpose(0, 1), l_d)
    rows = wl.sample_rows(w.Sq, 64, seed=3500)
    want_o, want_l = oracle.sdpa(q[:1].cpu(), k[:1].cpu(), v[:1].cpu(), causal=True,
                                 scale=w.scale, rows=rows)
    compare_o(o_p[:1, rows].transpose(1, 2), want_o, "packed MHA rows")
    compare_lse(l_p[:, :1, rows].transpose(0, 1), want_l, "packed MHA LSE rows")
