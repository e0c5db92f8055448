"""Token-major backward (attn_bwd_varlen, attn_bwd_qkvpacked): packed sequences of
different lengths, sliding windows and a packed QKV projection, through the C ABI,
against the float64 oracle; equal-length packed projections against the dense
attn_bwd, bit for bit."""

import pytest
import torch

import oracle
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import CANARY16, check_guards, guarded
from tests.test_bwd_gpu import compare_grad

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

PAD_Q, PAD_K = 5, 7  # rows after the last sequence, in no sequence


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_bwd_varlen_cases(case):
    import exact_attention_43_gb300 as ea

    name, lq, lk, Hq, Hkv, D, dtype, causal, window = case
    lk = lq if lk is None else lk
    q, k, v, cu_q, cu_k = wl.varlen_inputs(lq, lk, Hq, Hkv, D, dtype=dtype, seed=3100 + len(name),
                                           pad_q=PAD_Q)
    extra = wl.normal((PAD_K, Hkv, D), seed=3200, dtype=dtype)
    k, v = torch.cat([k, extra]), torch.cat([v, extra])
    do = wl.normal(tuple(q.shape), seed=3300 + len(name), dtype=dtype)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    cq, ck = cu_q.cuda(), cu_k.cuda()
    scale = D ** -0.5
    o, lse = ea.attn_fwd_varlen(qc, kc, vc, cq, ck, max(lq), max(lk), causal=causal, window=window,
                                scale=scale)
    dq_f, dq = guarded(tuple(q.shape), dtype)
    dk_f, dk = guarded(tuple(k.shape), dtype)
    dv_f, dv = guarded(tuple(v.shape), dtype)
    ea.attn_bwd_varlen(qc, kc, vc, o, lse, doc, cq, ck, max(lq), max(lk), causal=causal,
                       window=window, scale=scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    for f in (dq_f, dk_f, dv_f):
        check_guards(f)
    nq, nk = int(cu_q[-1]), int(cu_k[-1])
    # rows of tokens outside every sequence are not written
    for t, n in ((dq, nq), (dk, nk), (dv, nk)):
        assert bool((t[n:].contiguous().view(torch.int16) == CANARY16).all()), f"{name}: row past the sequences"
    want = oracle.sdpa_backward_varlen(q[:nq], k[:nk], v[:nk], do[:nq], cu_q, cu_k, causal=causal,
                                       scale=scale, window_left=window[0], window_right=window[1])
    for gname, got, w in zip(("dQ", "dK", "dV"), (dq[:nq], dk[:nk], dv[:nk]), want):
        compare_grad(got, w, f"{name} {gname}")


def _packed(B, S, H, D, dtype, seed, device="cuda"):
    q, k, v = wl.fwd_inputs(B, H, H, S, S, D, dtype=dtype, seed=seed, device=device)
    qkv = torch.stack([x.transpose(1, 2) for x in (q, k, v)], dim=2).contiguous()  # [B, S, 3, H, D]
    return q, k, v, qkv


@pytest.mark.parametrize("S,causal,window", [(300, True, (-1, -1)), (1000, True, (128, -1)),
                                             (257, False, (-1, -1))])
def test_bwd_qkvpacked_against_oracle(S, causal, window):
    import exact_attention_43_gb300 as ea

    B, H, D = 2, 4, 128
    q, k, v, qkv = _packed(B, H=H, S=S, D=D, dtype=torch.bfloat16, seed=3400 + S)
    do = wl.normal((B, S, H, D), seed=3401, dtype=torch.bfloat16, device="cuda")
    o, lse = ea.attn_fwd_qkvpacked(qkv, causal=causal, window=window)
    full, dqkv = guarded(tuple(qkv.shape), qkv.dtype)
    ea.attn_bwd_qkvpacked(qkv, o, lse, do, causal=causal, window=window, dqkv=dqkv)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    check_guards(full)
    want = oracle.sdpa_backward(q.cpu(), k.cpu(), v.cpu(), do.transpose(1, 2).cpu(), causal=causal,
                                scale=D ** -0.5, window_left=window[0], window_right=window[1])
    for i, (gname, w) in enumerate(zip(("dQ", "dK", "dV"), want)):
        compare_grad(dqkv[:, :, i].transpose(1, 2), w, f"packed S{S} {gname}")


def test_bwd_mha_workload_packed_qkv_equals_dense():
    """The MHA workload (B4 H32 S2048 D128 causal) as one packed projection: the
    token-major backward reproduces the dense attn_bwd bit for bit."""
    import exact_attention_43_gb300 as ea

    w = wl.MHA
    q, k, v = wl.workload_fwd_inputs(w, device="cuda")
    qkv = torch.stack([x.transpose(1, 2) for x in (q, k, v)], dim=2).contiguous()
    do = wl.normal(tuple(q.shape), seed=3500, dtype=q.dtype, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    o_p, lse_p = ea.attn_fwd_qkvpacked(qkv, causal=True, scale=w.scale)
    dqkv = ea.attn_bwd_qkvpacked(qkv, o_p, lse_p, do.transpose(1, 2).contiguous(), causal=True,
                                 scale=w.scale)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    for i, ref in enumerate((dq, dk, dv)):
        got = dqkv[:, :, i].transpose(1, 2).contiguous()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), ("dQ", "dK", "dV")[i]
