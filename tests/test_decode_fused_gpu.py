"""Single-launch flash-decoding (attn_decode_fused): the last split CTA of each
(sequence, head group) merges the chunk partials.  Parity against the float64
oracle through the C ABI, and agreement with the two-kernel attn_decode."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import check_guards, compare_o, guarded

pytestmark = pytest.mark.gpu


def run_fused(q, k, v, lens, num_splits):
    import exact_attention_43_gb300 as ea

    o_full, o = guarded(tuple(q.shape), q.dtype)
    ea.attn_decode_fused(q.cuda(), k.cuda(), v.cuda(), lens.cuda(), num_splits=num_splits, out=o)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    check_guards(o_full)
    return o


CASES = [
    # B, Hq, Hkv, max_S, D, dtype, lens, num_splits
    (4, 8, 2, 1024, 128, torch.bfloat16, [1, 511, 512, 513], 2),
    (3, 4, 4, 2048, 128, torch.float16, [2048, 1, 1500], 0),       # G = 1: eight warps per head
    (2, 8, 1, 700, 64, torch.bfloat16, [700, 333], 7),             # G = 8: one warp per head
    (2, 16, 2, 600, 128, torch.bfloat16, [600, 64], 3),
    (2, 6, 2, 300, 64, torch.float16, [299, 5], 1),                # G = 3, one chunk
    (2, 4, 2, 4096, 128, torch.bfloat16, [4096, 4095], 64),
    (1, 2, 1, 97, 128, torch.bfloat16, [97], 97),                  # chunk of one key
    (3, 4, 2, 64, 128, torch.bfloat16, [0, 10, 0], 4),             # empty sequences: O = 0
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}x{}S{}D{}s{}".format(
    c[0], c[1], c[2], c[3], c[4], c[7]))
def test_fused_decode_cases(case):
    B, Hq, Hkv, max_S, D, dtype, lens, splits = case
    lens_t = torch.tensor(lens, dtype=torch.int32)
    q, k, v, lens_t = wl.decode_inputs(B, Hq, Hkv, max_S, D, lens_t, dtype=dtype,
                                       seed=2600 + max_S + D)
    o = run_fused(q, k, v, lens_t, splits)
    ref = oracle.decode(q, k, v, lens_t, scale=1 / np.sqrt(D))
    compare_o(o, ref, f"fused decode {case}")
    for b, L in enumerate(lens):
        if L == 0:
            assert bool((o[b] == 0).all())


def test_multi_chunk_ctas_and_repeated_calls():
    """CTAs of four chunks each (16 x 8 pairs, 64 chunks of 125 keys), ragged
    lengths; three calls in a row with different lengths and chunkings, so each
    call relies on the previous one having left every counter at zero."""
    lens = [8000, 7999, 125, 126, 250, 499, 500, 501, 0, 1, 3000, 4321, 6000, 7500, 375, 626]
    B, Hq, Hkv, max_S, D = len(lens), 32, 8, 8000, 128
    for i, (splits, lens_i) in enumerate([(64, lens), (16, lens[::-1]), (64, lens)]):
        lens_t = torch.tensor(lens_i, dtype=torch.int32)
        q, k, v, lens_t = wl.decode_inputs(B, Hq, Hkv, max_S, D, lens_t, seed=2700 + i)
        o = run_fused(q, k, v, lens_t, splits)
        ref = oracle.decode(q, k, v, lens_t, scale=1 / np.sqrt(D))
        compare_o(o, ref, f"fused decode, call {i}")


def test_out_of_range_length_is_clamped_and_reported():
    import exact_attention_43_gb300 as ea

    lens = torch.tensor([70, 64], dtype=torch.int32)       # 70 > max_S = 64
    q, k, v, _ = wl.decode_inputs(2, 2, 1, 64, 64, lens, seed=12)
    o = ea.attn_decode_fused(q.cuda(), k.cuda(), v.cuda(), lens.cuda(), num_splits=2)
    assert ea.check_device_status() == 1                   # ATTN_ERR_INVALID_ARG
    ref = oracle.decode(q, k, v, torch.tensor([64, 64], dtype=torch.int32), scale=0.125)
    compare_o(o, ref, "clamped")
    assert ea.check_device_status() == 0


def test_fused_decode_workload_full_size():
    """B64 Hq32 Hkv8 D128 bf16, lens U[512, 32768], 64 splits: every sequence against
    the oracle, and against the two-kernel path (same partials, merge order aside)."""
    import exact_attention_43_gb300 as ea

    w = wl.DECODE
    q, k, v, lens = wl.workload_decode_inputs(w, device="cuda")
    o = ea.attn_decode_fused(q, k, v, lens.cuda(), num_splits=w.num_splits)
    o2 = ea.attn_decode(q, k, v, lens.cuda(), num_splits=w.num_splits)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    got = o.double().cpu().numpy()
    assert np.isfinite(got).all()
    # both merges round the same fp32 sums to bf16: at most one bf16 ulp apart
    d = (o.float() - o2.float()).abs()
    ulp = o2.float().abs().clamp_min(2 ** -14) * 2 ** -7
    assert bool((d <= ulp).all()), float((d / ulp).max())
    qc = q.cpu()
    errs = []
    for b in range(w.B):
        L = int(lens[b])
        ref = oracle.decode(qc[b:b + 1], k[b:b + 1, :, :L].cpu(), v[b:b + 1, :, :L].cpu(),
                            torch.tensor([L]), scale=w.scale)
        errs.append(np.abs(got[b:b + 1] - ref))
    err = np.concatenate(errs)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
