"""Flash-decoding parity: the CUDA path (through the C ABI) against the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import check_guards, compare_o, guarded

pytestmark = pytest.mark.gpu


def run_decode(q, k, v, lens, num_splits):
    import exact_attention_43_gb300 as ea

    o_full, o = guarded(tuple(q.shape), q.dtype)
    ea.attn_decode(q.cuda(), k.cuda(), v.cuda(), lens.cuda(), num_splits=num_splits, out=o)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    check_guards(o_full)
    return o


CASES = [
    # B, Hq, Hkv, max_S, D, dtype, lens, num_splits
    (4, 8, 2, 1024, 128, torch.bfloat16, [1, 511, 512, 513], 2),
    (3, 4, 4, 2048, 128, torch.float16, [2048, 1, 1500], 0),
    (2, 8, 1, 700, 64, torch.bfloat16, [700, 333], 7),
    (2, 16, 2, 600, 128, torch.bfloat16, [600, 64], 3),      # G = 8
    (2, 6, 2, 300, 64, torch.float16, [299, 5], 1),          # G = 3, one chunk
    (2, 4, 2, 4096, 128, torch.bfloat16, [4096, 4095], 64),
    (1, 2, 1, 97, 128, torch.bfloat16, [97], 97),            # chunk of one key
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}x{}S{}D{}s{}".format(
    c[0], c[1], c[2], c[3], c[4], c[7]))
def test_decode_cases(case):
    B, Hq, Hkv, max_S, D, dtype, lens, splits = case
    lens_t = torch.tensor(lens, dtype=torch.int32)
    q, k, v, lens_t = wl.decode_inputs(B, Hq, Hkv, max_S, D, lens_t, dtype=dtype,
                                       seed=2000 + max_S + D)
    o = run_decode(q, k, v, lens_t, splits)
    ref = oracle.decode(q, k, v, lens_t, scale=1 / np.sqrt(D))
    compare_o(o, ref, f"decode {case}")
    chunk = -(-max_S // splits) if splits else 512
    ref_c = oracle.decode_chunked(q, k, v, lens_t, chunk=chunk, scale=1 / np.sqrt(D))
    assert np.max(np.abs(ref - ref_c)) < 1e-12


def test_multi_chunk_ctas():
    """Enough (sequence, KV head) pairs that a CTA takes four consecutive chunks
    (on a 152-SM part: 16 x 8 pairs, 64 chunks of 125 keys), with lengths that end
    inside a CTA's range, on a chunk boundary, at zero and at one key; 125 is not
    a multiple of the 128-key sub-tile."""
    lens = [8000, 7999, 125, 126, 250, 499, 500, 501, 0, 1, 3000, 4321, 6000, 7500, 375, 626]
    B, Hq, Hkv, max_S, D = len(lens), 32, 8, 8000, 128
    lens_t = torch.tensor(lens, dtype=torch.int32)
    q, k, v, lens_t = wl.decode_inputs(B, Hq, Hkv, max_S, D, lens_t, seed=2500)
    o = run_decode(q, k, v, lens_t, 64)
    ref = oracle.decode(q, k, v, lens_t, scale=1 / np.sqrt(D))
    compare_o(o, ref, "decode multi-chunk CTAs")


def test_zero_length_sequences():
    lens = torch.tensor([0, 10, 0], dtype=torch.int32)
    q, k, v, lens = wl.decode_inputs(3, 4, 2, 64, 128, lens, seed=11)
    o = run_decode(q, k, v, lens, 4)
    assert bool((o[0] == 0).all()) and bool((o[2] == 0).all())
    compare_o(o[1:2], oracle.decode(q[1:2], k[1:2], v[1:2], lens[1:2], scale=128 ** -0.5))


def test_out_of_range_length_is_clamped_and_reported():
    import exact_attention_43_gb300 as ea

    lens = torch.tensor([70, 64], dtype=torch.int32)       # 70 > max_S = 64
    q, k, v, _ = wl.decode_inputs(2, 2, 1, 64, 64, lens, seed=12)
    o = ea.attn_decode(q.cuda(), k.cuda(), v.cuda(), lens.cuda(), num_splits=2)
    assert ea.check_device_status() == 1                   # ATTN_ERR_INVALID_ARG
    ref = oracle.decode(q, k, v, torch.tensor([64, 64], dtype=torch.int32), scale=0.125)
    compare_o(o, ref, "clamped")
    assert ea.check_device_status() == 0                   # status was cleared


def test_deterministic():
    import exact_attention_43_gb300 as ea

    lens = torch.tensor([3000, 17, 4096, 2048], dtype=torch.int32)
    q, k, v, lens = wl.decode_inputs(4, 32, 8, 4096, 128, lens, seed=13, device="cuda")
    a = ea.attn_decode(q, k, v, lens.cuda(), num_splits=8)
    b = ea.attn_decode(q, k, v, lens.cuda(), num_splits=8)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_decode_workload_full_size():
    """B64 Hq32 Hkv8 D128 bf16, cache [64, 8, 32768, 128], lens U[512, 32768], 64 splits."""
    import exact_attention_43_gb300 as ea

    w = wl.DECODE
    q, k, v, lens = wl.workload_decode_inputs(w, device="cuda")
    o = ea.attn_decode(q, k, v, lens.cuda(), num_splits=w.num_splits)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    got = o.double().cpu().numpy()
    assert np.isfinite(got).all()
    qc = q.cpu()
    errs = []
    for b in range(w.B):  # every sequence, against its full prefix (copied one sequence at a time)
        L = int(lens[b])
        ref = oracle.decode(qc[b:b + 1], k[b:b + 1, :, :L].cpu(), v[b:b + 1, :, :L].cpu(),
                            torch.tensor([L]), scale=w.scale)
        errs.append(np.abs(got[b:b + 1] - ref))
    err = np.concatenate(errs)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
