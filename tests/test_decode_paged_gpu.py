"""Flash-decoding over a paged KV cache: the CUDA path (through the C ABI)
against the float64 oracle on the same keys and values laid out contiguously,
and bit for bit against the contiguous-cache kernel at full size."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import check_guards, compare_o, guarded

pytestmark = pytest.mark.gpu


def run_paged(q, kp, vp, table, lens, num_splits):
    import exact_attention_43_gb300 as ea

    o_full, o = guarded(tuple(q.shape), q.dtype)
    ea.attn_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens.cuda(),
                         num_splits=num_splits, out=o)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    check_guards(o_full)
    return o


CASES = [
    # B, Hq, Hkv, max_S, D, dtype, lens, page_size, num_splits
    (4, 8, 2, 1024, 128, torch.bfloat16, [1, 511, 512, 513], 16, 2),
    (3, 16, 2, 700, 128, torch.bfloat16, [700, 0, 333], 100, 3),   # G = 8, pages not a power of two
    (2, 4, 4, 2048, 64, torch.float16, [2048, 1500], 128, 0),
    (2, 8, 1, 1000, 128, torch.bfloat16, [1000, 257], 256, 7),     # pages larger than a chunk
    (3, 8, 2, 300, 64, torch.bfloat16, [300, 17, 16], 1, 4),       # one position per page
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}x{}S{}D{}p{}s{}".format(
    c[0], c[1], c[2], c[3], c[4], c[7], c[8]))
def test_paged_decode_cases(case):
    B, Hq, Hkv, max_S, D, dtype, lens, page, splits = case
    lens_t = torch.tensor(lens, dtype=torch.int32)
    q, k, v, lens_t = wl.decode_inputs(B, Hq, Hkv, max_S, D, lens_t, dtype=dtype,
                                       seed=3000 + max_S + page)
    kp, vp, table = wl.paged_cache(k, v, lens, page, seed=3100 + page)
    o = run_paged(q, kp, vp, table, lens_t, splits)
    ref = oracle.decode(q, k, v, lens_t, scale=1 / np.sqrt(D))
    compare_o(o, ref, f"paged decode {case}")


@pytest.mark.parametrize("page", [16, 64])
def test_paged_equals_contiguous_at_full_size(page):
    """The decode workload (B64 Hq32 Hkv8 D128, lens U[512, 32768], 64 splits) with
    16- and 64-position pages (copies issued by warp 0's lanes, or by one thread)
    gives exactly the contiguous kernel's output: the same keys in the same
    sub-tiles, only fetched from other addresses."""
    import exact_attention_43_gb300 as ea

    w = wl.DECODE
    q, k, v, lens = wl.workload_decode_inputs(w, device="cuda")
    kp, vp, table = wl.paged_cache(k, v, [int(x) for x in lens], page, seed=3200)
    ref = ea.attn_decode(q, k, v, lens.cuda(), num_splits=w.num_splits)
    del k, v
    got = ea.attn_decode_paged(q, kp.cuda(), vp.cuda(), table.cuda(), lens.cuda(),
                               num_splits=w.num_splits)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
    assert torch.equal(got, ref)


@pytest.mark.parametrize("page", [16, 64])
def test_block_table_entry_outside_the_pool_is_reported(page):
    import exact_attention_43_gb300 as ea

    lens = [200, 100]
    q, k, v, lens_t = wl.decode_inputs(2, 8, 2, 256, 128, torch.tensor(lens, dtype=torch.int32),
                                       seed=3300)
    kp, vp, table = wl.paged_cache(k, v, lens, page, seed=3301)
    table[1, 0] = kp.shape[0] + 5  # past the pool: the kernel reads page 0 instead
    o = ea.attn_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), lens_t.cuda())
    torch.cuda.synchronize()
    assert ea.check_device_status() == 1  # ATTN_ERR_INVALID_ARG
    assert ea.check_device_status() == 0  # reading the status clears it
    assert bool(torch.isfinite(o.float()).all())
