"""attn_decode_noalloc, the decode entry point for callers that may not
allocate GPU memory during a call (a plugin whose host owns the whole device
memory budget, a serving loop that must not wait on or fail in an allocator).

Its chunk partials live in a fixed device array that every call reuses, so
the test makes two calls in a row through the C ABI -- a large problem, then a
smaller one that leaves stale partials of the first in the array -- and checks
each against attn_decode, which allocates its partials per call.  Both run the
same split and reduce kernels over the same chunking, so their outputs must be
identical bit for bit (a stale partial read back would change them); each is
also checked against the float64 oracle at the decode tolerance.  This file
runs last so that a failure here cannot hide the other GPU tests; it needs no
state from them.
"""

import pytest
import torch

import oracle
from exact_attention_43_gb300 import binding
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import compare_o

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, lens, out, num_splits):
    B, Hq, D = q.shape
    Hkv, max_S = k.shape[1], k.shape[2]
    return lib.attn_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), lens.data_ptr(),
                                   out.data_ptr(), B, Hq, Hkv, max_S, D, num_splits,
                                   binding.ATTN_BF16, torch.cuda.current_stream().cuda_stream)


def test_two_calls_in_a_row_match_the_allocating_entry_point():
    lib = binding.load()
    cases = [
        # lens, max_S, num_splits: 8 x 32 x 64 chunks x 130 floats = 8.5 MB of partials
        ([32768, 512, 20000, 1, 4097, 32000, 777, 16384], 32768, 64),
        # then a smaller problem over the same scratch
        ([4096, 1, 0, 2500], 4096, 8),
    ]
    for n, (lens, max_S, splits) in enumerate(cases):
        B = len(lens)
        assert binding.decode_workspace_bytes(B, 32, max_S, 128, splits) <= binding.NOALLOC_MAX_BYTES
        q, k, v, lens_t = wl.decode_inputs(B, 32, 8, max_S, 128, torch.tensor(lens, dtype=torch.int32),
                                           seed=4000 + n, device="cuda")
        lens_d = lens_t.cuda()
        ref = binding.attn_decode(q, k, v, lens_d, num_splits=splits)
        out = torch.full_like(q, float("nan"))
        assert _noalloc(lib, q, k, v, lens_d, out, splits) == binding.ATTN_OK
        torch.cuda.synchronize()
        assert binding.check_device_status() == binding.ATTN_OK
        assert bool(torch.isfinite(out.float()).all()), f"call {n}: unwritten or non-finite output"
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            f"call {n}: differs from attn_decode"
        want = oracle.decode(q.cpu(), k.cpu(), v.cpu(), lens_t, scale=1.0 / 128 ** 0.5)
        compare_o(out, want, f"call {n} against the oracle")


def test_oversized_problem_is_refused():
    lib = binding.load()
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((64, 8, 64, 128), dtype=torch.bfloat16, device="cuda")
    lens = torch.full((64,), 64, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    # 64 sequences x 32 heads x 64 one-key chunks x 130 floats x 4 B = 68 MB > 16 MiB
    assert _noalloc(lib, q, k, k, lens, out, 64) == binding.ATTN_ERR_UNSUPPORTED
    assert bool((out == 0).all())
