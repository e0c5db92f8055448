"""Bounded device waits: a withheld copy makes a kernel's waits run out; the
kernel unwinds (drains its copies and MMAs, frees TMEM), the host reads
ATTN_ERR_DEVICE_TIMEOUT, and the CUDA context stays usable.  Each case is
followed by the same call without the fault, which must be correct: for the
single-launch decode this also shows that the CTA which gave up still took its
merge ticket, leaving the counters at zero for the next call."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import compare_o
from tests.test_bwd_gpu import compare_grad

pytestmark = pytest.mark.gpu

LIMIT_US = 20000  # 20 ms per wait


def _with_fault(ea, fault, call):
    """Run `call` with the debug fault set; return the device status it left."""
    assert ea.check_device_status() == 0
    assert ea.debug_set(fault, LIMIT_US) == 0
    try:
        call()
        return ea.check_device_status()
    finally:
        ea.debug_set(0, 0)


def test_withheld_tile_reports_timeout_and_context_survives():
    import exact_attention_43_gb300 as ea

    q, k, v = wl.fwd_inputs(1, 2, 2, 256, 256, 64, dtype=torch.float16, seed=21, device="cuda")
    st = _with_fault(ea, 1, lambda: ea.attn_fwd(q, k, v, causal=True))
    assert st == ea.binding.ATTN_ERR_DEVICE_TIMEOUT
    # the same call now completes and is correct
    o, lse = ea.attn_fwd(q, k, v, causal=True)
    assert ea.check_device_status() == 0
    ro, _ = oracle.sdpa(q.cpu(), k.cpu(), v.cpu(), causal=True, scale=0.125)
    compare_o(o, ro, "after timeout")
    assert np.isfinite(lse.cpu().numpy()).all()


@pytest.mark.parametrize("entry", ["attn_decode", "attn_decode_fused"])
def test_decode_withheld_subtile_reports_timeout(entry):
    import exact_attention_43_gb300 as ea

    lens = torch.tensor([700, 300, 1, 1024, 0, 513], dtype=torch.int32)
    q, k, v, lens = wl.decode_inputs(6, 8, 2, 1024, 128, lens, seed=23, device="cuda")
    lens_d = lens.cuda()
    fn = getattr(ea, entry)
    st = _with_fault(ea, 2, lambda: fn(q, k, v, lens_d, num_splits=4))
    assert st == ea.binding.ATTN_ERR_DEVICE_TIMEOUT
    for _ in range(2):  # twice: the merge counters must be back at zero each time
        out = fn(q, k, v, lens_d, num_splits=4)
        assert ea.check_device_status() == 0
        ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), lens, scale=1.0 / 128 ** 0.5)
        compare_o(out, ref, f"{entry} after timeout")


def test_bwd_withheld_tile_reports_timeout():
    import exact_attention_43_gb300 as ea

    q, k, v = wl.fwd_inputs(1, 2, 2, 512, 512, 64, dtype=torch.float16, seed=24, device="cuda")
    do = wl.normal((1, 2, 512, 64), seed=25, dtype=torch.float16, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=True)
    st = _with_fault(ea, 3, lambda: ea.attn_bwd(q, k, v, o, lse, do, causal=True))
    assert st == ea.binding.ATTN_ERR_DEVICE_TIMEOUT
    dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, do, causal=True)
    assert ea.check_device_status() == 0
    want = oracle.sdpa_backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), causal=True, scale=0.125)
    for name, got, w in zip(("dQ", "dK", "dV"), (dq, dk, dv), want):
        compare_grad(got, w, f"{name} after timeout")

