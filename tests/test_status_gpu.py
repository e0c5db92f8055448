"""Bounded device waits: a withheld tile makes the prefill kernel's waits run
out; the kernel unwinds (drains its copies and MMAs, frees TMEM), the host
reads ATTN_ERR_DEVICE_TIMEOUT, and the CUDA context stays usable."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_43_gb300 import workloads as wl
from tests.gpu_util import compare_o

pytestmark = pytest.mark.gpu


def test_withheld_tile_reports_timeout_and_context_survives():
    import exact_attention_43_gb300 as ea

    q, k, v = wl.fwd_inputs(1, 2, 2, 256, 256, 64, dtype=torch.float16, seed=21, device="cuda")
    assert ea.check_device_status() == 0
    assert ea.debug_set(1, 20000) == 0  # withhold the first V tile; 20 ms wait limit
    try:
        ea.attn_fwd(q, k, v, causal=True)
        assert ea.check_device_status() == ea.binding.ATTN_ERR_DEVICE_TIMEOUT
    finally:
        ea.debug_set(0, 0)
    # the same call now completes and is correct
    o, lse = ea.attn_fwd(q, k, v, causal=True)
    assert ea.check_device_status() == 0
    ro, _ = oracle.sdpa(q.cpu(), k.cpu(), v.cpu(), causal=True, scale=0.125)
    compare_o(o, ro, "after timeout")
    assert np.isfinite(lse.cpu().numpy()).all()
