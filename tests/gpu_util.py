"""Helpers for the GPU parity tests: tolerances, canary-guarded outputs."""

from __future__ import annotations

import numpy as np
import torch

# fp32-accumulating kernels on 16-bit inputs against the float64 oracle
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3

GUARD = 64  # elements of canary on each side of an output (128 bytes for 16-bit types)
CANARY16 = 0x7FDA  # a NaN pattern in both fp16 and bf16
CANARY32 = 0x7FC0DEAD  # a float32 NaN pattern


def guarded(shape, dtype, device="cuda"):
    """Output buffer surrounded by canaries and pre-filled with NaN.

    Returns (full, view): view is the 16-byte aligned interior of `shape`.
    """
    n = int(np.prod(shape))
    if dtype in (torch.float16, torch.bfloat16):
        full = torch.full((n + 2 * GUARD,), CANARY16, dtype=torch.int16, device=device)
        view = full[GUARD:GUARD + n].view(dtype).view(shape)
    else:
        full = torch.full((n + 2 * GUARD,), CANARY32, dtype=torch.int32, device=device)
        view = full[GUARD:GUARD + n].view(torch.float32).view(shape)
    return full, view


def check_guards(full):
    pat = CANARY16 if full.dtype == torch.int16 else CANARY32
    head = full[:GUARD]
    tail = full[-GUARD:]
    assert bool((head == pat).all()), "write before the output buffer"
    assert bool((tail == pat).all()), "write after the output buffer"


def compare_o(got, want, what=""):
    """got: torch tensor (any device), want: float64 numpy of the same shape."""
    g = got.detach().double().cpu().numpy()
    assert g.shape == want.shape, f"{what}: shape {g.shape} vs {want.shape}"
    assert np.isfinite(g).all(), f"{what}: non-finite output (unwritten or NaN)"
    err = np.abs(g - want)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= O_MAX_ABS, f"{what}: O max abs err {mx:.3e} > {O_MAX_ABS}"
    assert mean <= O_MEAN_ABS, f"{what}: O mean abs err {mean:.3e} > {O_MEAN_ABS}"
    return mx, mean


def compare_lse(got, want, what=""):
    g = got.detach().double().cpu().numpy()
    assert g.shape == want.shape
    ninf_g, ninf_w = np.isneginf(g), np.isneginf(want)
    assert (ninf_g == ninf_w).all(), f"{what}: -inf LSE pattern differs"
    fin = ~ninf_w
    assert np.isfinite(g[fin]).all(), f"{what}: non-finite LSE"
    err = np.abs(g[fin] - want[fin])
    mx = float(err.max()) if err.size else 0.0
    assert mx <= LSE_ABS, f"{what}: LSE max abs err {mx:.3e} > {LSE_ABS}"
    return mx
