"""The float64 oracle against its pins (CPU only)."""

import types

import pytest

import oracle
from tests import pins

IMPL = types.SimpleNamespace(
    sdpa=oracle.sdpa, sdpa_varlen=oracle.sdpa_varlen, sdpa_backward=oracle.sdpa_backward,
    sdpa_backward_varlen=oracle.sdpa_backward_varlen,
    softmax_probs=oracle.softmax_probs,
    decode=oracle.decode,
    decode_partials=oracle.decode_partials, merge_partials=oracle.merge_partials)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(IMPL)


def test_decode_chunked_wrapper_matches_decode():
    import numpy as np
    rng = np.random.default_rng(5)
    q = rng.normal(size=(2, 4, 8))
    k = rng.normal(size=(2, 1, 30, 8))
    v = rng.normal(size=(2, 1, 30, 8))
    lens = np.array([30, 7])
    a = oracle.decode(q, k, v, lens, scale=0.5)
    b = oracle.decode_chunked(q, k, v, lens, chunk=4, scale=0.5)
    assert np.max(np.abs(a - b)) < 1e-12


def test_oracle_accepts_low_precision_torch_tensors():
    import torch
    q = torch.randn(1, 2, 5, 8).to(torch.bfloat16)
    k = torch.randn(1, 1, 5, 8).to(torch.bfloat16)
    v = torch.randn(1, 1, 5, 8).to(torch.bfloat16)
    o, lse = oracle.sdpa(q, k, v, causal=True, scale=0.3)
    o2, lse2 = oracle.sdpa(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                           causal=True, scale=0.3)
    assert (o == o2).all() and (lse == lse2).all()
