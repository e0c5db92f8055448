"""The binding refuses tensors that do not match the sizes it passes to the C ABI
(the library trusts them), before any launch."""

import pytest
import torch

from exact_attention_43_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_mismatched_tensors_raise_before_any_launch():
    import exact_attention_43_gb300 as ea

    q, k, v = wl.fwd_inputs(1, 4, 2, 256, 256, 64, seed=4500, device="cuda")
    with pytest.raises(ValueError):
        ea.attn_fwd(q, k, v, causal=True, out=torch.empty((1, 4, 128, 64), dtype=q.dtype,
                                                           device="cuda"))
    with pytest.raises(TypeError):
        ea.attn_fwd(q, k.float(), v, causal=True)
    with pytest.raises(ValueError):
        ea.attn_fwd(q.cpu(), k, v, causal=True)
    with pytest.raises(ValueError):
        ea.attn_fwd(q, k[:, :, :128], v, causal=True)                  # k and v disagree
    lens = torch.tensor([10], dtype=torch.int32, device="cuda")
    dq, dk, dv, _ = wl.decode_inputs(1, 4, 2, 64, 64, lens.cpu(), seed=4501, device="cuda")
    with pytest.raises(ValueError):
        ea.attn_decode(dq, dk, dv, lens.cpu())                          # lengths on the host
    with pytest.raises(ValueError):
        ea.attn_decode(dq, dk, dv, lens, out=torch.empty((1, 4, 32), dtype=dq.dtype, device="cuda"))
    o, lse = ea.attn_fwd(q, k, v, causal=True)
    with pytest.raises(ValueError):
        ea.attn_bwd(q, k, v, o, lse[:, :, :100].contiguous(), o, causal=True)
    torch.cuda.synchronize()
    assert ea.check_device_status() == 0
