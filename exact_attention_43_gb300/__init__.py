"""Fused exact attention for one NVIDIA GB300 (sm_103a).

``attn_fwd`` (prefill, causal or not, grouped-query heads, per-row LSE) and
``attn_decode`` (flash-decoding: split-KV chunk partials merged by an
LSE-rescaling reduce) run in hand-written CUDA kernels behind the C ABI of
``include/attn.h``; this package is the thin PyTorch-facing binding.  Beside
them: ``attn_fwd_varlen`` (packed sequences of different lengths, sliding
windows), ``attn_fwd_qkvpacked`` (a [B, S, 3, H, D] projection read in place),
``attn_bwd`` (dQ, dK, dV) with ``attn_bwd_varlen`` and ``attn_bwd_qkvpacked``
for the token-major layouts, ``attn_decode_paged`` (a paged KV cache),
``attn_decode_fused`` (flash-decoding in one launch) and
``attn_decode_noalloc`` (no allocation during the call).
"""

from .binding import (  # noqa: F401
    AttnError,
    ExtensionMissing,
    attn_bwd,
    attn_bwd_qkvpacked,
    attn_bwd_varlen,
    attn_decode,
    attn_decode_fused,
    attn_decode_noalloc,
    attn_decode_paged,
    attn_fwd,
    attn_fwd_qkvpacked,
    attn_fwd_varlen,
    check_device_status,
    debug_set,
    decode_chunk,
    decode_workspace_bytes,
    load,
    status_string,
    version,
)
