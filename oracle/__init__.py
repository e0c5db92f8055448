"""CPU float64 oracle for fused exact attention (prefill and flash-decoding).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, constant or helper with the CUDA library under
``exact_attention_43_gb300/csrc``; the two meet only at the seeded inputs.

Every routine materialises what the definition materialises (the score row
S = scale * Q K^T, the two-pass softmax, P V) in numpy float64, so a reader can
check it against the pages by eye.  See ``oracle/attention.py``.

Pins (checked by ``tests/test_oracle.py``, ``-m "not gpu"``): rows of P sum to
one, single-key and constant-V closed forms, causal row 0, scale = 0 gives the
mean of V and ln|A|, permutation invariance, GQA == MHA with repeated KV heads,
decode == prefill with one query over the prefix, chunked merge == unchunked,
hand-worked examples in ``tests/golden/``, PyTorch's float64 math-path
``scaled_dot_product_attention`` and a pure-Python brute force on tiny shapes;
sliding windows against a brute force with explicit key sets, the diagonal
window's closed form and PyTorch SDPA on the explicit key slice; packed
variable-length batches against the batched definition (equal lengths) and
PyTorch SDPA per sequence; the backward against PyTorch float64 autograd,
central finite differences of the forward and a single-key closed form, its
sliding windows against autograd through SDPA with explicitly enumerated key
masks and finite differences, and packed batches against autograd per sequence.
No function here is "parity unpinned".
"""

from .attention import (  # noqa: F401
    sdpa,
    sdpa_backward,
    sdpa_backward_varlen,
    sdpa_varlen,
    softmax_probs,
    decode,
    decode_partials,
    merge_partials,
    decode_chunked,
    num_chunks,
)
