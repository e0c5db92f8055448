"""Plain CPU float64 definition of exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Sources (page title, then the part of the page followed):

* abaddon 0.2.0-rc.2, ``src/cuda_inference/kernels/attention.rs`` -- module doc
  "Algorithm" (O = softmax(Q K^T / sqrt(d)) V, causal mask, final divide),
  kernel ``flash_attention_f16`` (GQA head mapping ``kv_head_id = head_id *
  kv_heads / heads``, layouts [batch, heads, seq, head_dim] and
  [batch, kv_heads, seq, head_dim]), ``FlashAttentionKernel::forward_cached``
  (decode against a cache, scale 1/sqrt(head_dim)).
* rustytorch ``flash_attention_forward.cu`` -- ``OnlineSoftmaxState``
  (``get_log_sum_exp`` = m + log(l), natural log, of the *scaled* scores) and
  ``flash_attention_forward_small_kernel`` (materialise the score row, apply
  the causal mask ``k_idx > q_idx -> -inf``, max pass, exp-sum pass, LSE,
  normalise, multiply by V).
* llm.c ``llmc/attention.cuh`` -- ``softmax_forward_kernel5`` (causal row
  softmax: only positions <= own_pos take part).
* aprender-gpu 0.32.0, ``kernels/attention/paged/flash_decoding/
  reduce_kernel.rs`` -- ``FlashDecodingReduceKernel``: partials laid out
  [M, num_heads, max_chunks, head_dim + 2] (o at [0, D), chunk max at D, chunk
  exp-sum at D + 1), ``num_chunks = ceil(seq_len / chunk_size)``, first pass =
  global max over chunks, second pass = sum of o_c * e^(m_c - M) and
  l_c * e^(m_c - M) skipping empty chunks, final normalisation by the sum.

Readings where the pages are silent (each also listed in the design doc):

* causal alignment for Sq != Skv is bottom-right: key j is visible to query i
  iff j <= i + (Skv - Sq); it equals the pages' j <= i when Sq == Skv;
* a row with no visible key has O = 0 and LSE = -inf; a decode sequence of
  length 0 has O = 0;
* the per-chunk partial o_c is unnormalised (sum of e^(s - m_c) v), the only
  reading under which the reduce's arithmetic gives the softmax;
* the chunk max m_c is in the natural-log units of the scaled scores.

Every array is converted to float64 first; no blocking, fusion or reordering
is applied beyond restricting the score matrix to the requested query rows.
"""

from __future__ import annotations

import math

import numpy as np


def _f64(x) -> np.ndarray:
    """Upcast any array-like (numpy, or a CPU torch tensor) to float64 numpy."""
    if hasattr(x, "detach"):  # torch tensor: bf16 has no numpy dtype
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _visible(rows: np.ndarray, Sq: int, Skv: int, causal: bool) -> np.ndarray:
    """Boolean [R, Skv] mask of the keys each query row may attend to.

    Causal mask as in rustytorch ``flash_attention_forward_small_kernel``
    (score set to -inf when the key position is after the query position),
    aligned bottom-right so that the last query sees every key.
    """
    j = np.arange(Skv)[None, :]
    if not causal:
        return np.ones((rows.shape[0], Skv), dtype=bool)
    return j <= (rows[:, None] + (Skv - Sq))


def softmax_probs(q, k, *, causal: bool, scale: float, rows=None):
    """Materialised attention probabilities P for one head.

    q: [Sq, D], k: [Skv, D].  Returns (P [R, Skv], m [R], l [R]) in float64,
    where m is the row max of the scaled, masked scores and l the sum of
    exp(s - m) -- the two passes of the small kernel in rustytorch
    ``flash_attention_forward.cu``.  An empty row has P = 0, m = -inf, l = 0.
    """
    q = _f64(q)
    k = _f64(k)
    Sq, Skv = q.shape[0], k.shape[0]
    rows = np.arange(Sq) if rows is None else np.asarray(rows, dtype=np.int64)
    s = scale * (q[rows] @ k.T)                      # score rows, materialised
    vis = _visible(rows, Sq, Skv, causal)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1) if Skv > 0 else np.full(rows.shape[0], -np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])                  # masked keys give exp(-inf) = 0
    l = e.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        p = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, l)[:, None])
    return p, np.where(empty, -np.inf, m), np.where(empty, 0.0, l)


def sdpa(q, k, v, *, causal: bool, scale: float, rows=None):
    """Exact attention O = softmax(scale Q K^T [+ causal mask]) V and its LSE.

    q: [B, Hq, Sq, D]; k, v: [B, Hkv, Skv, D] with Hq a multiple of Hkv.
    Query head h reads KV head h // (Hq / Hkv) (contiguous groups, as the GQA
    mapping in abaddon ``flash_attention_f16``).

    rows: None (every query row), a 1-D index array used for every head, or a
    2-D [Hq, R] array of per-head row indices.  Returns
    (O [B, Hq, R, D], LSE [B, Hq, R]) in float64; LSE = m + ln(l) in natural
    log of the scaled scores, -inf for a row with no visible key.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Skv, Dk = k.shape
    if Bk != B or Dk != D or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k and v")
    if Hkv == 0 or Hq % Hkv:
        raise ValueError("Hq must be a positive multiple of Hkv")
    group = Hq // Hkv
    if rows is None:
        rows_h = np.broadcast_to(np.arange(Sq), (Hq, Sq))
    else:
        rows = np.asarray(rows, dtype=np.int64)
        rows_h = np.broadcast_to(rows, (Hq, rows.shape[-1])) if rows.ndim == 1 else rows
    R = rows_h.shape[1]
    out = np.zeros((B, Hq, R, D))
    lse = np.full((B, Hq, R), -np.inf)
    for b in range(B):
        for h in range(Hq):
            kv = h // group
            p, m, l = softmax_probs(q[b, h], k[b, kv], causal=causal, scale=scale,
                                    rows=rows_h[h])
            out[b, h] = p @ v[b, kv]
            with np.errstate(divide="ignore"):
                lse[b, h] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return out, lse


def decode(q, k_cache, v_cache, seq_lens, *, scale: float):
    """Single-query attention of each sequence against its cache prefix.

    q: [B, Hq, D]; k_cache, v_cache: [B, Hkv, max_S, D]; seq_lens: [B] with
    0 <= L_b <= max_S.  For every (b, h): scores over keys [0, L_b) of KV head
    h // (Hq / Hkv), max pass, exp-sum pass, normalise, times V -- the role of
    abaddon ``flash_attention_cached_f16`` written as the plain definition.
    Returns O [B, Hq, D] float64 (zeros where L_b == 0).
    """
    q = _f64(q)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    group = Hq // Hkv
    lens = [int(x) for x in np.asarray(_f64(seq_lens)).reshape(-1)]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = lens[b]
        if L == 0:
            continue
        kb = _f64(k_cache[b, :, :L])
        vb = _f64(v_cache[b, :, :L])
        for h in range(Hq):
            kv = h // group
            s = scale * (kb[kv] @ q[b, h])           # [L]
            m = s.max()
            e = np.exp(s - m)
            out[b, h] = (e / e.sum()) @ vb[kv]
    return out


def num_chunks(seq_len: int, chunk: int) -> int:
    """ceil(seq_len / chunk), the per-sequence chunk count of the reduce kernel."""
    return (int(seq_len) + chunk - 1) // chunk


def decode_partials(q, k_cache, v_cache, seq_lens, *, chunk: int, scale: float,
                    max_chunks: int | None = None):
    """Per-chunk flash-decoding partials, laid out as the aprender-gpu reduce reads them.

    Returns partials [B, Hq, max_chunks, D + 2] float64 where, for every chunk
    c < ceil(L_b / chunk) covering keys [c*chunk, min((c+1)*chunk, L_b)):
    [..., :D] = o_c = sum_j exp(s_j - m_c) v_j (unnormalised), [..., D] = m_c =
    max_j s_j, [..., D + 1] = l_c = sum_j exp(s_j - m_c).  Entries of chunks
    past ceil(L_b / chunk) are left at o = 0, m = -inf, l = 0.
    """
    q = _f64(q)
    B, Hq, D = q.shape
    Hkv, max_S = k_cache.shape[1], k_cache.shape[2]
    group = Hq // Hkv
    lens = [int(x) for x in np.asarray(_f64(seq_lens)).reshape(-1)]
    if max_chunks is None:
        max_chunks = num_chunks(max_S, chunk)
    part = np.zeros((B, Hq, max_chunks, D + 2))
    part[..., D] = -np.inf
    for b in range(B):
        L = lens[b]
        if L == 0:
            continue
        kb = _f64(k_cache[b, :, :L])
        vb = _f64(v_cache[b, :, :L])
        for h in range(Hq):
            kv = h // group
            for c in range(num_chunks(L, chunk)):
                lo, hi = c * chunk, min((c + 1) * chunk, L)
                s = scale * (kb[kv, lo:hi] @ q[b, h])
                m_c = s.max()
                e = np.exp(s - m_c)
                part[b, h, c, :D] = e @ vb[kv, lo:hi]
                part[b, h, c, D] = m_c
                part[b, h, c, D + 1] = e.sum()
    return part


def merge_partials(partials, seq_lens, *, chunk: int):
    """LSE-rescaling merge of chunk partials (aprender-gpu ``FlashDecodingReduceKernel``).

    For every (b, h): num_chunks = ceil(L_b / chunk); first pass M = max_c m_c;
    second pass, skipping chunks whose m_c is not above -1e30 (empty),
    acc += o_c * exp(m_c - M) and sum += l_c * exp(m_c - M); O = acc / sum.
    A sequence with no chunk (L_b = 0) gets O = 0.  Returns O [B, Hq, D].
    """
    part = _f64(partials)
    B, Hq, _, D2 = part.shape
    D = D2 - 2
    lens = [int(x) for x in np.asarray(_f64(seq_lens)).reshape(-1)]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        n = num_chunks(lens[b], chunk)
        for h in range(Hq):
            if n == 0:
                continue
            M = -math.inf
            for c in range(n):                     # first pass: global max
                M = max(M, part[b, h, c, D])
            acc = np.zeros(D)
            total = 0.0
            for c in range(n):                     # second pass: rescaled sums
                m_c = part[b, h, c, D]
                if not m_c > -1e30:
                    continue
                w = math.exp(m_c - M)
                total += part[b, h, c, D + 1] * w
                acc += part[b, h, c, :D] * w
            out[b, h] = acc / total if total > 0 else 0.0
    return out


def decode_chunked(q, k_cache, v_cache, seq_lens, *, chunk: int, scale: float):
    """Flash-decoding as the pages split it: chunk partials, then the reduce."""
    part = decode_partials(q, k_cache, v_cache, seq_lens, chunk=chunk, scale=scale)
    return merge_partials(part, seq_lens, chunk=chunk)
