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
* llm.c ``llmc/attention.cuh`` -- ``attention_backward`` and
  ``softmax_autoregressive_backward_inplace_kernel``: datt = dout V^T,
  dv = att^T dout, dpreatt = scale * att * (datt - sum_j att * datt) per row,
  dq = dpreatt K, dk = dpreatt^T Q.
* aprender-gpu 0.32.0, ``kernels/attention/paged/flash_decoding/
  reduce_kernel.rs`` -- ``FlashDecodingReduceKernel``: partials laid out
  [M, num_heads, max_chunks, head_dim + 2] (o at [0, D), chunk max at D, chunk
  exp-sum at D + 1), ``num_chunks = ceil(seq_len / chunk_size)``, first pass =
  global max over chunks, second pass = sum of o_c * e^(m_c - M) and
  l_c * e^(m_c - M) skipping empty chunks, final normalisation by the sum.

Readings where the pages are silent:

* causal alignment for Sq != Skv is bottom-right: key j is visible to query i
  iff j <= i + (Skv - Sq); it equals the pages' j <= i when Sq == Skv;
* a row with no visible key has O = 0 and LSE = -inf; a decode sequence of
  length 0 has O = 0;
* the per-chunk partial o_c is unnormalised (sum of e^(s - m_c) v), the only
  reading under which the reduce's arithmetic gives the softmax;
* the chunk max m_c is in the natural-log units of the scaled scores;
* local (sliding-window) attention, which the flash-attention backward page
  names only as an ``Is_local`` switch, keeps key j for query i iff
  i + d - window_left <= j <= i + d + window_right with d = Skv - Sq (the
  same bottom-right alignment as the causal mask); a bound of -1 is absent,
  and causal is the right bound 0;
* with grouped-query heads, the gradient of a shared K or V head is the sum
  over the query heads that read it (llm.c has one KV head per query head);
* variable-length batches (the same page's ``Varlen`` switch) are packed:
  sequence b owns query rows [cu_q[b], cu_q[b+1]) of a [total_q, H, D] array
  and key rows [cu_k[b], cu_k[b+1]) of [total_k, Hkv, D]; each sequence is
  attended on its own, and its LSE goes to an [H, total_q] array.

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


def _visible(rows: np.ndarray, Sq: int, Skv: int, causal: bool, window_left: int = -1,
             window_right: int = -1) -> np.ndarray:
    """Boolean [R, Skv] mask of the keys each query row may attend to.

    Causal mask as in rustytorch ``flash_attention_forward_small_kernel``
    (score set to -inf when the key position is after the query position),
    aligned bottom-right so that the last query sees every key.  A window
    bound w >= 0 keeps only keys within w positions of the row's diagonal
    key on that side.
    """
    j = np.arange(Skv)[None, :]
    diag = rows[:, None] + (Skv - Sq)               # the row's diagonal key
    keep = np.ones((rows.shape[0], Skv), dtype=bool)
    if causal:
        keep &= j <= diag
    if window_right >= 0:
        keep &= j <= diag + window_right
    if window_left >= 0:
        keep &= j >= diag - window_left
    return keep


def softmax_probs(q, k, *, causal: bool, scale: float, rows=None, window_left: int = -1,
                  window_right: int = -1):
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
    if window_left == -1 and window_right == -1:
        vis = _visible(rows, Sq, Skv, causal)
    else:
        vis = _visible(rows, Sq, Skv, causal, window_left, window_right)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1) if Skv > 0 else np.full(rows.shape[0], -np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])                  # masked keys give exp(-inf) = 0
    l = e.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        p = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, l)[:, None])
    return p, np.where(empty, -np.inf, m), np.where(empty, 0.0, l)


def sdpa(q, k, v, *, causal: bool, scale: float, rows=None, window_left: int = -1,
         window_right: int = -1):
    """Exact attention O = softmax(scale Q K^T [+ causal mask]) V and its LSE.

    q: [B, Hq, Sq, D]; k, v: [B, Hkv, Skv, D] with Hq a multiple of Hkv.
    Query head h reads KV head h // (Hq / Hkv) (contiguous groups, as the GQA
    mapping in abaddon ``flash_attention_f16``).

    rows: None (every query row), a 1-D index array used for every head, or a
    2-D [Hq, R] array of per-head row indices.  window_left / window_right:
    sliding-window bounds (-1: none), see ``_visible``.  Returns
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
                                    rows=rows_h[h], window_left=window_left,
                                    window_right=window_right)
            out[b, h] = p @ v[b, kv]
            with np.errstate(divide="ignore"):
                lse[b, h] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return out, lse


def sdpa_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, *, causal: bool, scale: float,
                window_left: int = -1, window_right: int = -1):
    """Attention over a packed batch of sequences of different lengths.

    q: [total_q, Hq, D]; k, v: [total_k, Hkv, D]; cu_seqlens_q, cu_seqlens_k:
    [B + 1] non-decreasing offsets.  Sequence b is the plain ``sdpa`` of its
    own rows (query rows cu_q[b]..cu_q[b+1]-1, key rows cu_k[b]..cu_k[b+1]-1),
    with its own bottom-right causal / window alignment.  Returns
    (O [total_q, Hq, D], LSE [Hq, total_q]) float64; rows outside every
    sequence are 0 in O and -inf in LSE.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    cq = [int(x) for x in np.asarray(_f64(cu_seqlens_q)).reshape(-1)]
    ck = [int(x) for x in np.asarray(_f64(cu_seqlens_k)).reshape(-1)]
    if len(cq) != len(ck):
        raise ValueError("cu_seqlens_q and cu_seqlens_k need the same length")
    total_q, Hq, D = q.shape
    out = np.zeros((total_q, Hq, D))
    lse = np.full((Hq, total_q), -np.inf)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 <= q0:
            continue
        qb = q[q0:q1].transpose(1, 0, 2)[None]       # [1, Hq, Sq_b, D]
        kb = k[k0:k1].transpose(1, 0, 2)[None]
        vb = v[k0:k1].transpose(1, 0, 2)[None]
        ob, lb = sdpa(qb, kb, vb, causal=causal, scale=scale, window_left=window_left,
                      window_right=window_right)
        out[q0:q1] = ob[0].transpose(1, 0, 2)
        lse[:, q0:q1] = lb[0]
    return out, lse


def sdpa_backward(q, k, v, dout, *, causal: bool, scale: float, window_left: int = -1,
                  window_right: int = -1):
    """Gradients of O = sdpa(q, k, v) for an incoming dO, as the llm.c page's
    ``attention_backward`` computes them for each (batch, query head):

    datt = dO V^T; dV += att^T dO; local = sum_j att * datt (per row);
    dpreatt = scale * att * (datt - local); dQ = dpreatt K; dK += dpreatt^T Q,

    att being the materialised probabilities (bottom-right causal mask and the
    sliding-window bounds of ``sdpa``).  Shapes as ``sdpa``; dout [B, Hq, Sq, D].
    Returns (dQ, dK, dV) in float64, dK and dV summed over the query heads of
    each KV head.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    do = _f64(dout)
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            kv = h // group
            att, _, _ = softmax_probs(q[b, h], k[b, kv], causal=causal, scale=scale,
                                      window_left=window_left, window_right=window_right)
            datt = do[b, h] @ v[b, kv].T                    # [Sq, Skv]
            dv[b, kv] += att.T @ do[b, h]
            local = (att * datt).sum(axis=1, keepdims=True)
            dpre = scale * att * (datt - local)
            dq[b, h] = dpre @ k[b, kv]
            dk[b, kv] += dpre.T @ q[b, h]
    return dq, dk, dv


def sdpa_backward_varlen(q, k, v, dout, cu_seqlens_q, cu_seqlens_k, *, causal: bool,
                         scale: float, window_left: int = -1, window_right: int = -1):
    """Gradients of ``sdpa_varlen`` for an incoming dO: each packed sequence is the
    plain ``sdpa_backward`` of its own rows (layouts of ``sdpa_varlen``; dout like
    q).  Returns (dQ [total_q, Hq, D], dK, dV [total_k, Hkv, D]) float64; rows
    outside every sequence get zero gradients.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    do = _f64(dout)
    cq = [int(x) for x in np.asarray(_f64(cu_seqlens_q)).reshape(-1)]
    ck = [int(x) for x in np.asarray(_f64(cu_seqlens_k)).reshape(-1)]
    if len(cq) != len(ck):
        raise ValueError("cu_seqlens_q and cu_seqlens_k need the same length")
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 <= q0 or k1 <= k0:
            continue                                  # no query, or no key: zero gradients
        t = lambda x, a, e: x[a:e].transpose(1, 0, 2)[None]   # [1, H, S_b, D]
        g = sdpa_backward(t(q, q0, q1), t(k, k0, k1), t(v, k0, k1), t(do, q0, q1), causal=causal,
                          scale=scale, window_left=window_left, window_right=window_right)
        dq[q0:q1] = g[0][0].transpose(1, 0, 2)
        dk[k0:k1] = g[1][0].transpose(1, 0, 2)
        dv[k0:k1] = g[2][0].transpose(1, 0, 2)
    return dq, dk, dv


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
