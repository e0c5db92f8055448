"""Plant one plausible mistake at a time in the oracle (on the CPU) and check
that the pins catch it.  A pin set that let a mutant through would not be
pinning the oracle to anything."""

import math
import types

import numpy as np
import pytest

import oracle
from oracle import attention as A
from tests import pins

BASE = dict(sdpa=oracle.sdpa, sdpa_varlen=oracle.sdpa_varlen, sdpa_backward=oracle.sdpa_backward,
    sdpa_backward_varlen=oracle.sdpa_backward_varlen,
            softmax_probs=oracle.softmax_probs,
            decode=oracle.decode, decode_partials=oracle.decode_partials,
            merge_partials=oracle.merge_partials)


def _impl(**over):
    d = dict(BASE)
    d.update(over)
    return types.SimpleNamespace(**d)


def _with_visible(fn):
    """Run the oracle with a mutated causal visibility rule."""
    def sdpa(q, k, v, *, causal, scale, rows=None, **kw):
        saved = A._visible
        A._visible = fn
        try:
            return oracle.sdpa(q, k, v, causal=causal, scale=scale, rows=rows, **kw)
        finally:
            A._visible = saved

    def probs(q, k, *, causal, scale, rows=None, **kw):
        saved = A._visible
        A._visible = fn
        try:
            return oracle.softmax_probs(q, k, causal=causal, scale=scale, rows=rows, **kw)
        finally:
            A._visible = saved

    def varlen(*a, **kw):
        saved = A._visible
        A._visible = fn
        try:
            return oracle.sdpa_varlen(*a, **kw)
        finally:
            A._visible = saved
    return dict(sdpa=sdpa, softmax_probs=probs, sdpa_varlen=varlen)


def _windowed(causal_rule):
    """A visibility rule with the given causal test and the real window bounds."""
    def rule(rows, Sq, Skv, causal, window_left=-1, window_right=-1):
        j = np.arange(Skv)[None, :]
        diag = rows[:, None] + (Skv - Sq)
        keep = causal_rule(j, rows[:, None], diag) if causal else np.ones((rows.shape[0], Skv), bool)
        if window_right >= 0:
            keep = keep & (j <= diag + window_right)
        if window_left >= 0:
            keep = keep & (j >= diag - window_left)
        return keep
    return rule


_strict = _windowed(lambda j, i, diag: j < diag)
_top_left = _windowed(lambda j, i, diag: j <= i)


def _window_left_strict(rows, Sq, Skv, causal, window_left=-1, window_right=-1):
    j = np.arange(Skv)[None, :]
    diag = rows[:, None] + (Skv - Sq)
    keep = (j <= diag) if causal else np.ones((rows.shape[0], Skv), bool)
    if window_right >= 0:
        keep = keep & (j <= diag + window_right)
    if window_left >= 0:
        keep = keep & (j > diag - window_left)     # mistake: drops the key at the bound
    return keep


def _window_top_left(rows, Sq, Skv, causal, window_left=-1, window_right=-1):
    j = np.arange(Skv)[None, :]
    diag = rows[:, None] + (Skv - Sq)
    keep = (j <= diag) if causal else np.ones((rows.shape[0], Skv), bool)
    if window_right >= 0:
        keep = keep & (j <= diag + window_right)
    if window_left >= 0:
        keep = keep & (j >= rows[:, None] - window_left)   # mistake: left bound not aligned
    return keep


def _window_right_ignored(rows, Sq, Skv, causal, window_left=-1, window_right=-1):
    j = np.arange(Skv)[None, :]
    diag = rows[:, None] + (Skv - Sq)
    keep = (j <= diag) if causal else np.ones((rows.shape[0], Skv), bool)
    if window_left >= 0:
        keep = keep & (j >= diag - window_left)
    return keep


def _varlen_shared_offsets(q, k, v, cq, ck, **kw):
    # mistake: the key rows of each sequence taken at the query offsets
    return oracle.sdpa_varlen(q, k, v, cq, cq, **kw)


def _varlen_lse_row_major(q, k, v, cq, ck, **kw):
    o, lse = oracle.sdpa_varlen(q, k, v, cq, ck, **kw)
    return o, lse.reshape(-1).reshape(lse.shape[1], lse.shape[0]).T


def _sdpa_gqa_modulo(q, k, v, *, causal, scale, rows=None, **kw):
    q, k, v = (A._f64(x) for x in (q, k, v))
    Hq, Hkv = q.shape[1], k.shape[1]
    outs, lses = [], []
    for h in range(Hq):
        kv = h % Hkv
        o, l = oracle.sdpa(q[:, h:h + 1], k[:, kv:kv + 1], v[:, kv:kv + 1], causal=causal,
                           scale=scale, rows=None if rows is None else np.atleast_2d(rows)[
                               min(h, np.atleast_2d(rows).shape[0] - 1)])
        outs.append(o)
        lses.append(l)
    return np.concatenate(outs, axis=1), np.concatenate(lses, axis=1)


def _sdpa_no_scale(q, k, v, *, causal, scale, rows=None, **kw):
    return oracle.sdpa(q, k, v, causal=causal, scale=1.0, rows=rows, **kw)


def _sdpa_lse_log2(q, k, v, *, causal, scale, rows=None, **kw):
    o, lse = oracle.sdpa(q, k, v, causal=causal, scale=scale, rows=rows, **kw)
    return o, lse / math.log(2.0)


def _sdpa_lse_no_max(q, k, v, *, causal, scale, rows=None, **kw):
    o, lse = oracle.sdpa(q, k, v, causal=causal, scale=scale, rows=rows)
    _, m, l = (None, None, None)
    out_l = np.empty_like(lse)
    q, k = A._f64(q), A._f64(k)
    G = q.shape[1] // k.shape[1]
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            rr = None if rows is None else np.atleast_2d(rows)[min(h, np.atleast_2d(rows).shape[0] - 1)]
            _, m, l = oracle.softmax_probs(q[b, h], k[b, h // G], causal=causal, scale=scale, rows=rr)
            with np.errstate(divide="ignore"):
                out_l[b, h] = np.log(l)
    return o, out_l


def _sdpa_transposed_scores(q, k, v, *, causal, scale, rows=None, **kw):
    q, k, v = (A._f64(x) for x in (q, k, v))
    if q.shape[2] != k.shape[2] or q.shape[1] != k.shape[1]:
        raise ValueError("mutant only defined for square MHA")
    # swap the roles of Q and K: scores become S^T
    return oracle.sdpa(k, q, v, causal=causal, scale=scale, rows=rows)


def _decode_gqa_modulo(q, k_cache, v_cache, seq_lens, *, scale):
    q = A._f64(q)
    Hq, Hkv = q.shape[1], k_cache.shape[1]
    k2 = np.stack([A._f64(k_cache)[:, h % Hkv] for h in range(Hq)], axis=1)
    v2 = np.stack([A._f64(v_cache)[:, h % Hkv] for h in range(Hq)], axis=1)
    return oracle.decode(q, k2, v2, seq_lens, scale=scale)


def _partials_normalised(q, k, v, lens, *, chunk, scale, max_chunks=None):
    p = oracle.decode_partials(q, k, v, lens, chunk=chunk, scale=scale, max_chunks=max_chunks)
    D = p.shape[-1] - 2
    with np.errstate(invalid="ignore", divide="ignore"):
        p[..., :D] = np.where(p[..., D + 1:] > 0, p[..., :D] / p[..., D + 1:], 0.0)
    return p


def _merge_without_rescale(partials, seq_lens, *, chunk):
    p = np.array(partials, dtype=np.float64)
    D = p.shape[-1] - 2
    finite = np.isfinite(p[..., D])
    p[..., D] = np.where(finite, 0.0, p[..., D])     # every weight e^(m_c - M) becomes 1
    return oracle.merge_partials(p, seq_lens, chunk=chunk)


def _merge_drops_l_weight(partials, seq_lens, *, chunk):
    p = np.array(partials, dtype=np.float64)
    D = p.shape[-1] - 2
    out = oracle.merge_partials(p, seq_lens, chunk=chunk)
    # mistake: divide by the plain sum of l_c instead of the rescaled one
    B, H = p.shape[:2]
    for b in range(B):
        n = oracle.num_chunks(int(seq_lens[b]), chunk)
        for h in range(H):
            if n == 0:
                continue
            M = p[b, h, :n, D].max()
            w = np.exp(p[b, h, :n, D] - M)
            out[b, h] = (p[b, h, :n, :D] * w[:, None]).sum(0) / p[b, h, :n, D + 1].sum()
    return out


def _bwd_without_local_sum(q, k, v, dout, *, causal, scale, **win):
    # mistake: dpreatt = scale * att * datt, the row term sum_j att * datt dropped
    q, k, v, do = (A._f64(x) for x in (q, k, v, dout))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    G = q.shape[1] // k.shape[1]
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            att, _, _ = oracle.softmax_probs(q[b, h], k[b, h // G], causal=causal, scale=scale, **win)
            datt = do[b, h] @ v[b, h // G].T
            dv[b, h // G] += att.T @ do[b, h]
            dpre = scale * att * datt
            dq[b, h] = dpre @ k[b, h // G]
            dk[b, h // G] += dpre.T @ q[b, h]
    return dq, dk, dv


def _bwd_dk_not_summed_over_group(q, k, v, dout, *, causal, scale, **win):
    dq, dk, dv = oracle.sdpa_backward(q, k, v, dout, causal=causal, scale=scale, **win)
    G = A._f64(q).shape[1] // A._f64(k).shape[1]
    return dq, dk / G, dv                           # mistake: an average, not the sum


def _bwd_unscaled(q, k, v, dout, *, causal, scale, **win):
    dq, dk, dv = oracle.sdpa_backward(q, k, v, dout, causal=causal, scale=scale, **win)
    return dq / scale, dk / scale, dv               # mistake: the chain rule's scale dropped


def _bwd_window_ignored(q, k, v, dout, *, causal, scale, **win):
    # mistake: the backward re-forms P without the window's bounds
    return oracle.sdpa_backward(q, k, v, dout, causal=causal, scale=scale)


def _bwd_varlen_key_offsets_from_queries(q, k, v, dout, cu_q, cu_k, **kw):
    # mistake: the keys of sequence b taken at the query offsets
    return oracle.sdpa_backward_varlen(q, k, v, dout, cu_q, cu_q, **kw)


MUTANTS = {
    "causal_strict_diagonal": _impl(**_with_visible(_strict)),
    "causal_top_left_alignment": _impl(**_with_visible(_top_left)),
    "gqa_head_modulo": _impl(sdpa=_sdpa_gqa_modulo),
    "scale_dropped": _impl(sdpa=_sdpa_no_scale),
    "lse_in_log2": _impl(sdpa=_sdpa_lse_log2),
    "lse_missing_max": _impl(sdpa=_sdpa_lse_no_max),
    "q_k_transposed": _impl(sdpa=_sdpa_transposed_scores),
    "decode_gqa_modulo": _impl(decode=_decode_gqa_modulo),
    "partials_normalised": _impl(decode_partials=_partials_normalised),
    "merge_without_rescale": _impl(merge_partials=_merge_without_rescale),
    "merge_unweighted_l": _impl(merge_partials=_merge_drops_l_weight),
    "window_left_bound_exclusive": _impl(**_with_visible(_window_left_strict)),
    "window_left_not_bottom_right": _impl(**_with_visible(_window_top_left)),
    "window_right_bound_ignored": _impl(**_with_visible(_window_right_ignored)),
    "varlen_key_offsets_from_queries": _impl(sdpa_varlen=_varlen_shared_offsets),
    "varlen_lse_row_major": _impl(sdpa_varlen=_varlen_lse_row_major),
    "backward_row_term_dropped": _impl(sdpa_backward=_bwd_without_local_sum),
    "backward_group_average": _impl(sdpa_backward=_bwd_dk_not_summed_over_group),
    "backward_unscaled": _impl(sdpa_backward=_bwd_unscaled),
    "backward_window_ignored": _impl(sdpa_backward=_bwd_window_ignored),
    "backward_varlen_key_offsets_from_queries":
        _impl(sdpa_backward_varlen=_bwd_varlen_key_offsets_from_queries),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    bad = pins.failing_pins(MUTANTS[name])
    assert bad, f"mutant {name} passed every pin"


def test_real_oracle_passes_every_pin():
    assert pins.failing_pins(_impl()) == []
