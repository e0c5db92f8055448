"""Pins that tie the float64 oracle to what the definition of attention fixes.

Each pin is a function ``pin_*(impl)`` that raises AssertionError when the
implementation ``impl`` (a namespace with ``sdpa``, ``sdpa_varlen``, ``sdpa_backward``,
``sdpa_backward_varlen``,
``softmax_probs``, ``decode``, ``decode_partials`` and ``merge_partials``)
disagrees with a fact
that does not depend on the oracle: a closed form, an invariant, a hand-worked
example, an independent library routine or a brute-force loop.  The same pins
run against the real oracle (must all pass) and against mutants of it with a
planted mistake (each must trip at least one pin).
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).normal(0.0, std, size=shape)


def _close(a, b, tol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(a - b))
    assert np.all(np.isfinite(err)), f"{what}: non-finite mismatch"
    scale = np.maximum(1.0, np.abs(np.where(both_inf, 0.0, b)))
    worst = float(np.max(err / scale)) if err.size else 0.0
    assert worst <= tol, f"{what}: max rel err {worst:.3e} > {tol:.1e}"


def _ev(x):
    if isinstance(x, list):
        return [_ev(y) for y in x]
    return float(eval(x, {"__builtins__": {}}, {"log": math.log, "inf": math.inf}))


# ---------------------------------------------------------------- prefill pins

def pin_rows_sum_to_one(impl):
    q, k = _rand((37, 8), 1), _rand((53, 8), 2)
    for causal in (False, True):
        p, m, l = impl.softmax_probs(q, k, causal=causal, scale=0.7)
        sums = p.sum(axis=1)
        nonempty = l > 0
        _close(sums[nonempty], np.ones(int(nonempty.sum())), 1e-12, "P row sums")
        assert np.all(p >= 0), "negative probability"


def pin_single_key(impl):
    q, k, v = _rand((1, 3, 5, 16), 3), _rand((1, 3, 1, 16), 4), _rand((1, 3, 1, 16), 5)
    o, lse = impl.sdpa(q, k, v, causal=False, scale=0.3)
    _close(o, np.broadcast_to(v, o.shape), 1e-12, "single key O")
    want = 0.3 * np.einsum("bhsd,bhd->bhs", q, k[:, :, 0])
    _close(lse, want, 1e-12, "single key LSE")


def pin_constant_v(impl):
    q, k = _rand((2, 2, 9, 8), 6, std=3.0), _rand((2, 2, 11, 8), 7)
    row = _rand((8,), 8)
    v = np.broadcast_to(row, (2, 2, 11, 8)).copy()
    for causal in (False, True):
        o, _ = impl.sdpa(q, k, v, causal=causal, scale=0.5)
        _close(o, np.broadcast_to(row, o.shape), 1e-12, "constant V")


def pin_causal_row0(impl):
    q, k, v = _rand((1, 2, 7, 8), 9), _rand((1, 2, 7, 8), 10), _rand((1, 2, 7, 8), 11)
    o, lse = impl.sdpa(q, k, v, causal=True, scale=0.9)
    _close(o[:, :, 0], v[:, :, 0], 1e-12, "causal row 0 O")
    _close(lse[:, :, 0], 0.9 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), 1e-12,
           "causal row 0 LSE")


def pin_scale_zero(impl):
    q, k, v = _rand((1, 1, 6, 4), 12), _rand((1, 1, 6, 4), 13), _rand((1, 1, 6, 4), 14)
    o, lse = impl.sdpa(q, k, v, causal=True, scale=0.0)
    for i in range(6):
        _close(o[0, 0, i], v[0, 0, : i + 1].mean(axis=0), 1e-12, f"scale 0 row {i}")
        _close(lse[0, 0, i], math.log(i + 1), 1e-12, f"scale 0 LSE row {i}")
    o, lse = impl.sdpa(q, k, v, causal=False, scale=0.0)
    _close(o[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (6, 4)), 1e-12, "scale 0 non-causal")
    _close(lse, np.full((1, 1, 6), math.log(6)), 1e-12, "scale 0 non-causal LSE")


def pin_permutation(impl):
    q, k, v = _rand((1, 2, 5, 8), 15), _rand((1, 2, 13, 8), 16), _rand((1, 2, 13, 8), 17)
    perm = np.random.default_rng(18).permutation(13)
    o1, l1 = impl.sdpa(q, k, v, causal=False, scale=0.4)
    o2, l2 = impl.sdpa(q, k[:, :, perm], v[:, :, perm], causal=False, scale=0.4)
    _close(o1, o2, 1e-12, "permutation O")
    _close(l1, l2, 1e-12, "permutation LSE")


def pin_gqa_equals_repeated_mha(impl):
    q, k, v = _rand((2, 8, 6, 4), 19), _rand((2, 2, 6, 4), 20), _rand((2, 2, 6, 4), 21)
    for causal in (False, True):
        o1, l1 = impl.sdpa(q, k, v, causal=causal, scale=0.6)
        o2, l2 = impl.sdpa(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1),
                           causal=causal, scale=0.6)
        _close(o1, o2, 1e-12, "GQA O")
        _close(l1, l2, 1e-12, "GQA LSE")


def pin_rows_subset(impl):
    q, k, v = _rand((1, 2, 20, 4), 22), _rand((1, 2, 20, 4), 23), _rand((1, 2, 20, 4), 24)
    rows = np.array([0, 3, 19])
    o1, l1 = impl.sdpa(q, k, v, causal=True, scale=0.5)
    o2, l2 = impl.sdpa(q, k, v, causal=True, scale=0.5, rows=rows)
    _close(o2, o1[:, :, rows], 1e-12, "row subset O")
    _close(l2, l1[:, :, rows], 1e-12, "row subset LSE")
    per_head = np.array([[1, 2], [5, 18]])
    o3, _ = impl.sdpa(q, k, v, causal=True, scale=0.5, rows=per_head)
    _close(o3[:, 0], o1[:, 0, [1, 2]], 1e-12, "per-head rows h0")
    _close(o3[:, 1], o1[:, 1, [5, 18]], 1e-12, "per-head rows h1")


def pin_torch_math_sdpa(impl):
    """Independent library routine: PyTorch CPU float64 SDPA and logsumexp (Sq == Skv)."""
    for causal in (False, True):
        q, k, v = _rand((2, 3, 17, 8), 25), _rand((2, 3, 17, 8), 26), _rand((2, 3, 17, 8), 27)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        want = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, is_causal=causal, scale=0.35).numpy()
        s = 0.35 * torch.einsum("bhid,bhjd->bhij", tq, tk)
        if causal:
            s = s.masked_fill(torch.ones(17, 17, dtype=torch.bool).triu(1), float("-inf"))
        want_lse = torch.logsumexp(s, dim=-1).numpy()
        o, lse = impl.sdpa(q, k, v, causal=causal, scale=0.35)
        _close(o, want, 1e-10, f"torch sdpa causal={causal}")
        _close(lse, want_lse, 1e-10, f"torch logsumexp causal={causal}")


def _brute(q, k, v, causal, scale):
    """Pure-Python triple loop, written independently of the oracle."""
    B, Hq, Sq, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv, Skv = len(k[0]), len(k[0][0])
    out = [[[[0.0] * D for _ in range(Sq)] for _ in range(Hq)] for _ in range(B)]
    lse = [[[-math.inf] * Sq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            g = h * Hkv // Hq
            for i in range(Sq):
                keys = [j for j in range(Skv) if not causal or j <= i + Skv - Sq]
                if not keys:
                    continue
                sc = {j: scale * sum(q[b][h][i][d] * k[b][g][j][d] for d in range(D)) for j in keys}
                mx = max(sc.values())
                w = {j: math.exp(sc[j] - mx) for j in keys}
                tot = sum(w.values())
                for d in range(D):
                    out[b][h][i][d] = sum(w[j] * v[b][g][j][d] for j in keys) / tot
                lse[b][h][i] = mx + math.log(tot)
    return np.array(out), np.array(lse)


def pin_brute_force(impl):
    cases = [((1, 2, 5, 3), (1, 1, 5, 3), True), ((2, 2, 4, 2), (2, 2, 6, 2), False),
             ((1, 4, 6, 3), (1, 2, 3, 3), True), ((1, 1, 2, 4), (1, 1, 7, 4), True)]
    for n, (qs, ks, causal) in enumerate(cases):
        q, k, v = _rand(qs, 30 + n), _rand(ks, 40 + n), _rand(ks, 50 + n)
        want_o, want_l = _brute(q.tolist(), k.tolist(), v.tolist(), causal, 0.8)
        o, lse = impl.sdpa(q, k, v, causal=causal, scale=0.8)
        _close(o, want_o, 1e-12, f"brute force case {n} O")
        _close(lse, want_l, 1e-12, f"brute force case {n} LSE")


def pin_hand_worked(impl):
    with open(GOLDEN) as f:
        gold = json.load(f)
    for ex in gold["fwd"]:
        q, k, v = (np.array(_ev(ex[n]))[None] for n in ("q", "k", "v"))
        o, lse = impl.sdpa(q, k, v, causal=ex["causal"], scale=ex["scale"])
        _close(o, np.array(_ev(ex["O"]))[None], 1e-12, ex["name"] + " O")
        _close(lse, np.array(_ev(ex["LSE"]))[None], 1e-12, ex["name"] + " LSE")
    for ex in gold["decode_chunks"]:
        q = np.array(_ev(ex["q"]))[None, None]                 # [1, 1, D]
        k = np.array(_ev(ex["k"]))[None, None]                 # [1, 1, L, D]
        v = np.array(_ev(ex["v"]))[None, None]
        lens = np.array([ex["seq_len"]])
        part = impl.decode_partials(q, k, v, lens, chunk=ex["chunk"], scale=ex["scale"])
        want = np.array([[[_ev(x) for x in row] for row in ex["partials"]]])[None]
        _close(part[..., : want.shape[2], :], want, 1e-12, ex["name"] + " partials")
        o = impl.merge_partials(part, lens, chunk=ex["chunk"])
        _close(o, np.array(_ev(ex["O"]))[None, None], 1e-12, ex["name"] + " O")


def pin_empty_rows(impl):
    q, k, v = _rand((1, 1, 5, 4), 60), _rand((1, 1, 2, 4), 61), _rand((1, 1, 2, 4), 62)
    o, lse = impl.sdpa(q, k, v, causal=True, scale=1.0)   # Sq=5 > Skv=2: rows 0..2 empty
    assert np.all(o[0, 0, :3] == 0.0), "empty causal rows must be 0"
    assert np.all(np.isneginf(lse[0, 0, :3])), "empty causal rows must have LSE = -inf"
    _close(o[0, 0, 3], v[0, 0, 0], 1e-12, "first non-empty row")


# ------------------------------------------------ sliding window and varlen pins

def _window_keys(i, Sq, Skv, causal, wl, wr):
    """Keys query i keeps, enumerated one by one from the window's wording."""
    diag = i + Skv - Sq
    keys = []
    for j in range(Skv):
        if causal and j > diag:
            continue
        if wr >= 0 and j > diag + wr:
            continue
        if wl >= 0 and j < diag - wl:
            continue
        keys.append(j)
    return keys


WINDOW_CASES = [  # (Sq, Skv, causal, window_left, window_right)
    (6, 6, True, 2, -1), (6, 6, False, 1, 2), (5, 9, True, 3, -1), (9, 5, True, 0, -1),
    (7, 7, False, -1, 0), (7, 7, False, 0, -1), (4, 10, False, 2, 2), (8, 3, False, 1, 1),
    (6, 6, True, 0, 5),
]


def pin_window_brute_force(impl):
    """Pure-Python loops over the explicitly enumerated key set of each row."""
    for n, (Sq, Skv, causal, wl, wr) in enumerate(WINDOW_CASES):
        q, k, v = _rand((1, 2, Sq, 3), 300 + n), _rand((1, 1, Skv, 3), 320 + n), _rand((1, 1, Skv, 3), 340 + n)
        o, lse = impl.sdpa(q, k, v, causal=causal, scale=0.9, window_left=wl, window_right=wr)
        for h in range(2):
            for i in range(Sq):
                keys = _window_keys(i, Sq, Skv, causal, wl, wr)
                if not keys:
                    assert np.all(o[0, h, i] == 0) and np.isneginf(lse[0, h, i]), f"window {n} empty row"
                    continue
                sc = [0.9 * sum(q[0, h, i, d] * k[0, 0, j, d] for d in range(3)) for j in keys]
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                tot = sum(w)
                want = [sum(w[t] * v[0, 0, j, d] for t, j in enumerate(keys)) / tot for d in range(3)]
                _close(o[0, h, i], want, 1e-12, f"window case {n} row {i} O")
                _close(lse[0, h, i], mx + math.log(tot), 1e-12, f"window case {n} row {i} LSE")


def pin_window_diagonal(impl):
    """A window of width zero keeps only the diagonal key: O = V[i + d], LSE = its score."""
    for Sq, Skv in ((5, 5), (3, 8)):
        q, k, v = _rand((1, 1, Sq, 4), 360), _rand((1, 1, Skv, 4), 361), _rand((1, 1, Skv, 4), 362)
        d = Skv - Sq
        for causal, wr in ((True, -1), (False, 0)):
            o, lse = impl.sdpa(q, k, v, causal=causal, scale=0.6, window_left=0, window_right=wr)
            _close(o[0, 0], v[0, 0, d:d + Sq], 1e-12, "diagonal window O")
            _close(lse[0, 0], 0.6 * np.einsum("id,id->i", q[0, 0], k[0, 0, d:d + Sq]), 1e-12,
                   "diagonal window LSE")


def pin_window_torch_slice(impl):
    """Each row equals PyTorch SDPA (no mask) over that row's contiguous key slice."""
    Sq, Skv = 9, 13
    q, k, v = _rand((1, 1, Sq, 5), 370), _rand((1, 1, Skv, 5), 371), _rand((1, 1, Skv, 5), 372)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    for causal, wl, wr in ((True, 3, -1), (False, 2, 4), (False, 5, 0)):
        o, lse = impl.sdpa(q, k, v, causal=causal, scale=0.4, window_left=wl, window_right=wr)
        for i in range(Sq):
            diag = i + Skv - Sq
            lo = max(0, diag - wl)
            hi = min(Skv - 1, diag if causal else diag + wr)
            want = torch.nn.functional.scaled_dot_product_attention(
                tq[:, :, i:i + 1], tk[:, :, lo:hi + 1], tv[:, :, lo:hi + 1], scale=0.4)
            want_l = torch.logsumexp(0.4 * (tk[0, 0, lo:hi + 1] @ tq[0, 0, i]), dim=0)
            _close(o[0, 0, i], want[0, 0, 0].numpy(), 1e-10, f"slice row {i} O")
            _close(lse[0, 0, i], float(want_l), 1e-10, f"slice row {i} LSE")


def pin_window_wide_is_plain(impl):
    """Windows at least as wide as the keys change nothing."""
    q, k, v = _rand((2, 2, 7, 4), 380), _rand((2, 1, 11, 4), 381), _rand((2, 1, 11, 4), 382)
    for causal in (False, True):
        o0, l0 = impl.sdpa(q, k, v, causal=causal, scale=0.7)
        o1, l1 = impl.sdpa(q, k, v, causal=causal, scale=0.7, window_left=11, window_right=11)
        _close(o1, o0, 1e-12, "wide window O")
        _close(l1, l0, 1e-12, "wide window LSE")


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)


def pin_varlen_equal_lengths(impl):
    """Packed sequences of one length equal the batched [B, H, S, D] definition."""
    B, S, Hq, Hkv, D = 3, 6, 4, 2, 5
    q, k, v = _rand((B, S, Hq, D), 390), _rand((B, S, Hkv, D), 391), _rand((B, S, Hkv, D), 392)
    cu = _cu([S] * B)
    for causal, wl in ((True, -1), (False, -1), (True, 2)):
        o, lse = impl.sdpa_varlen(q.reshape(B * S, Hq, D), k.reshape(B * S, Hkv, D),
                                  v.reshape(B * S, Hkv, D), cu, cu, causal=causal, scale=0.5,
                                  window_left=wl)
        want_o, want_l = impl.sdpa(q.transpose(0, 2, 1, 3), k.transpose(0, 2, 1, 3),
                                   v.transpose(0, 2, 1, 3), causal=causal, scale=0.5, window_left=wl)
        _close(o, want_o.transpose(0, 2, 1, 3).reshape(B * S, Hq, D), 1e-12, "varlen equal O")
        _close(lse, want_l.transpose(1, 0, 2).reshape(Hq, B * S), 1e-12, "varlen equal LSE")


def pin_varlen_torch_per_sequence(impl):
    """Ragged packed batches: every sequence equals PyTorch SDPA on its own rows."""
    lq, lk = [5, 0, 3, 7], [4, 6, 3, 9]          # query and key lengths differ per sequence
    cq, ck = _cu(lq), _cu(lk)
    Hq, D = 2, 4
    q, k, v = _rand((int(cq[-1]) + 2, Hq, D), 400), _rand((int(ck[-1]), 1, D), 401), _rand((int(ck[-1]), 1, D), 402)
    o, lse = impl.sdpa_varlen(q, k, v, cq, ck, causal=False, scale=0.8)
    for b in range(4):
        if lq[b] == 0:
            continue
        tq = torch.from_numpy(q[cq[b]:cq[b + 1]]).permute(1, 0, 2)[None]
        tk = torch.from_numpy(k[ck[b]:ck[b + 1]]).permute(1, 0, 2)[None].expand(1, Hq, -1, -1)
        tv = torch.from_numpy(v[ck[b]:ck[b + 1]]).permute(1, 0, 2)[None].expand(1, Hq, -1, -1)
        want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.8)
        want_l = torch.logsumexp(0.8 * tq @ tk.transpose(-1, -2), dim=-1)
        _close(o[cq[b]:cq[b + 1]], want[0].permute(1, 0, 2).numpy(), 1e-10, f"varlen seq {b} O")
        _close(lse[:, cq[b]:cq[b + 1]], want_l[0].numpy(), 1e-10, f"varlen seq {b} LSE")
    assert np.all(o[int(cq[-1]):] == 0) and np.all(np.isneginf(lse[:, int(cq[-1]):])), \
        "rows outside every sequence"


# ---------------------------------------------------------------- backward pins

def pin_backward_torch_autograd(impl):
    """PyTorch float64 autograd through its own SDPA (GQA by repeating K and V heads)."""
    for causal, (Hq, Hkv) in ((True, (4, 2)), (False, (2, 2)), (True, (3, 1))):
        q, k, v = _rand((2, Hq, 9, 6), 500), _rand((2, Hkv, 9, 6), 501), _rand((2, Hkv, 9, 6), 502)
        do = _rand((2, Hq, 9, 6), 503)
        tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
        G = Hq // Hkv
        o = torch.nn.functional.scaled_dot_product_attention(
            tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1), is_causal=causal,
            scale=0.45)
        o.backward(torch.from_numpy(do))
        dq, dk, dv = impl.sdpa_backward(q, k, v, do, causal=causal, scale=0.45)
        _close(dq, tq.grad.numpy(), 1e-10, f"autograd dQ causal={causal}")
        _close(dk, tk.grad.numpy(), 1e-10, f"autograd dK causal={causal}")
        _close(dv, tv.grad.numpy(), 1e-10, f"autograd dV causal={causal}")


def pin_backward_finite_differences(impl):
    """Central differences of sum(dO * O) through the forward, Sq != Skv bottom-right causal."""
    q, k, v = _rand((1, 2, 4, 3), 510), _rand((1, 1, 6, 3), 511), _rand((1, 1, 6, 3), 512)
    do = _rand((1, 2, 4, 3), 513)
    dq, dk, dv = impl.sdpa_backward(q, k, v, do, causal=True, scale=0.7)
    eps = 1e-6

    def loss(q_, k_, v_):
        o, _ = impl.sdpa(q_, k_, v_, causal=True, scale=0.7)
        return float((o * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        _close(g, num, 1e-7, f"finite differences d{name}")


def pin_backward_single_key(impl):
    """One key: P = 1 whatever Q and K are, so dQ = dK = 0 and dV = sum of dO."""
    q, k, v = _rand((1, 2, 5, 4), 520), _rand((1, 2, 1, 4), 521), _rand((1, 2, 1, 4), 522)
    do = _rand((1, 2, 5, 4), 523)
    dq, dk, dv = impl.sdpa_backward(q, k, v, do, causal=False, scale=0.9)
    _close(dq, np.zeros_like(dq), 1e-12, "single key dQ")
    _close(dk, np.zeros_like(dk), 1e-12, "single key dK")
    _close(dv[0, :, 0], do[0].sum(axis=1), 1e-12, "single key dV")


def _mask_from_keys(Sq, Skv, causal, wl, wr):
    """Boolean [Sq, Skv] mask of the keys each query keeps, from the window's wording."""
    m = np.zeros((Sq, Skv), dtype=bool)
    for i in range(Sq):
        for j in _window_keys(i, Sq, Skv, causal, wl, wr):
            m[i, j] = True
    return m


def _torch_grads(q, k, v, do, mask, scale):
    """PyTorch float64 autograd through its SDPA with an explicit boolean mask [Sq, Skv]
    (GQA by repeating K and V heads); every row must keep at least one key."""
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    G = q.shape[1] // k.shape[1]
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1),
        attn_mask=torch.from_numpy(mask), scale=scale)
    o.backward(torch.from_numpy(do))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


BWD_WINDOW_CASES = [  # (Sq, Skv, causal, window_left, window_right, Hq, Hkv); every row keeps a key
    (9, 9, True, 2, -1, 4, 2),
    (6, 10, True, 3, -1, 2, 1),
    (8, 8, False, 1, 2, 2, 2),
    (7, 5, False, -1, 2, 3, 1),
]


def pin_backward_window_autograd(impl):
    """Sliding windows: PyTorch float64 autograd through SDPA with the window's key
    sets enumerated one by one (bottom-right alignment, GQA, Sq != Skv both ways)."""
    for n, (Sq, Skv, causal, wl, wr, Hq, Hkv) in enumerate(BWD_WINDOW_CASES):
        q, k, v = _rand((1, Hq, Sq, 5), 540 + n), _rand((1, Hkv, Skv, 5), 550 + n), _rand((1, Hkv, Skv, 5), 560 + n)
        do = _rand((1, Hq, Sq, 5), 570 + n)
        mask = _mask_from_keys(Sq, Skv, causal, wl, wr)
        assert mask.any(axis=1).all(), "every row of a pin case keeps a key"
        want = _torch_grads(q, k, v, do, mask, 0.55)
        got = impl.sdpa_backward(q, k, v, do, causal=causal, scale=0.55, window_left=wl, window_right=wr)
        for name, g, w in zip(("dQ", "dK", "dV"), got, want):
            _close(g, w, 1e-10, f"window backward case {n} {name}")


def pin_backward_window_finite_differences(impl):
    """Central differences of sum(dO * O) through the windowed forward."""
    q, k, v = _rand((1, 2, 5, 3), 580), _rand((1, 1, 7, 3), 581), _rand((1, 1, 7, 3), 582)
    do = _rand((1, 2, 5, 3), 583)
    kw = dict(causal=True, scale=0.8, window_left=2, window_right=-1)
    dq, dk, dv = impl.sdpa_backward(q, k, v, do, **kw)
    eps = 1e-6

    def loss(q_, k_, v_):
        o, _ = impl.sdpa(q_, k_, v_, **kw)
        return float((o * do).sum())

    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        _close(g, num, 1e-7, f"window finite differences d{name}")


def pin_backward_varlen_per_sequence(impl):
    """Packed batches: each sequence's gradients equal PyTorch autograd on its own rows
    (bottom-right causal window, GQA 2, query and key lengths differing per sequence);
    rows outside every sequence get zero gradients."""
    lq, lk = [4, 0, 6, 3], [5, 3, 6, 7]
    cq, ck = _cu(lq), _cu(lk)
    Hq, Hkv, D = 2, 1, 4
    q, do = _rand((int(cq[-1]) + 2, Hq, D), 590), _rand((int(cq[-1]) + 2, Hq, D), 593)
    k, v = _rand((int(ck[-1]) + 1, Hkv, D), 591), _rand((int(ck[-1]) + 1, Hkv, D), 592)
    wl = 3
    dq, dk, dv = impl.sdpa_backward_varlen(q, k, v, do, cq, ck, causal=True, scale=0.6, window_left=wl)
    for b in range(4):
        if lq[b] == 0:
            continue
        t = lambda x, a, e: np.ascontiguousarray(x[a:e].transpose(1, 0, 2)[None])
        mask = _mask_from_keys(lq[b], lk[b], True, wl, -1)
        want = _torch_grads(t(q, cq[b], cq[b + 1]), t(k, ck[b], ck[b + 1]), t(v, ck[b], ck[b + 1]),
                            t(do, cq[b], cq[b + 1]), mask, 0.6)
        _close(dq[cq[b]:cq[b + 1]], want[0][0].transpose(1, 0, 2), 1e-10, f"varlen backward seq {b} dQ")
        _close(dk[ck[b]:ck[b + 1]], want[1][0].transpose(1, 0, 2), 1e-10, f"varlen backward seq {b} dK")
        _close(dv[ck[b]:ck[b + 1]], want[2][0].transpose(1, 0, 2), 1e-10, f"varlen backward seq {b} dV")
    # sequence 1 has no query: its keys get no gradient; nor do rows outside every sequence
    assert np.all(dk[ck[1]:ck[2]] == 0) and np.all(dv[ck[1]:ck[2]] == 0), "keys of a query-less sequence"
    assert np.all(dq[int(cq[-1]):] == 0) and np.all(dk[int(ck[-1]):] == 0), "rows outside every sequence"


# ----------------------------------------------------------------- decode pins

def _decode_case(seed, B=3, Hq=4, Hkv=2, max_S=40, D=8):
    q = _rand((B, Hq, D), seed)
    k = _rand((B, Hkv, max_S, D), seed + 1)
    v = _rand((B, Hkv, max_S, D), seed + 2)
    lens = np.array([max_S, 17, 1][:B])
    return q, k, v, lens


def pin_decode_equals_prefill(impl):
    q, k, v, lens = _decode_case(70)
    o = impl.decode(q, k, v, lens, scale=0.45)
    for b, L in enumerate(lens):
        want, _ = impl.sdpa(q[b][None, :, None], k[b][None, :, :L], v[b][None, :, :L],
                            causal=False, scale=0.45)
        _close(o[b], want[0, :, 0], 1e-12, f"decode b={b}")
        # Sq = 1 with a causal mask aligned bottom-right sees the whole prefix too
        want_c, _ = impl.sdpa(q[b][None, :, None], k[b][None, :, :L], v[b][None, :, :L],
                              causal=True, scale=0.45)
        _close(o[b], want_c[0, :, 0], 1e-12, f"decode causal b={b}")


def pin_decode_zero_len(impl):
    q, k, v, _ = _decode_case(80)
    o = impl.decode(q, k, v, np.array([0, 5, 0]), scale=0.5)
    assert np.all(o[0] == 0) and np.all(o[2] == 0), "L = 0 gives O = 0"
    o2 = impl.merge_partials(impl.decode_partials(q, k, v, np.array([0, 5, 0]), chunk=4,
                                                  scale=0.5), np.array([0, 5, 0]), chunk=4)
    assert np.all(o2[0] == 0) and np.all(o2[2] == 0), "merge with no chunk gives O = 0"


def pin_chunked_equals_unchunked(impl):
    q, k, v, lens = _decode_case(90)
    full = impl.decode(q, k, v, lens, scale=0.6)
    for chunk in (1, 3, 8, 16, 40, 64):
        part = impl.decode_partials(q, k, v, lens, chunk=chunk, scale=0.6)
        o = impl.merge_partials(part, lens, chunk=chunk)
        _close(o, full, 1e-12, f"chunk {chunk}")


def pin_partials_definition(impl):
    """Each partial's o/l equals attention over that chunk alone; m is its max score."""
    q, k, v, lens = _decode_case(100, B=1, max_S=21)
    part = impl.decode_partials(q, k, v, lens, chunk=8, scale=0.3)
    D = q.shape[-1]
    for c, (lo, hi) in enumerate(((0, 8), (8, 16), (16, 21))):
        for h in range(q.shape[1]):
            kv = h // 2
            s = 0.3 * (k[0, kv, lo:hi] @ q[0, h])
            _close(part[0, h, c, D], s.max(), 1e-12, "chunk max")
            want, _ = impl.sdpa(q[0, h][None, None, None], k[0, kv, lo:hi][None, None],
                                v[0, kv, lo:hi][None, None], causal=False, scale=0.3)
            _close(part[0, h, c, :D] / part[0, h, c, D + 1], want[0, 0, 0], 1e-12,
                   "chunk o / l")


ALL_PINS = [
    pin_rows_sum_to_one, pin_single_key, pin_constant_v, pin_causal_row0, pin_scale_zero,
    pin_permutation, pin_gqa_equals_repeated_mha, pin_rows_subset, pin_torch_math_sdpa,
    pin_brute_force, pin_hand_worked, pin_empty_rows, pin_decode_equals_prefill,
    pin_decode_zero_len, pin_chunked_equals_unchunked, pin_partials_definition,
    pin_window_brute_force, pin_window_diagonal, pin_window_torch_slice, pin_window_wide_is_plain,
    pin_varlen_equal_lengths, pin_varlen_torch_per_sequence,
    pin_backward_torch_autograd, pin_backward_finite_differences, pin_backward_single_key,
    pin_backward_window_autograd, pin_backward_window_finite_differences,
    pin_backward_varlen_per_sequence,
]


def failing_pins(impl):
    """Names of the pins that ``impl`` fails."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(impl)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            bad.append(pin.__name__)
    return bad
