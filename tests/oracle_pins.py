"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, none of which re-types the oracle's own formula.

Every ``pin_*`` function takes an oracle object (``oracle.OracleLib`` or the
``oracle`` module) and raises AssertionError when the oracle disagrees.  The
same battery runs on the real oracle (tests/test_oracle_pins.py) and on
deliberately broken copies of it (tests/test_oracle_mutants.py), which shows
that a plausible mistake anywhere in the oracle trips at least one pin.
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _qkv(seed, B, H, N, D, std=1.0):
    r = _rng(seed)
    return (r.standard_normal((B, H, N, D)) * std,
            r.standard_normal((B, H, N, D)),
            r.standard_normal((B, H, N, D)))


def _close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), (what, "non-finite values")
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, "%s: max abs err %.3e > %.1e" % (what, err, tol)


# ---------------------------------------------------------------------------
# Invariants of softmax and of the weighted average (cishoon.github.io page,
# §1.1.2: every row of the normalised weights sums to 1; subtracting the row
# max leaves softmax unchanged).
# ---------------------------------------------------------------------------
def pin_row_sums(orc):
    q, k, _ = _qkv(11, 1, 2, 37, 8)
    for causal in (False, True):
        for bh in (0, 1):
            p = orc.probabilities(q, k, 1.0 / math.sqrt(8), causal, bh)
            assert np.all(p >= 0.0)
            _close(p.sum(axis=1), np.ones(37), 1e-12, "row sums causal=%s" % causal)
            if causal:
                assert np.all(np.triu(p, 1) == 0.0), "causal P must vanish above the diagonal"
                assert np.all(np.diag(p) > 0.0)


def pin_ones_v(orc):
    """V = 1 everywhere => O = 1 (a convex combination of equal rows)."""
    q, k, _ = _qkv(12, 2, 2, 29, 16, std=3.0)
    v = np.ones_like(q)
    for causal in (False, True):
        o, _ = orc.attention(q, k, v, 0.25, causal)
        _close(o, np.ones_like(o), 1e-13, "V=1 causal=%s" % causal)


def pin_zero_q(orc):
    """Q = 0 => uniform weights: O = mean of the visible V rows, lse = ln(#visible)."""
    B, H, N, D = 1, 2, 23, 5
    _, k, v = _qkv(13, B, H, N, D)
    q = np.zeros((B, H, N, D))
    o, lse = orc.attention(q, k, v, 0.7, False)
    _close(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), 1e-13, "Q=0 mean")
    _close(lse, np.full((B, H, N), math.log(N)), 1e-13, "Q=0 lse")
    o, lse = orc.attention(q, k, v, 0.7, True)
    counts = np.arange(1, N + 1, dtype=np.float64)
    prefix = np.cumsum(v, axis=2) / counts[None, None, :, None]
    _close(o, prefix, 1e-13, "Q=0 causal prefix mean")
    _close(lse, np.broadcast_to(np.log(counts), lse.shape), 1e-13, "Q=0 causal lse")


def pin_basis_v(orc):
    """Basis-vector V (V[kk][c0] = 1, else 0) => O[:, c0] = P[:, kk], other columns 0.
    (hjcheng0602.cn flashattn_G7 page, V46: the basis-vector probe.)"""
    B, H, N, D = 1, 1, 19, 6
    q, k, _ = _qkv(14, B, H, N, D)
    scale = 0.4
    for causal in (False, True):
        p = orc.probabilities(q, k, scale, causal, 0)
        for kk, c0 in ((0, 0), (7, 3), (18, 5)):
            v = np.zeros((B, H, N, D))
            v[0, 0, kk, c0] = 1.0
            o, _ = orc.attention(q, k, v, scale, causal)
            _close(o[0, 0, :, c0], p[:, kk], 1e-14, "basis V column")
            rest = np.delete(o[0, 0], c0, axis=1)
            _close(rest, np.zeros_like(rest), 0.0, "basis V other columns")


def pin_shift_invariance(orc):
    """K' = K + 1 u^T adds scale*(q_i . u) to every score of row i: O is
    unchanged and lse' = lse + scale*(q_i . u)."""
    B, H, N, D = 1, 2, 31, 7
    q, k, v = _qkv(15, B, H, N, D)
    u = _rng(16).standard_normal(D)
    scale = 0.37
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, scale, causal)
        o2, lse2 = orc.attention(q, k + u[None, None, None, :], v, scale, causal)
        _close(o2, o, 1e-12, "shift O causal=%s" % causal)
        _close(lse2 - lse, scale * (q @ u), 1e-12, "shift lse causal=%s" % causal)


def pin_single_key(orc):
    """N = 1: the one key gets weight 1, so O = V[0] and lse = scale*(q . k)."""
    q, k, v = _qkv(17, 3, 2, 1, 9)
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, 0.9, causal)
        _close(o, v, 0.0, "N=1 O")
        _close(lse, 0.9 * np.sum(q * k, axis=-1), 1e-14, "N=1 lse")


def pin_causal_first_rows(orc):
    """Causal row 0 sees only key 0 (O = V[0]); row 1 mixes keys 0 and 1 with the
    logistic weight of their score difference."""
    q, k, v = _qkv(18, 1, 1, 12, 4)
    scale = 0.5
    o, lse = orc.attention(q, k, v, scale, True)
    _close(o[0, 0, 0], v[0, 0, 0], 0.0, "causal row 0")
    s0 = scale * float(q[0, 0, 1] @ k[0, 0, 0])
    s1 = scale * float(q[0, 0, 1] @ k[0, 0, 1])
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    _close(o[0, 0, 1], (1 - w1) * v[0, 0, 0] + w1 * v[0, 0, 1], 1e-14, "causal row 1")
    _close(lse[0, 0, 0], scale * float(q[0, 0, 0] @ k[0, 0, 0]), 1e-14, "causal row 0 lse")
    _close(lse[0, 0, 1], max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))), 1e-14,
           "causal row 1 lse")


def pin_permutation(orc):
    """Non-causal attention is invariant under one joint permutation of the K and V rows."""
    B, H, N, D = 1, 2, 17, 5
    q, k, v = _qkv(19, B, H, N, D)
    perm = _rng(20).permutation(N)
    o, lse = orc.attention(q, k, v, 0.6, False)
    o2, lse2 = orc.attention(q, k[:, :, perm], v[:, :, perm], 0.6, False)
    _close(o2, o, 1e-13, "perm O")
    _close(lse2, lse, 1e-13, "perm lse")


def _decimal_attention(q, k, v, scale, causal):
    """Independent brute force: two passes in 40-digit decimal arithmetic, no max
    subtraction (the naive three-step definition: scores, row softmax, P.V)."""
    getcontext().prec = 40
    B, H, N, D = q.shape
    o = np.zeros((B, H, N, D))
    lse = np.zeros((B, H, N))
    p_all = np.zeros((B, H, N, N))
    sc = Decimal(float(scale))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                keys = range(i + 1) if causal else range(N)
                e = {}
                for j in keys:
                    dot = sum(Decimal(float(q[b, h, i, d])) * Decimal(float(k[b, h, j, d]))
                              for d in range(D))
                    e[j] = (sc * dot).exp()
                z = sum(e.values())
                for j in keys:
                    p_all[b, h, i, j] = float(e[j] / z)
                for c in range(D):
                    acc = sum(e[j] / z * Decimal(float(v[b, h, j, c])) for j in keys)
                    o[b, h, i, c] = float(acc)
                lse[b, h, i] = float(z.ln())
    return o, lse, p_all


def pin_bruteforce(orc):
    for (B, H, N, D, seed, std) in ((1, 1, 1, 1, 21, 1.0), (1, 2, 5, 3, 22, 1.0),
                                    (2, 1, 7, 2, 23, 2.0), (1, 1, 8, 4, 24, 0.5)):
        q, k, v = _qkv(seed, B, H, N, D, std)
        for causal in (False, True):
            scale = 0.8
            o, lse = orc.attention(q, k, v, scale, causal)
            ob, lb, pb = _decimal_attention(q, k, v, scale, causal)
            _close(o, ob, 1e-13, "brute O")
            _close(lse, lb, 1e-13, "brute lse")
            for bh in range(B * H):
                p = orc.probabilities(q, k, scale, causal, bh)
                _close(p, pb[bh // H, bh % H], 1e-14, "brute P")


def pin_rows_match_full(orc):
    """The selected-rows entry point returns exactly the full forward's rows."""
    B, H, N, D = 2, 3, 41, 8
    q, k, v = _qkv(25, B, H, N, D)
    r = _rng(26)
    bh = r.integers(0, B * H, 30)
    ri = r.integers(0, N, 30)
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, 0.3, causal)
        orow, lrow = orc.attention_rows(q, k, v, 0.3, causal, bh, ri)
        _close(orow, o.reshape(B * H, N, D)[bh, ri], 0.0, "rows O")
        _close(lrow, lse.reshape(B * H, N)[bh, ri], 0.0, "rows lse")


def pin_online_matches_definition(orc):
    """The tiled online-softmax restatement (outer Q tiles of Br rows, inner K/V
    tiles of Bc keys, causal skip + diagonal mask, tails) agrees with the
    definition on shapes that are not tile multiples."""
    cases = ((1, 1, 1, 4, 128, 32), (1, 2, 17, 8, 16, 8), (1, 1, 127, 8, 32, 16),
             (2, 1, 129, 8, 128, 32), (1, 1, 200, 16, 64, 32), (1, 1, 96, 8, 32, 32))
    for (B, H, N, D, Br, Bc) in cases:
        q, k, v = _qkv(27 + N, B, H, N, D, std=2.0)
        for causal in (False, True):
            o, lse = orc.attention(q, k, v, 0.35, causal)
            o2, lse2 = orc.attention_online(q, k, v, 0.35, causal, Br, Bc)
            _close(o2, o, 1e-12, "online O N=%d Br=%d Bc=%d causal=%s" % (N, Br, Bc, causal))
            _close(lse2, lse, 1e-12, "online lse")


def pin_golden_dot(orc):
    g = json.load(open(os.path.join(GOLDEN, "dot_product_worked.json")))
    q = np.array(g["q"], np.float64).reshape(1, 1, 1, -1)
    k = np.array(g["k"], np.float64).reshape(1, 1, 1, -1)
    v = np.array([[[[1.0, -2.0]]]])
    _, lse = orc.attention(q, k, v, 1.0, False)
    assert lse[0, 0, 0] == g["dot"], (lse, g["dot"])


def pin_golden_max_row(orc):
    g = json.load(open(os.path.join(GOLDEN, "max_reduction_row.json")))
    row = np.array(g["row"], np.float64)
    N = row.size
    q = np.zeros((1, 1, N, 1))
    q[0, 0, 0, 0] = 1.0
    k = row.reshape(1, 1, N, 1)
    p = orc.probabilities(q, k, 1.0, False, 0)
    assert int(np.argmax(p[0])) == g["argmax"]
    assert row[int(np.argmax(p[0]))] == g["max"]
    _, lse = orc.attention(q, k, np.ones((1, 1, N, 1)), 1.0, False)
    assert g["max"] <= lse[0, 0, 0] <= g["max"] + math.log(N)


def pin_gqa_equals_repeated_heads(orc):
    """Grouped-query attention is multi-head attention on K/V heads repeated
    H/Hkv times (consecutive query heads share one K/V head); Hkv = H is MHA."""
    r = _rng(31)
    B, H, N, D = 2, 6, 23, 8
    q = r.standard_normal((B, H, N, D))
    for Hkv in (1, 2, 3, 6):
        k = r.standard_normal((B, Hkv, N, D))
        v = r.standard_normal((B, Hkv, N, D))
        krep = np.repeat(k, H // Hkv, axis=1)
        vrep = np.repeat(v, H // Hkv, axis=1)
        for causal in (False, True):
            o, lse = orc.attention_gqa(q, k, v, 0.45, causal)
            o2, lse2 = orc.attention(q, krep, vrep, 0.45, causal)
            _close(o, o2, 0.0, "gqa O Hkv=%d" % Hkv)
            _close(lse, lse2, 0.0, "gqa lse Hkv=%d" % Hkv)
            bh = r.integers(0, B * H, 17)
            ri = r.integers(0, N, 17)
            orow, lrow = orc.attention_rows_gqa(q, k, v, 0.45, causal, bh, ri)
            _close(orow, o.reshape(B * H, N, D)[bh, ri], 0.0, "gqa rows O")
            _close(lrow, lse.reshape(B * H, N)[bh, ri], 0.0, "gqa rows lse")


def pin_gqa_bruteforce(orc):
    """Tiny multi-query case against the 40-digit decimal brute force run per
    query head on its (shared) K/V head."""
    r = _rng(32)
    B, H, Hkv, N, D = 1, 4, 2, 5, 3
    q = r.standard_normal((B, H, N, D))
    k = r.standard_normal((B, Hkv, N, D))
    v = r.standard_normal((B, Hkv, N, D))
    for causal in (False, True):
        o, lse = orc.attention_gqa(q, k, v, 0.7, causal)
        for h in range(H):
            kv = h // (H // Hkv)
            ob, lb, _ = _decimal_attention(q[:, h:h + 1], k[:, kv:kv + 1], v[:, kv:kv + 1], 0.7, causal)
            _close(o[:, h:h + 1], ob, 1e-13, "gqa brute O")
            _close(lse[:, h:h + 1], lb, 1e-13, "gqa brute lse")


# ---------------------------------------------------------------------------
# Backward pass.  The pages give no formulas (the FA2 report only sketches the
# kernel), so the gradients are pinned to the forward definition itself by
# central finite differences, and to closed forms that follow from softmax
# rows summing to one.
# ---------------------------------------------------------------------------
def _loss(orc, q, k, v, dout, scale, causal):
    o, _ = orc.attention(q, k, v, scale, causal)
    return float(np.sum(o * dout))


def pin_bwd_finite_differences(orc):
    """dQ, dK, dV equal the central differences of L = sum(dO * O(Q, K, V))
    computed with the forward oracle (step 1e-6, error O(h^2) + rounding)."""
    r = _rng(41)
    for (N, D, causal) in ((5, 3, False), (6, 2, True), (1, 2, True)):
        q, k, v, do = (r.standard_normal((1, 2, N, D)) for _ in range(4))
        scale = 0.8
        grads = orc.backward(q, k, v, do, scale, causal)
        h = 1e-6
        for t, (x, g) in enumerate(zip((q, k, v), grads)):
            for idx in np.ndindex(x.shape):
                args = [q, k, v]
                xp = x.copy()
                xp[idx] += h
                xm = x.copy()
                xm[idx] -= h
                args[t] = xp
                lp = _loss(orc, *args, do, scale, causal)
                args[t] = xm
                lm = _loss(orc, *args, do, scale, causal)
                fd = (lp - lm) / (2 * h)
                assert abs(fd - g[idx]) <= 1e-7 * (1 + abs(fd)), \
                    ("finite differences", "qkv"[t], idx, causal, fd, g[idx])


def pin_bwd_closed_forms(orc):
    """N = 1: O = V, so dV = dO and dQ = dK = 0.  dO = 0: every gradient is 0.
    Equal value rows: O = v for every row whatever Q and K, so dQ = dK = 0 and
    the dV rows sum to the dO rows' sum (each P row sums to 1)."""
    r = _rng(42)
    q, k, v, do = (r.standard_normal((2, 3, 1, 4)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = orc.backward(q, k, v, do, 0.5, causal)
        _close(dv, do, 1e-15, "N=1 dV")
        _close(dq, np.zeros_like(dq), 1e-15, "N=1 dQ")
        _close(dk, np.zeros_like(dk), 1e-15, "N=1 dK")
    q, k, v = (r.standard_normal((1, 2, 9, 4)) for _ in range(3))
    for causal in (False, True):
        grads = orc.backward(q, k, v, np.zeros_like(q), 0.5, causal)
        for g in grads:
            _close(g, np.zeros_like(g), 0.0, "dO = 0")
    vconst = np.broadcast_to(r.standard_normal((1, 2, 1, 4)), (1, 2, 9, 4)).copy()
    do = r.standard_normal((1, 2, 9, 4))
    for causal in (False, True):
        dq, dk, dv = orc.backward(q, k, vconst, do, 0.5, causal)
        _close(dq, np.zeros_like(dq), 1e-13, "constant V dQ")
        _close(dk, np.zeros_like(dk), 1e-13, "constant V dK")
        _close(dv.sum(axis=2), do.sum(axis=2), 1e-12, "constant V sum dV")


def pin_bwd_invariances(orc):
    """Shifting every key by one vector u changes each score row by a constant,
    so O and every gradient are unchanged; and since each row of dS sums to
    zero, the key gradients of a head sum to zero."""
    r = _rng(43)
    q, k, v, do = (r.standard_normal((2, 2, 13, 5)) for _ in range(4))
    u = r.standard_normal((1, 1, 1, 5))
    for causal in (False, True):
        g0 = orc.backward(q, k, v, do, 0.6, causal)
        g1 = orc.backward(q, k + u, v, do, 0.6, causal)
        for a, b, n in zip(g0, g1, ("dQ", "dK", "dV")):
            _close(a, b, 1e-12, "key shift " + n)
        _close(g0[1].sum(axis=2), np.zeros((2, 2, 5)), 1e-12, "sum_j dK_j")


def pin_bwd_rows_match_full(orc):
    r = _rng(44)
    B, H, N, D = 2, 2, 19, 6
    q, k, v, do = (r.standard_normal((B, H, N, D)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = orc.backward(q, k, v, do, 0.4, causal)
        bh_r, rows = r.integers(0, B * H, 11), r.integers(0, N, 11)
        bh_k, keys = r.integers(0, B * H, 9), r.integers(0, N, 9)
        sq, sk, sv = orc.backward_rows(q, k, v, do, 0.4, causal, bh_r, rows, bh_k, keys)
        _close(sq, dq.reshape(B * H, N, D)[bh_r, rows], 0.0, "rows dQ")
        _close(sk, dk.reshape(B * H, N, D)[bh_k, keys], 0.0, "rows dK")
        _close(sv, dv.reshape(B * H, N, D)[bh_k, keys], 0.0, "rows dV")


def pin_bwd_gqa(orc):
    """Grouped-query backward: Hkv = H is the multi-head backward; otherwise
    dQ equals the multi-head dQ on K/V repeated per group, and the dK, dV of a
    shared head equal the sums of the repeated heads' gradients over the
    group; and on a tiny case, the gradient of a shared key equals central
    differences of the grouped-query forward."""
    r = _rng(45)
    B, H, N, D = 2, 6, 11, 4
    q = r.standard_normal((B, H, N, D))
    do = r.standard_normal((B, H, N, D))
    for Hkv in (1, 2, 3, 6):
        k = r.standard_normal((B, Hkv, N, D))
        v = r.standard_normal((B, Hkv, N, D))
        G = H // Hkv
        for causal in (False, True):
            dq, dk, dv = orc.backward_gqa(q, k, v, do, 0.7, causal)
            rq, rk, rv = orc.backward(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), do, 0.7, causal)
            _close(dq, rq, 1e-12, "gqa dQ Hkv=%d" % Hkv)
            _close(dk, rk.reshape(B, Hkv, G, N, D).sum(axis=2), 1e-12, "gqa dK Hkv=%d" % Hkv)
            _close(dv, rv.reshape(B, Hkv, G, N, D).sum(axis=2), 1e-12, "gqa dV Hkv=%d" % Hkv)
    q, do = r.standard_normal((1, 4, 5, 3)), r.standard_normal((1, 4, 5, 3))
    k, v = r.standard_normal((1, 2, 5, 3)), r.standard_normal((1, 2, 5, 3))
    for causal in (False, True):
        _, dk, dv = orc.backward_gqa(q, k, v, do, 0.8, causal)
        h = 1e-6
        for t, (x, g) in enumerate(((k, dk), (v, dv))):
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = [k, v]
                args_m = [k, v]
                args_p[t], args_m[t] = xp, xm
                lp = float(np.sum(orc.attention_gqa(q, *args_p, 0.8, causal)[0] * do))
                lm = float(np.sum(orc.attention_gqa(q, *args_m, 0.8, causal)[0] * do))
                fd = (lp - lm) / (2 * h)
                assert abs(fd - g[idx]) <= 1e-7 * (1 + abs(fd)), ("gqa finite differences", t, idx, fd, g[idx])


ALL_PINS = [pin_row_sums, pin_ones_v, pin_zero_q, pin_basis_v, pin_shift_invariance,
            pin_single_key, pin_causal_first_rows, pin_permutation, pin_bruteforce,
            pin_rows_match_full, pin_online_matches_definition, pin_golden_dot,
            pin_golden_max_row, pin_gqa_equals_repeated_heads, pin_gqa_bruteforce,
            pin_bwd_finite_differences, pin_bwd_closed_forms, pin_bwd_invariances,
            pin_bwd_rows_match_full, pin_bwd_gqa]
