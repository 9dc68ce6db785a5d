"""Comparison of the CUDA path with the fp64 oracle, with the tolerances the
method's target states:

  * bf16 / fp16: max |O - O_ref| <= 1e-2 and mean |O - O_ref| <= 1e-3;
  * fp32:        max |O - O_ref| <= 1e-4;
  * LSE (fp32, natural log): max |LSE - LSE_ref| <= 1e-3.

O is delivered in the input dtype.  Rounding the exact result to bf16 alone
moves it by up to half a bf16 ulp, 2^-7 ~ 0.0078 for |O| in [2, 4) and
2^-6 ~ 0.0156 for |O| in [4, 8), so an element can miss the flat 1e-2 gate
with no error at all before the output rounding.  Such an element is
accepted only where the output rounding explains it:

  * half an ulp of the output dtype at the oracle's value exceeds 2^-8
    (bf16 |O| >= 2, fp16 |O| >= 16; below that the flat gate applies
    unchanged);
  * some value within 1e-2 of the oracle rounds to the delivered value: the
    delivered value's rounding interval (half its ulp on each side) meets
    [O_ref - 1e-2, O_ref + 1e-2];
  * the delivered value is the oracle's own rounding to the output dtype or
    one of its two neighbours.

The number of such elements is counted in the statistics (``n_over_gate``)
and reported.  Asking instead that they lie within 1e-2 of the oracle rounded
to the output dtype cannot work for bf16 |O| in [2, 4): an element more than
1e-2 (> half an ulp) from the oracle never shares its rounding, so its
distance to the rounded oracle is a whole ulp, 2^-6 > 1e-2, whatever the
error before rounding.
"""
import numpy as np
import torch

MANTISSA_BITS = {torch.bfloat16: 7, torch.float16: 10, torch.float32: 23}
MIN_NORMAL_EXP = {torch.bfloat16: -126, torch.float16: -14, torch.float32: -126}
GATE = {torch.bfloat16: 1e-2, torch.float16: 1e-2, torch.float32: 1e-4}

# Statistics of the comparisons a test asks to have reported at the end of the
# run (tests/conftest.py prints them).
REPORTED = []


def ulp(x, dtype):
    """Spacing of `dtype` numbers at |x| (subnormals: the smallest normal spacing)."""
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** MIN_NORMAL_EXP[dtype])))
    return np.exp2(e - MANTISSA_BITS[dtype])


def half_ulp(ref, dtype):
    """Half a unit in the last place of `dtype` at |ref|."""
    return 0.5 * ulp(ref, dtype)


def round_to(x, dtype):
    """x (fp64) rounded to `dtype` and widened back to fp64."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float64)).to(dtype).to(torch.float64).numpy()


def compare(o_gpu, o_ref, lse_gpu, lse_ref, dtype, what="", report=False):
    """Raise AssertionError with statistics if the GPU result misses the gate."""
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.all(np.isfinite(o_gpu)), "%s: non-finite output" % what
    gate = GATE[dtype]
    err = np.abs(o_gpu - o_ref)
    over = err > gate
    stats = dict(n=int(err.size),
                 max_abs=float(err.max()) if err.size else 0.0,
                 mean_abs=float(err.mean()) if err.size else 0.0,
                 n_over_gate=int(over.sum()),
                 worst_ref=float(np.abs(o_ref).ravel()[int(err.argmax())]) if err.size else 0.0)
    if over.any():
        g, r = o_gpu[over], o_ref[over]
        # (0) only where output rounding alone can come near the gate
        unexplained = half_ulp(r, dtype) <= 2.0 ** -8
        # (1) a value within the gate of the oracle rounds to the delivered one
        unexplained |= np.abs(g - r) > gate + half_ulp(g, dtype)
        # (2) the delivered value is the oracle's rounding or a neighbour of it
        off_by = np.abs(g - round_to(r, dtype)) / ulp(g, dtype)
        unexplained |= off_by > 1.0 + 1e-9
        stats["over_gate_max_abs"] = float(np.abs(g - r).max())
        stats["over_gate_max_ulps_from_rounded_oracle"] = float(off_by.max())
        assert not unexplained.any(), "%s: %d elements over the gate not explained by output rounding %s" % (
            what, int(unexplained.sum()), stats)
    if dtype != torch.float32:
        assert stats["mean_abs"] <= 1e-3, "%s: mean abs %s" % (what, stats)
    if lse_gpu is not None:
        lse_gpu = np.asarray(lse_gpu, np.float64)
        lse_ref = np.asarray(lse_ref, np.float64)
        assert np.all(np.isfinite(lse_gpu)), "%s: non-finite LSE" % what
        lerr = float(np.abs(lse_gpu - lse_ref).max()) if lse_gpu.size else 0.0
        stats["lse_max_abs"] = lerr
        assert lerr <= 1e-3, "%s: LSE max abs %.3e" % (what, lerr)
    if report:
        REPORTED.append((what, stats))
    return stats


def to_f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def sample_rows(B, H, N, count, seed, causal):
    """Rows checked on a large problem: every row of the first and last head's
    first and last 64 rows, plus `count` random (head, row) pairs."""
    r = np.random.default_rng(seed)
    bh = [0] * min(N, 64) + [B * H - 1] * min(N, 64)
    rows = list(range(min(N, 64))) + list(range(max(0, N - 64), N))
    bh += [0, B * H - 1] * 2
    rows += [0, 0, N - 1, N - 1]
    bh += list(r.integers(0, B * H, count))
    rows += list(r.integers(0, N, count))
    return np.asarray(bh, np.int64), np.asarray(rows, np.int64)


def workload_rows(B, H, N, per_head, seed):
    """Rows checked on a full-size workload: every row of the first and of the
    last head, plus `per_head` random rows of every head (drawn without
    replacement within the head)."""
    r = np.random.default_rng(seed)
    BH = B * H
    heads = [0] if BH == 1 else [0, BH - 1]
    bh = [np.full(N, h, np.int64) for h in heads]
    rows = [np.arange(N, dtype=np.int64) for _ in heads]
    k = min(per_head, N)
    for h in range(BH):
        if h in heads:
            continue
        bh.append(np.full(k, h, np.int64))
        rows.append(np.sort(r.choice(N, size=k, replace=False)).astype(np.int64))
    return np.concatenate(bh), np.concatenate(rows)


# ---------------------------------------------------------------------------
# Backward pass.  The target states no tolerance for gradients, so the bound
# is derived from the arithmetic of the kernels, per element, from fp64
# quantities of the inputs (never from the CUDA path):
#   * P = exp(s - LSE) in fp32 from the forward's LSE: relative error EPS_P
#     (covers the forward's LSE error and exp2.approx) plus the fp32
#     accumulation of the products (one rounding per 16-deep MMA step);
#   * P (for dV) and dS (for dK, dQ) rounded once to the input dtype:
#     relative U = 2^-8 (bf16) / 2^-11 (fp16), plus the fp16 subnormal
#     spacing 2^-24 absolute;
#   * Delta = dO . O from the 16-bit O: |dDelta_i| <= U sum_c |dO_ic O_ic|;
#   * the result rounded to the output dtype: half an ulp.
# ---------------------------------------------------------------------------
UNIT_ROUNDOFF = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
EPS_P = 1e-4


def _subnormal(dtype):
    """Half the spacing of the output dtype's subnormals (fp16 2^-25)."""
    return 2.0 ** -25 if dtype == torch.float16 else 2.0 ** -134


def _bwd_eps(N):
    return EPS_P + (N / 16.0 + 8.0) * 2.0 ** -24


def _head_terms(q, k, v, do, o, lse, scale, causal, rows, keys):
    """P, dP, dS and Delta on rows x keys of one head (fp64; q,k,v,do,o [N,D])."""
    s = scale * (q[rows] @ k[keys].T)
    p = np.exp(s - lse[rows][:, None])
    if causal:
        p = np.where(np.asarray(keys)[None, :] <= np.asarray(rows)[:, None], p, 0.0)
    dp = do[rows] @ v[keys].T
    delta = np.sum(do[rows] * o[rows], axis=1)
    ds = p * (dp - delta[:, None])
    doo = np.sum(np.abs(do[rows]) * np.abs(o[rows]), axis=1)
    return p, dp, ds, delta, doo


def bwd_bound_dq(q, k, v, do, o, lse, scale, causal, rows, dtype, dq_ref):
    """Per-element bound for dQ rows `rows` of one head ([len(rows), D])."""
    N = q.shape[0]
    u, eps = UNIT_ROUNDOFF[dtype], _bwd_eps(N)
    keys = np.arange(N)
    p, dp, ds, delta, doo = _head_terms(q, k, v, do, o, lse, scale, causal, rows, keys)
    w = (1.05 * u + eps) * np.abs(ds) + p * (u * doo[:, None] + eps * (np.abs(dp) + np.abs(delta)[:, None])) \
        + 2.0 ** -24 * (p > 0)
    return scale * (w @ np.abs(k)) + half_ulp(dq_ref, dtype) + _subnormal(dtype)


def bwd_bound_dkdv(q, k, v, do, o, lse, scale, causal, keys, dtype, dk_ref, dv_ref):
    """Per-element bounds for dK and dV rows `keys` of one head."""
    N = q.shape[0]
    u, eps = UNIT_ROUNDOFF[dtype], _bwd_eps(N)
    rows = np.arange(N)
    p, dp, ds, delta, doo = _head_terms(q, k, v, do, o, lse, scale, causal, rows, keys)
    wk = (1.05 * u + eps) * np.abs(ds) + p * (u * doo[:, None] + eps * (np.abs(dp) + np.abs(delta)[:, None])) \
        + 2.0 ** -24 * (p > 0)
    wv = (1.05 * u + eps) * p + 2.0 ** -24 * (p > 0)
    bk = scale * (wk.T @ np.abs(q)) + half_ulp(dk_ref, dtype) + _subnormal(dtype)
    bv = wv.T @ np.abs(do) + half_ulp(dv_ref, dtype) + _subnormal(dtype)
    return bk, bv


def compare_bound(got, ref, bound, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite" % what
    err = np.abs(got - ref)
    ratio = err / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    assert worst <= 1.0, "%s: %d elements over the bound (worst err/bound %.2f, max err %.3e, max |ref| %.3e)" % (
        what, int((ratio > 1).sum()), worst, float(err.max()), float(np.abs(ref).max()))
    return worst
