"""Attention backward (fattn_bwd) against the fp64 oracle's gradients, with
the per-element bound tests/parity.py derives from the kernels' arithmetic."""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_forward_gb300 as fattn
from tiled_attention_forward_gb300.inputs import WORKLOADS, workload_inputs
from tests.parity import bwd_bound_dkdv, bwd_bound_dq, compare_bound, to_f64

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def make(B, H, N, D, dtype, seed, q_std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, N, D, generator=g) * q_std).to(dtype)
    k, v, do = (torch.randn(B, H, N, D, generator=g).to(dtype) for _ in range(3))
    return q, k, v, do


def run_bwd(q, k, v, do, causal, scale):
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fattn.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fattn.bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    return dq, dk, dv


def check_head(q64, k64, v64, do64, o_ref, lse_ref, got, scale, causal, dtype, rows, keys, what,
               dq_ref, dk_ref, dv_ref):
    dq, dk, dv = got
    bq = bwd_bound_dq(q64, k64, v64, do64, o_ref, lse_ref, scale, causal, rows, dtype, dq_ref)
    bk, bv = bwd_bound_dkdv(q64, k64, v64, do64, o_ref, lse_ref, scale, causal, keys, dtype, dk_ref, dv_ref)
    return (compare_bound(dq, dq_ref, bq, what + " dQ"), compare_bound(dk, dk_ref, bk, what + " dK"),
            compare_bound(dv, dv_ref, bv, what + " dV"))


@pytest.mark.parametrize("N", [1, 17, 128, 129, 300])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("fp16", 128), ("fp16", 64)])
def test_bwd_matches_oracle(dtype, D, causal, N):
    B, H = 1, 2
    q, k, v, do = make(B, H, N, D, DT[dtype], 900 + N + D)
    scale = fattn._default_scale(D)
    got = run_bwd(q, k, v, do, causal, scale)
    q64, k64, v64, do64 = (to_f64(t) for t in (q, k, v, do))
    dq_ref, dk_ref, dv_ref = oracle.backward(q64, k64, v64, do64, scale, causal)
    o_ref, lse_ref = oracle.attention(q64, k64, v64, scale, causal)
    allr = np.arange(N)
    for bh in range(B * H):
        b, h = divmod(bh, H)
        check_head(q64[b, h], k64[b, h], v64[b, h], do64[b, h], o_ref[b, h], lse_ref[b, h],
                   tuple(to_f64(g)[b, h] for g in got), scale, causal, DT[dtype], allr, allr,
                   "bwd %s D%d N%d causal=%s head %d" % (dtype, D, N, causal, bh),
                   dq_ref[b, h], dk_ref[b, h], dv_ref[b, h])


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_many_tiles_and_large_scores(causal):
    """Several key blocks and query tiles per head with a ragged tail, and
    std-4 queries (scores up to ~40)."""
    B, H, N, D = 2, 2, 1000, 128
    for q_std in (1.0, 4.0):
        q, k, v, do = make(B, H, N, D, torch.bfloat16, 77, q_std)
        scale = fattn._default_scale(D)
        got = run_bwd(q, k, v, do, causal, scale)
        q64, k64, v64, do64 = (to_f64(t) for t in (q, k, v, do))
        dq_ref, dk_ref, dv_ref = oracle.backward(q64, k64, v64, do64, scale, causal)
        o_ref, lse_ref = oracle.attention(q64, k64, v64, scale, causal)
        allr = np.arange(N)
        for bh in (0, 3):
            b, h = divmod(bh, H)
            check_head(q64[b, h], k64[b, h], v64[b, h], do64[b, h], o_ref[b, h], lse_ref[b, h],
                       tuple(to_f64(g)[b, h] for g in got), scale, causal, torch.bfloat16, allr, allr,
                       "bwd N1000 q_std %g causal=%s head %d" % (q_std, causal, bh),
                       dq_ref[b, h], dk_ref[b, h], dv_ref[b, h])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp16", 64)])
def test_bwd_many_heads(dtype, D, causal):
    """192 heads of 257 rows: 576 CTAs per kernel, several waves of them on
    the 152 SMs, checked on heads spread over the whole range."""
    B, H, N = 4, 48, 257
    q, k, v, do = make(B, H, N, D, DT[dtype], 500 + D)
    scale = fattn._default_scale(D)
    got = run_bwd(q, k, v, do, causal, scale)
    q64, k64, v64, do64 = (to_f64(t) for t in (q, k, v, do))
    dq_ref, dk_ref, dv_ref = oracle.backward(q64, k64, v64, do64, scale, causal)
    o_ref, lse_ref = oracle.attention(q64, k64, v64, scale, causal)
    allr = np.arange(N)
    gots = tuple(to_f64(g) for g in got)
    for bh in list(range(0, B * H, 13)) + [B * H - 1]:
        b, h = divmod(bh, H)
        check_head(q64[b, h], k64[b, h], v64[b, h], do64[b, h], o_ref[b, h], lse_ref[b, h],
                   tuple(g[b, h] for g in gots), scale, causal, DT[dtype], allr, allr,
                   "bwd B4 H48 N257 %s D%d causal=%s head %d" % (dtype, D, causal, bh),
                   dq_ref[b, h], dk_ref[b, h], dv_ref[b, h])


def test_bwd_is_deterministic():
    q, k, v, do = make(1, 3, 777, 64, torch.float16, 5)
    a = run_bwd(q, k, v, do, True, 0.125)
    b = run_bwd(q, k, v, do, True, 0.125)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_argument_errors():
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 64, dtype=torch.float32, device="cuda")
    small = torch.empty(fattn.bwd_workspace_bytes(1, 1, 64) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fattn.FattnError) as e:
        fattn.bwd(q, q.clone(), q.clone(), q.clone(), lse, q.clone(), workspace=small)
    assert e.value.code == 1
    k, v, o, do = (q.clone() for _ in range(4))
    with pytest.raises(fattn.FattnError) as e:  # dK written over dQ
        dq = torch.empty_like(q)
        fattn.bwd(q, k, v, o, lse, do, dq=dq, dk=dq)
    assert e.value.code == 1
    q32 = torch.zeros(1, 1, 64, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(fattn.FattnError) as e:
        fattn.bwd(q32, q32.clone(), q32.clone(), q32.clone(), lse, q32.clone())
    assert e.value.code == 2


SIXTEEN_BIT = [w for w in WORKLOADS if w.torch_dtype != torch.float32]


@pytest.mark.parametrize("w", SIXTEEN_BIT, ids=[w.name for w in SIXTEEN_BIT])
def test_bwd_full_size_sampled(w):
    """The 16-bit workloads at full size with a seeded dO: for the first and
    last head, 48 rows of dQ and 48 rows of dK and dV (first, last and random)
    against the oracle's sampled gradients."""
    q, k, v = workload_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 50)
    do = torch.randn(q.shape, generator=g).to(w.torch_dtype)
    got = run_bwd(q, k, v, do, w.causal, w.scale)
    r = np.random.default_rng(w.seed)
    idx = np.unique(np.concatenate([np.arange(16), np.arange(w.N - 16, w.N), r.integers(0, w.N, 16)]))
    for bh in (0, w.B * w.H - 1):
        b, h = divmod(bh, w.H)
        q64, k64, v64, do64 = (to_f64(t[b:b + 1, h:h + 1]) for t in (q, k, v, do))
        heads = np.zeros(len(idx), np.int64)
        dq_ref, dk_ref, dv_ref = oracle.backward_rows(q64, k64, v64, do64, w.scale, w.causal,
                                                      heads, idx, heads, idx)
        o_ref, lse_ref = oracle.attention(q64, k64, v64, w.scale, w.causal)
        gh = tuple(to_f64(t[b, h])[idx] for t in got)
        check_head(q64[0, 0], k64[0, 0], v64[0, 0], do64[0, 0], o_ref[0, 0], lse_ref[0, 0], gh,
                   w.scale, w.causal, w.torch_dtype, idx, idx, "bwd %s head %d" % (w.name, bh),
                   dq_ref, dk_ref, dv_ref)


def make_gqa(B, H, Hkv, N, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, D, generator=g).to(dtype)
    k = torch.randn(B, Hkv, N, D, generator=g).to(dtype)
    v = torch.randn(B, Hkv, N, D, generator=g).to(dtype)
    do = torch.randn(B, H, N, D, generator=g).to(dtype)
    return q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp16", 64)])
@pytest.mark.parametrize("Hkv", [1, 2])
def test_bwd_gqa_matches_oracle(Hkv, dtype, D, causal):
    """Grouped-query backward: dQ per query head and dK, dV summed over each
    group, against the oracle's grouped-query backward; the bound of a shared
    row is the sum of the per-query-head bounds plus one output rounding."""
    B, H, N = 1, 4, 300
    dt = DT[dtype]
    q, k, v, do = make_gqa(B, H, Hkv, N, D, dt, 60 + Hkv + D)
    scale = fattn._default_scale(D)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fattn.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fattn.bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    assert dk.shape == k.shape and dv.shape == v.shape and dq.shape == q.shape
    q64, k64, v64, do64 = (to_f64(t) for t in (q, k, v, do))
    dq_ref, dk_ref, dv_ref = oracle.backward_gqa(q64, k64, v64, do64, scale, causal)
    o_ref, lse_ref = oracle.attention_gqa(q64, k64, v64, scale, causal)
    G = H // Hkv
    allr = np.arange(N)
    gq, gk, gv = to_f64(dq), to_f64(dk), to_f64(dv)
    for hk in range(Hkv):
        bk = np.zeros((N, D))
        bv = np.zeros((N, D))
        for g in range(G):
            h = hk * G + g
            bq = bwd_bound_dq(q64[0, h], k64[0, hk], v64[0, hk], do64[0, h], o_ref[0, h], lse_ref[0, h],
                              scale, causal, allr, dt, dq_ref[0, h])
            compare_bound(gq[0, h], dq_ref[0, h], bq, "gqa dQ head %d" % h)
            zk, zv = bwd_bound_dkdv(q64[0, h], k64[0, hk], v64[0, hk], do64[0, h], o_ref[0, h],
                                    lse_ref[0, h], scale, causal, allr, dt, np.zeros((N, D)),
                                    np.zeros((N, D)))
            bk += zk
            bv += zv
        from tests.parity import half_ulp
        compare_bound(gk[0, hk], dk_ref[0, hk], bk + half_ulp(dk_ref[0, hk], dt), "gqa dK head %d" % hk)
        compare_bound(gv[0, hk], dv_ref[0, hk], bv + half_ulp(dv_ref[0, hk], dt), "gqa dV head %d" % hk)


def test_bwd_gqa_dq_equals_mha_on_repeated_heads():
    """dQ of a query head depends on its K/V head only, so the grouped-query
    dQ is bit-identical to the multi-head dQ on explicitly repeated K/V."""
    B, H, Hkv, N, D = 1, 8, 2, 400, 128
    q, k, v, do = make_gqa(B, H, Hkv, N, D, torch.bfloat16, 3)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fattn.fwd(qd, kd, vd, causal=True)
    dq1, _, _ = fattn.bwd(qd, kd, vd, o, lse, dod, causal=True)
    kr = kd.repeat_interleave(H // Hkv, dim=1).contiguous()
    vr = vd.repeat_interleave(H // Hkv, dim=1).contiguous()
    dq2, _, _ = fattn.bwd(qd, kr, vr, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    assert torch.equal(dq1, dq2)


@pytest.mark.parametrize("BH", [(1, 3), (2, 4)])
def test_bwd_host_entry_matches_device_entry(BH):
    """The host-buffer backward (groups of heads with overlapped copies)
    gives the device entry's gradients bit for bit, on a non-default stream."""
    B, H = BH
    N, D = 333, 128
    q, k, v, do = make(B, H, N, D, torch.bfloat16, 123)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fattn.fwd(qd, kd, vd, causal=True)
    ref = fattn.bwd(qd, kd, vd, o, lse, dod, causal=True)
    torch.cuda.synchronize()
    hosts = [t.cpu().pin_memory() for t in (q, k, v, o, do, lse)]
    devs = [torch.empty_like(t, device="cuda") for t in hosts]
    grads_h = [torch.full_like(q, float("nan")).pin_memory() for _ in range(3)]
    grads_d = [torch.empty_like(qd) for _ in range(3)]
    ws = torch.empty(fattn.bwd_workspace_bytes(B, H, N), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fattn.bwd_host(hosts, devs, grads_h, grads_d, ws, causal=True, stream=s)
    s.synchronize()
    assert fattn.get_device_status() == 0
    for got, want in zip(grads_h, ref):
        assert torch.equal(got, want.cpu())
