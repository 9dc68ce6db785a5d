"""Seeded random shapes through the forward (all three dtypes) and the
backward (16-bit), against the fp64 oracle: a sweep beyond the hand-picked
edge cases, over batch, heads, grouped K/V heads, ragged lengths, head dims,
causal masking and query scales."""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_forward_gb300 as fattn
from tests.parity import bwd_bound_dkdv, bwd_bound_dq, compare, compare_bound, half_ulp, to_f64

pytestmark = pytest.mark.gpu

DTYPES = [torch.bfloat16, torch.float16, torch.float32]


def draw(seed):
    r = np.random.default_rng(9000 + seed)
    dtype = DTYPES[seed % 3]
    B = int(r.integers(1, 4))
    Hkv = int(r.integers(1, 4))
    H = Hkv * int(r.integers(1, 3))
    N = int(r.integers(1, 700))
    D = int(r.choice([64, 128]))
    causal = bool(r.integers(0, 2))
    q_std = float(r.choice([1.0, 2.0, 4.0]))
    return dtype, B, H, Hkv, N, D, causal, q_std


@pytest.mark.parametrize("seed", range(24))
def test_random_forward(seed):
    dtype, B, H, Hkv, N, D, causal, q_std = draw(seed)
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, N, D, generator=g) * q_std).to(dtype)
    k = torch.randn(B, Hkv, N, D, generator=g).to(dtype)
    v = torch.randn(B, Hkv, N, D, generator=g).to(dtype)
    scale = fattn._default_scale(D)
    o, lse = fattn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    o_ref, lse_ref = oracle.attention_gqa(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    compare(to_f64(o), o_ref, to_f64(lse), lse_ref, dtype,
            "random fwd %s B%d H%d Hkv%d N%d D%d causal=%s q_std=%g" % (dtype, B, H, Hkv, N, D, causal, q_std))


@pytest.mark.parametrize("seed", [s for s in range(24) if s % 3 != 2][:12])
def test_random_backward(seed):
    dtype, B, H, Hkv, N, D, causal, q_std = draw(seed)
    g = torch.Generator().manual_seed(seed + 100)
    q = (torch.randn(B, H, N, D, generator=g) * min(q_std, 2.0)).to(dtype)
    k = torch.randn(B, Hkv, N, D, generator=g).to(dtype)
    v = torch.randn(B, Hkv, N, D, generator=g).to(dtype)
    do = torch.randn(B, H, N, D, generator=g).to(dtype)
    scale = fattn._default_scale(D)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fattn.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fattn.bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    q64, k64, v64, do64 = (to_f64(t) for t in (q, k, v, do))
    dq_ref, dk_ref, dv_ref = oracle.backward_gqa(q64, k64, v64, do64, scale, causal)
    o_ref, lse_ref = oracle.attention_gqa(q64, k64, v64, scale, causal)
    G = H // Hkv
    allr = np.arange(N)
    gq, gk, gv = to_f64(dq), to_f64(dk), to_f64(dv)
    what = "random bwd %s B%d H%d Hkv%d N%d D%d causal=%s" % (dtype, B, H, Hkv, N, D, causal)
    for b in range(B):
        for hk in range(Hkv):
            bk = np.zeros((N, D))
            bv = np.zeros((N, D))
            for gi in range(G):
                h = hk * G + gi
                args = (q64[b, h], k64[b, hk], v64[b, hk], do64[b, h], o_ref[b, h], lse_ref[b, h], scale, causal)
                compare_bound(gq[b, h], dq_ref[b, h], bwd_bound_dq(*args, allr, dtype, dq_ref[b, h]), what + " dQ")
                zk, zv = bwd_bound_dkdv(*args, allr, dtype, np.zeros((N, D)), np.zeros((N, D)))
                bk += zk
                bv += zv
            compare_bound(gk[b, hk], dk_ref[b, hk], bk + half_ulp(dk_ref[b, hk], dtype), what + " dK")
            compare_bound(gv[b, hk], dv_ref[b, hk], bv + half_ulp(dv_ref[b, hk], dtype), what + " dV")
