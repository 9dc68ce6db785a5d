"""Parity of fattn_fwd_f32_rowwise (the fp32 kernel with one query row per
thread) with the fp64 oracle: small and ragged shapes element by element,
the fp32 named workloads at full size on sampled rows, and its agreement
with fattn_fwd's own fp32 kernel."""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_forward_gb300 as fattn
from tiled_attention_forward_gb300.inputs import WORKLOADS, make_qkv, workload_inputs
from tests.parity import compare, to_f64, workload_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", [1, 17, 129, 257, 1000])
def test_rowwise_small(N, D, causal):
    B, H = 1, 2
    q, k, v = make_qkv(B, H, N, D, "fp32", seed=700 + N)
    scale = fattn._default_scale(D)
    o, lse = fattn.fwd_f32_rowwise(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    o_ref, lse_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    compare(to_f64(o), o_ref, to_f64(lse), lse_ref, torch.float32,
            "rowwise N%d D%d causal=%s" % (N, D, causal))


FP32_WORKLOADS = [w for w in WORKLOADS if w.dtype == "fp32"]


@pytest.mark.parametrize("w", FP32_WORKLOADS, ids=[w.name for w in FP32_WORKLOADS])
def test_rowwise_workload_sampled_rows(w):
    q, k, v = workload_inputs(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fattn.fwd_f32_rowwise(qd, kd, vd, causal=w.causal, scale=w.scale)
    o_t, lse_t = fattn.fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    o = o.reshape(w.B * w.H, w.N, w.D)
    lse = lse.reshape(w.B * w.H, w.N)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    # the two fp32 kernels differ only in summation order
    assert (o - o_t.reshape_as(o)).abs().max().item() <= 1e-5
    assert (lse - lse_t.reshape_as(lse)).abs().max().item() <= 1e-5
    if w.N * w.B * w.H <= 4096:
        bh = np.repeat(np.arange(w.B * w.H), w.N)
        rows = np.tile(np.arange(w.N), w.B * w.H)
    else:
        bh, rows = workload_rows(w.B, w.H, w.N, 64, w.seed)
    o_ref, lse_ref = oracle.attention_rows(to_f64(q), to_f64(k), to_f64(v), w.scale, w.causal,
                                           bh, rows)
    bt, rt = torch.as_tensor(bh).cuda(), torch.as_tensor(rows).cuda()
    compare(to_f64(o[bt, rt]), o_ref, to_f64(lse[bt, rt]), lse_ref, torch.float32,
            "rowwise " + w.name, report=True)


def test_rowwise_rejects_other_dtypes():
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fattn.fwd_f32_rowwise(q, q, q)
