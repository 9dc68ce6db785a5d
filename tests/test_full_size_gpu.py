"""The five named workloads at full size, launched exactly as bench.py times
them, checked on the rows the oracle computes one by one: every row of the
first and of the last head, plus 64 random rows of every head.  The
statistics (including how many elements needed the output-rounding
allowance) are printed at the end of the run."""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_forward_gb300 as fattn
from tiled_attention_forward_gb300.inputs import WORKLOADS, workload_inputs
from tests.parity import compare, to_f64, workload_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_workload_sampled_rows(w):
    q, k, v = workload_inputs(w)
    o, lse = fattn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    o = o.reshape(w.B * w.H, w.N, w.D)
    lse = lse.reshape(w.B * w.H, w.N)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    if w.N * w.B * w.H <= 4096:
        bh = np.repeat(np.arange(w.B * w.H), w.N)
        rows = np.tile(np.arange(w.N), w.B * w.H)
    else:
        bh, rows = workload_rows(w.B, w.H, w.N, 64, w.seed)
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    o_ref, lse_ref = oracle.attention_rows(q64, k64, v64, w.scale, w.causal, bh, rows)
    bt = torch.as_tensor(bh)
    rt = torch.as_tensor(rows)
    got_o = to_f64(o[bt.cuda(), rt.cuda()])
    got_l = to_f64(lse[bt.cuda(), rt.cuda()])
    compare(got_o, o_ref, got_l, lse_ref, w.torch_dtype, w.name, report=True)
