"""The persistent grid's task schedule: CTAs take tasks from a per-launch
counter, and causal problems run their heads in groups whose K/V fits in L2.

What is checked: head groups that do not divide the head count (and grouped
K/V heads) against the oracle on sampled rows; the counter state left by one
launch does not disturb the next (many launches in a row, bit-identical);
launches running at the same time on several streams each get their own
counter (bit-identical to the same problems run one after another)."""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_forward_gb300 as fattn
from tests.parity import compare, to_f64

pytestmark = pytest.mark.gpu


def make(B, H, Hkv, N, D, dtype, seed, q_std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, N, D, generator=g) * q_std).to(dtype)
    k = torch.randn(B, Hkv, N, D, generator=g).to(dtype)
    v = torch.randn(B, Hkv, N, D, generator=g).to(dtype)
    return q, k, v


def sampled_rows(BH, N, per_head, seed):
    """The first and last 8 rows of every head and `per_head` random ones."""
    rng = np.random.default_rng(seed)
    bh, rows = [], []
    for h in range(BH):
        r = np.unique(np.concatenate([np.arange(8), np.arange(N - 8, N),
                                      rng.integers(0, N, per_head)]))
        bh.append(np.full(r.size, h))
        rows.append(r)
    return np.concatenate(bh).astype(np.int64), np.concatenate(rows).astype(np.int64)


@pytest.mark.parametrize("B,H,Hkv,N,D,dtype", [
    # 21 heads of 4 MiB K/V: two groups of 11 and 10 heads
    (3, 7, 7, 8192, 128, torch.bfloat16),
    # 16 query heads on 8 K/V heads of 8 MiB: two groups of 8 query heads
    (1, 16, 8, 32768, 64, torch.float16),
])
def test_grouped_causal_order(B, H, Hkv, N, D, dtype):
    q, k, v = make(B, H, Hkv, N, D, dtype, 900 + H, q_std=2.0)
    scale = fattn._default_scale(D)
    o, lse = fattn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    o = o.reshape(B * H, N, D)
    lse = lse.reshape(B * H, N)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    bh, rows = sampled_rows(B * H, N, 24, 17)
    o_ref, lse_ref = oracle.attention_rows_gqa(to_f64(q), to_f64(k), to_f64(v), scale, True, bh,
                                               rows)
    bt, rt = torch.as_tensor(bh).cuda(), torch.as_tensor(rows).cuda()
    compare(to_f64(o[bt, rt]), o_ref, to_f64(lse[bt, rt]), lse_ref, dtype,
            "grouped causal B%d H%d Hkv%d N%d D%d" % (B, H, Hkv, N, D))


def test_counter_left_clean_across_launches():
    q, k, v = (t.cuda() for t in make(2, 12, 12, 4096, 128, torch.bfloat16, 31))
    o0, l0 = fattn.fwd(q, k, v, causal=True)
    for _ in range(40):
        o, l = fattn.fwd(q, k, v, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o, o0) and torch.equal(l, l0)
    assert fattn.get_device_status() == 0


def test_concurrent_launches_on_streams():
    probs = [
        (make(2, 16, 16, 4096, 128, torch.bfloat16, 41), True),
        (make(1, 16, 16, 8000, 64, torch.float16, 42), True),
        (make(4, 8, 8, 2048, 128, torch.float16, 43), False),
        (make(1, 24, 24, 4096, 64, torch.bfloat16, 44), True),
    ]
    probs = [(tuple(t.cuda() for t in qkv), c) for qkv, c in probs]
    ref = []
    for (q, k, v), c in probs:
        ref.append(fattn.fwd(q, k, v, causal=c))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in probs]
    outs = [[] for _ in probs]
    for _ in range(5):
        for i, (((q, k, v), c), s) in enumerate(zip(probs, streams)):
            with torch.cuda.stream(s):
                outs[i].append(fattn.fwd(q, k, v, causal=c, stream=s))
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    for r, got in zip(ref, outs):
        for o, l in got:
            assert torch.equal(o, r[0]) and torch.equal(l, r[1])
