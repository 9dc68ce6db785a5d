"""Grouped-query / multi-query attention (K/V heads shared by consecutive
query heads) through fattn_fwd_gqa, against the fp64 oracle."""
import pytest
import torch

import oracle
import tiled_attention_forward_gb300 as fattn
from tests.parity import compare, to_f64

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def make(B, H, Hkv, N, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, D, generator=g).to(DT[dtype])
    k = torch.randn(B, Hkv, N, D, generator=g).to(DT[dtype])
    v = torch.randn(B, Hkv, N, D, generator=g).to(DT[dtype])
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp16", 64), ("fp32", 64), ("fp32", 128)])
@pytest.mark.parametrize("Hkv", [1, 2, 4])
def test_gqa_matches_oracle(Hkv, dtype, D, causal):
    B, H, N = 2, 8, 333
    q, k, v = make(B, H, Hkv, N, D, dtype, 40 + Hkv)
    scale = fattn._default_scale(D)
    o, lse = fattn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    o_ref, lse_ref = oracle.attention_gqa(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    compare(to_f64(o), o_ref, to_f64(lse), lse_ref, DT[dtype],
            "gqa H8 Hkv%d %s D%d causal=%s" % (Hkv, dtype, D, causal))


def test_gqa_equals_mha_on_repeated_heads():
    """The kernel's GQA path and its MHA path on explicitly repeated K/V heads
    give bit-identical results (same kernel, same arithmetic)."""
    B, H, Hkv, N, D = 1, 8, 2, 600, 128
    q, k, v = make(B, H, Hkv, N, D, "bf16", 77)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = fattn.fwd(q, k, v, causal=True)
    krep = k.repeat_interleave(H // Hkv, dim=1).contiguous()
    vrep = v.repeat_interleave(H // Hkv, dim=1).contiguous()
    o2, l2 = fattn.fwd(q, krep, vrep, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gqa_bad_grouping_rejected():
    q = torch.zeros(1, 6, 16, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 4, 16, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fattn.FattnError) as e:
        fattn.fwd(q, k, k)
    assert e.value.code == 1
