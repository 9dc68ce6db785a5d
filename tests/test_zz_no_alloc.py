"""fattn_fwd_unfused_static: the materialising comparator with its workspace
in the library's fixed per-device array (FATTN_UNFUSED_STATIC_BYTES), so the
call allocates nothing.  Host-side checks run without a GPU; the rest compare
it with the fp64 oracle and with fattn_fwd_unfused on a caller workspace."""
import os
import re

import pytest
import torch

import oracle
import tiled_attention_forward_gb300 as fattn
from tests.parity import compare, sample_rows, to_f64

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, NO_DEVICE = 0, 1, 2, 6
CAP = fattn.UNFUSED_STATIC_BYTES


def pitch(n):
    return (n + 7) // 8 * 8


def largest_n_that_fits():
    n = 1
    while 6 * (n + 1) * pitch(n + 1) <= CAP:
        n += 1
    return n


def call(lib, B=1, H=1, N=16, D=64, dtype=2, q=1 << 40):
    """Fake, never dereferenced, 16-byte aligned and far-apart device pointers."""
    return lib.fattn_fwd_unfused_static(q, 2 << 40, 3 << 40, 4 << 40, None,
                                        B, H, N, D, 0.125, 1, dtype, None)


def test_header_capacity_matches_binding():
    text = open(os.path.join(ROOT, "include", "fattn.h")).read()
    m = re.search(r"#define FATTN_UNFUSED_STATIC_BYTES \((\d+)ll << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == CAP
    assert "fattn_fwd_unfused_static" in text


def test_host_side_rejections():
    lib = fattn.load()
    n = largest_n_that_fits()
    assert 6 * n * pitch(n) <= CAP < 6 * (n + 1) * pitch(n + 1)
    assert call(lib, N=n + 1) == UNSUPPORTED       # workspace over the array
    assert call(lib, B=4, H=16, N=4096) == UNSUPPORTED
    assert call(lib, dtype=0) == UNSUPPORTED                   # fp32: no comparator
    assert call(lib, D=80) == UNSUPPORTED
    assert call(lib, q=None) == INVALID
    assert call(lib, B=0) == OK                                # empty problem


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_a_device():
    assert call(fattn.load()) == NO_DEVICE


def make(B, H, N, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return tuple(torch.randn(B, H, N, D, generator=g).to(dtype) for _ in range(3))


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float16, 64)])
def test_static_matches_oracle_and_caller_workspace(dtype, D, causal):
    B, H, N = 2, 3, 300
    q, k, v = make(B, H, N, D, dtype, 2024 + D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = fattn._default_scale(D)
    o, lse = fattn.fwd_unfused_static(qd, kd, vd, causal=causal, scale=scale)
    o2, lse2 = fattn.fwd_unfused(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    o_ref, lse_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    compare(to_f64(o), o_ref, to_f64(lse), lse_ref, dtype, "static %s D%d" % (dtype, D))


@pytest.mark.gpu
def test_static_largest_problem_and_rejection():
    n = largest_n_that_fits()
    q, k, v = make(1, 1, n, 64, torch.bfloat16, 5)
    scale = fattn._default_scale(64)
    o, lse = fattn.fwd_unfused_static(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    bh, rows = sample_rows(1, 1, n, 128, 3, True)
    o_ref, lse_ref = oracle.attention_rows(to_f64(q), to_f64(k), to_f64(v), scale, True, bh, rows)
    bt, rt = torch.as_tensor(bh).cuda(), torch.as_tensor(rows).cuda()
    compare(to_f64(o.reshape(1, n, 64)[bt, rt]), o_ref, to_f64(lse.reshape(1, n)[bt, rt]), lse_ref,
            torch.bfloat16, "static largest N=%d" % n)
    q2 = torch.zeros(1, 1, n + 1, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fattn.FattnError) as e:
        fattn.fwd_unfused_static(q2, q2, q2)
    assert e.value.code == UNSUPPORTED


@pytest.mark.gpu
def test_static_allocates_nothing_and_reuses_the_array_in_order():
    """After a first call on the device, further calls change neither the
    device's free memory nor torch's allocator; back-to-back calls on one
    stream, which share the array, each give their own correct result."""
    B, H, N, D = 1, 4, 700, 128
    xs = [make(B, H, N, D, torch.bfloat16, s) for s in (11, 12, 13)]
    dev = [tuple(t.cuda() for t in x) for x in xs]
    outs = [torch.empty_like(d[0]) for d in dev]
    lses = [torch.empty((B, H, N), dtype=torch.float32, device="cuda") for _ in dev]
    scale = fattn._default_scale(D)
    fattn.fwd_unfused_static(*dev[0], causal=True, scale=scale, out=outs[0], lse=lses[0])
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0  # every module the status call touches is loaded now
    import gc
    gc.collect()  # garbage of earlier tests must not be released inside the measured window
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for d, o, l in zip(dev, outs, lses):
        fattn.fwd_unfused_static(*d, causal=True, scale=scale, out=o, lse=l)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() <= alloc0  # nothing allocated through torch either
    for x, o, l in zip(xs, outs, lses):
        o_ref, lse_ref = oracle.attention(*(to_f64(t) for t in x), scale, True)
        compare(to_f64(o), o_ref, to_f64(l), lse_ref, torch.bfloat16, "static in order")
