"""The materialising comparator (fattn_fwd_unfused: S and P written to a
workspace, O = P V read back) against the fp64 oracle: O and LSE to the same
gate as the fused kernel, and the S and P matrices it leaves in the workspace
against the plain definition."""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_forward_gb300 as fattn
from tiled_attention_forward_gb300.inputs import WORKLOADS, workload_inputs
from tests.parity import MANTISSA_BITS, compare, sample_rows, to_f64

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def make(B, H, N, D, dtype, seed, std=1.0, v_std=1.0):
    """Q, K of standard deviation `std`, V of `v_std` (the absolute gate is
    stated for unit-scale V)."""
    g = torch.Generator().manual_seed(seed)
    return tuple((torch.randn(B, H, N, D, generator=g) * sd).to(DT[dtype])
                 for sd in (std, std, v_std))


def np_pitch(N):
    return (N + 7) // 8 * 8


def test_workspace_size_formula():
    for (B, H, N) in ((1, 1, 1), (2, 3, 17), (4, 16, 4096), (1, 16, 16000)):
        assert fattn.unfused_workspace_bytes(B, H, N) == 6 * B * H * N * np_pitch(N)
    assert fattn.unfused_workspace_bytes(0, 3, 17) == 0


@pytest.mark.parametrize("N", [1, 17, 128, 129, 300, 1000, 1500])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("fp16", 128), ("fp16", 64)])
def test_unfused_matches_oracle(dtype, D, causal, N):
    B, H = 2, 3
    q, k, v = make(B, H, N, D, dtype, 500 + N + D)
    scale = fattn._default_scale(D)
    o, lse = fattn.fwd_unfused(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    o_ref, lse_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    compare(to_f64(o), o_ref, to_f64(lse), lse_ref, DT[dtype],
            "unfused %s D%d N%d causal=%s" % (dtype, D, N, causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_workspace_holds_s_and_p(dtype, causal):
    """S (fp32) is scale * q.k of the 16-bit inputs for every visible pair;
    P (16-bit) is the oracle's probability rounded once, zero for hidden keys
    up to the end of the row's 128-key tile, and each row of P sums to ~1."""
    B, H, N, D = 1, 2, 300, 64
    q, k, v = make(B, H, N, D, dtype, 91, std=2.0)
    scale = fattn._default_scale(D)
    need = fattn.unfused_workspace_bytes(B, H, N)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    fattn.fwd_unfused(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    npch = np_pitch(N)
    s_bytes = B * H * N * npch * 4
    S = ws[:s_bytes].view(torch.float32).view(B * H, N, npch).cpu().double().numpy()
    P = ws[s_bytes:].view(DT[dtype]).view(B * H, N, npch).cpu().double().numpy()
    q64, k64 = to_f64(q).reshape(B * H, N, D), to_f64(k).reshape(B * H, N, D)
    vis = np.tril(np.ones((N, N), bool)) if causal else np.ones((N, N), bool)
    rel = 2.0 ** -(MANTISSA_BITS[DT[dtype]] + 1) + 1e-4
    for bh in range(B * H):
        s_ref = scale * (q64[bh] @ k64[bh].T)
        ds = np.abs(S[bh, :, :N] - s_ref)[vis]
        assert ds.max() <= 1e-5 * np.abs(s_ref[vis]).max() + 1e-5, ds.max()
        p_ref = oracle.probabilities(to_f64(q), to_f64(k), scale, causal, bh=bh)
        # columns of row i the comparator writes (later ones are left untouched)
        ncols = np.array([min(npch, (i // 128 + 1) * 128) if causal else npch for i in range(N)])
        written = np.arange(N)[None, :] < ncols[:, None]
        dp = np.abs(P[bh, :, :N] - p_ref)[written]
        assert np.all(dp <= rel * p_ref[written] + 2.0 ** -24), float(dp.max())
        for i in range(N):
            hidden = P[bh, i, (i + 1 if causal else N):ncols[i]]
            assert np.all(hidden == 0.0), (bh, i)
        row_sums = np.where(written, P[bh, :, :N], 0.0).sum(axis=1)
        assert np.allclose(row_sums, 1.0, atol=N * 2.0 ** -8)


def test_unfused_and_fused_agree_on_large_scores():
    """Scores of magnitude up to ~100 (std-4 Q and K, unit V): the max
    subtraction keeps both paths finite, and both meet the gate."""
    B, H, N, D = 1, 2, 700, 128
    q, k, v = make(B, H, N, D, "bf16", 5, std=4.0)
    scale = fattn._default_scale(D)
    o_ref, lse_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, True)
    for f in (fattn.fwd, fattn.fwd_unfused):
        o, lse = f(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
        torch.cuda.synchronize()
        assert fattn.get_device_status() == 0
        compare(to_f64(o), o_ref, to_f64(lse), lse_ref, torch.bfloat16, f.__name__)


@pytest.mark.parametrize("N", [2100, 16400])
def test_unfused_row_lengths_on_sampled_rows(N):
    """Rows cached in registers in 4 float4 slots per thread (N = 2100) and
    rows longer than the register cache (N = 16400: the two-pass softmax)."""
    B, H, D = 1, 2, 64
    q, k, v = make(B, H, N, D, "bf16", N)
    scale = fattn._default_scale(D)
    for causal in (False, True):
        o, lse = fattn.fwd_unfused(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert fattn.get_device_status() == 0
        bh, rows = sample_rows(B, H, N, 128, 7, causal)
        o_ref, lse_ref = oracle.attention_rows(to_f64(q), to_f64(k), to_f64(v), scale, causal,
                                               bh, rows)
        o = o.reshape(B * H, N, D)
        lse = lse.reshape(B * H, N)
        bt, rt = torch.as_tensor(bh).cuda(), torch.as_tensor(rows).cuda()
        compare(to_f64(o[bt, rt]), o_ref, to_f64(lse[bt, rt]), lse_ref, torch.bfloat16,
                "unfused N%d causal=%s" % (N, causal))


def test_unfused_rejects_small_workspace_and_fp32():
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    small = torch.empty(fattn.unfused_workspace_bytes(1, 1, 64) - 16, dtype=torch.uint8,
                        device="cuda")
    with pytest.raises(fattn.FattnError) as e:
        fattn.fwd_unfused(q, q, q, workspace=small)
    assert e.value.code == 1
    q32 = torch.zeros(1, 1, 64, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(fattn.FattnError) as e:
        fattn.fwd_unfused(q32, q32, q32)
    assert e.value.code == 2


SIXTEEN_BIT = [w for w in WORKLOADS if w.torch_dtype != torch.float32]


@pytest.mark.parametrize("w", SIXTEEN_BIT, ids=[w.name for w in SIXTEEN_BIT])
def test_unfused_full_size_sampled_rows(w):
    q, k, v = workload_inputs(w)
    o, lse = fattn.fwd_unfused(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    o = o.reshape(w.B * w.H, w.N, w.D)
    lse = lse.reshape(w.B * w.H, w.N)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    bh, rows = sample_rows(w.B, w.H, w.N, 256, w.seed + 1, w.causal)
    o_ref, lse_ref = oracle.attention_rows(to_f64(q), to_f64(k), to_f64(v), w.scale, w.causal,
                                           bh, rows)
    bt, rt = torch.as_tensor(bh).cuda(), torch.as_tensor(rows).cuda()
    compare(to_f64(o[bt, rt]), o_ref, to_f64(lse[bt, rt]), lse_ref, w.torch_dtype,
            "unfused " + w.name)
