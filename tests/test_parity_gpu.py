"""Parity of the CUDA path (through the C ABI via the binding) with the fp64
oracle on identical seeded inputs.  Small and ragged shapes are compared
element by element; every shape spans several tiles or a ragged tail."""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_forward_gb300 as fattn
from tiled_attention_forward_gb300.inputs import make_qkv
from tests.parity import compare, to_f64

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
N_SET = [1, 17, 127, 128, 129, 255, 256, 257, 383, 1000]


def run_case(B, H, N, D, dtype, causal, seed, q_std=1.0):
    q, k, v = make_qkv(B, H, N, D, dtype, seed, q_std=q_std)
    scale = fattn._default_scale(D)
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = fattn.fwd(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    o_ref, lse_ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    return compare(to_f64(o), o_ref, to_f64(lse), lse_ref, DT[dtype],
                   "B%d H%d N%d D%d %s causal=%s" % (B, H, N, D, dtype, causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("N", N_SET)
def test_tensor_core_small(N, dtype, D, causal):
    run_case(1, 2, N, D, dtype, causal, seed=100 + N)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", N_SET)
def test_ffma_small(N, D, causal):
    run_case(1, 2, N, D, "fp32", causal, seed=200 + N)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp16", 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_tensor_core_many_tasks(dtype, D, causal):
    """More tasks than SMs: every CTA runs several tasks, so barrier phases and
    the K/V ring carry across task boundaries; N=520 leaves a ragged tail."""
    run_case(2, 40, 520, D, dtype, causal, seed=300)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_tensor_core_large_scores(dtype, causal):
    """Q ~ N(0, 16): scores of std 4 make the running max move by large steps,
    exercising the (conditional) O rescale; fp16 also exercises O normalised
    by the sum of the unrounded P while the largest P of a row can exceed 1."""
    run_case(1, 4, 700, 128, dtype, causal, seed=400, q_std=4.0)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_tensor_core_large_scores_d64(dtype, causal):
    """The same at D = 64, where the two Q tiles rotate through three S
    buffers and an O rescale first waits for the tile's previous P.V product;
    B*H*blocks well above the SM count so buffers and phases wrap many times."""
    run_case(2, 24, 700, 64, dtype, causal, seed=410, q_std=4.0)


def test_ffma_many_blocks():
    run_case(2, 3, 1100, 64, "fp32", True, seed=500)


def test_basis_vector_v_probe():
    """V[kk][c0] = 1, else 0  =>  O[:, c0] = P[:, kk] (the hjcheng0602.cn
    flashattn_G7 page's probe, V46): pins the P.V operand layout of V."""
    B, H, N, D = 1, 1, 256, 128
    q, k, _ = make_qkv(B, H, N, D, "bf16", 600)
    scale = fattn._default_scale(D)
    for causal in (False, True):
        p = oracle.probabilities(to_f64(q), to_f64(k), scale, causal, 0)
        for kk, c0 in ((0, 0), (1, 0), (0, 8), (9, 64), (1, 72), (130, 127), (255, 65)):
            v = torch.zeros(B, H, N, D, dtype=torch.bfloat16)
            v[0, 0, kk, c0] = 1.0
            o, _ = fattn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
            o = to_f64(o)[0, 0]
            col = o[:, c0]
            err = np.abs(col - p[:, kk]).max()
            assert err <= 1e-2, (kk, c0, causal, err)
            others = np.delete(o, c0, axis=1)
            assert np.abs(others).max() == 0.0, (kk, c0, "leaked into other columns")


def test_outputs_do_not_spill_and_every_row_is_written():
    """Guard bands around O and LSE stay untouched; a NaN pre-fill of O and
    LSE is fully overwritten (no row left unwritten)."""
    for dtype, D, N, causal in (("bf16", 128, 200, True), ("fp16", 64, 383, False),
                                ("fp32", 64, 200, True)):
        B, H = 1, 3
        q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, dtype, 700))
        td = DT[dtype]
        n = B * H * N * D
        guard = 4096
        big = torch.full((n + 2 * guard,), 7.0, dtype=td, device="cuda")
        out = big[guard:guard + n].view(B, H, N, D)
        out.fill_(float("nan"))
        lbig = torch.full((B * H * N + 2 * guard,), 7.0, dtype=torch.float32, device="cuda")
        lse = lbig[guard:guard + B * H * N].view(B, H, N)
        lse.fill_(float("nan"))
        fattn.fwd(q, k, v, causal=causal, out=out, lse=lse)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
        assert (big[:guard] == 7.0).all() and (big[guard + n:] == 7.0).all()
        assert (lbig[:guard] == 7.0).all() and (lbig[guard + B * H * N:] == 7.0).all()


def test_deterministic():
    q, k, v = (t.cuda() for t in make_qkv(2, 4, 777, 128, "bf16", 800))
    o1, l1 = fattn.fwd(q, k, v, causal=True)
    o2, l2 = fattn.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lse_optional():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 300, 64, "fp16", 900))
    o1, _ = fattn.fwd(q, k, v, causal=True)
    o2, none = fattn.fwd(q, k, v, causal=True, return_lse=False)
    torch.cuda.synchronize()
    assert none is None and torch.equal(o1, o2)


def test_host_buffer_entry_point_matches_device_entry_point():
    for dtype, D in (("bf16", 128), ("fp32", 64)):
        B, H, N = 1, 2, 300
        q, k, v = make_qkv(B, H, N, D, dtype, 1000)
        pin = [t.pin_memory() for t in (q, k, v)]
        dev = [torch.empty_like(t, device="cuda") for t in (q, k, v)]
        o_dev = torch.empty_like(dev[0])
        lse_dev = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        o_host = torch.empty_like(q).pin_memory()
        lse_host = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        fattn.fwd_host(*pin, *dev, o_dev, o_host, lse_dev, lse_host, causal=True)
        torch.cuda.synchronize()
        o_ref, l_ref = fattn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o_host, o_ref.cpu()) and torch.equal(lse_host, l_ref.cpu())


@pytest.mark.parametrize("BH", [(1, 1), (1, 3), (2, 5), (4, 16)])
def test_host_entry_point_chunked_and_ordered(BH):
    """The host entry splits the heads into up to four groups on internal
    copy streams: results match the device entry bit for bit for head counts
    below, at and above the group count, with and without LSE, on a
    non-default stream, and later work on that stream sees O and LSE."""
    B, H = BH
    N, D = 333, 64
    q, k, v = make_qkv(B, H, N, D, "fp16", 77)
    pin = [t.pin_memory() for t in (q, k, v)]
    dev = [torch.empty_like(t, device="cuda") for t in (q, k, v)]
    o_dev = torch.empty_like(dev[0])
    lse_dev = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    o_ref, l_ref = fattn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=False)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    for with_lse in (True, False):
        o_host = torch.full_like(q, float("nan")).pin_memory()
        lse_host = torch.full((B, H, N), float("nan"), dtype=torch.float32).pin_memory()
        o_dev.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            fattn.fwd_host(*pin, *dev, o_dev, o_host, lse_dev if with_lse else None,
                           lse_host if with_lse else None, causal=False, stream=s)
            o_copy = o_dev.clone()  # enqueued after the call on the same stream
        s.synchronize()
        assert fattn.get_device_status() == 0
        assert torch.equal(o_host, o_ref.cpu())
        assert torch.equal(o_copy, o_ref)
        if with_lse:
            assert torch.equal(lse_host, l_ref.cpu())


def test_empty_inputs():
    q = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = fattn.fwd(q, q, q)
    assert o.shape == q.shape and lse.shape == (1, 2, 0)


def test_bad_arguments_raise():
    q = torch.zeros(1, 1, 16, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fattn.FattnError) as e:
        fattn.fwd(q, q, q)
    assert e.value.code == 2
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fattn.FattnError):
        fattn.fwd(q, q, q, out=q)  # O may not alias the inputs
