"""FLOP convention against the numbers the pages print, and the seeded input
generator (CPU only)."""
import json
import os

import pytest
import torch

from tiled_attention_forward_gb300.inputs import WORKLOADS, Workload, make_qkv, workload_inputs


def test_flop_convention_matches_pages(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "flop_convention.json")))
    for c in g["cases"]:
        w = Workload("x", c["B"], c["H"], c["N"], c["D"], "fp16", c["causal"], 0)
        if "gflop_printed" in c:
            assert abs(w.flops() / 1e9 - c["gflop_printed"]) <= c["rel_tol"] * c["gflop_printed"]
        if "tflops_printed" in c:
            tflops = w.flops() / (c["ms"] * 1e-3) / 1e12
            assert abs(tflops - c["tflops_printed"]) <= c["rel_tol"] * c["tflops_printed"]


def test_generator_is_deterministic_and_independent():
    a = make_qkv(1, 2, 33, 64, "bf16", seed=5)
    b = make_qkv(1, 2, 33, 64, "bf16", seed=5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    q, k, v = a
    assert not torch.equal(q, k) and not torch.equal(k, v)
    c = make_qkv(1, 2, 33, 64, "bf16", seed=6)
    assert not torch.equal(a[0], c[0])
    # k of seed s is q of seed s+1 (sub-seeds +0, +1, +2)
    assert torch.equal(a[1], c[0])


def test_generator_dtypes_and_scale():
    q, k, v = make_qkv(1, 1, 64, 64, "fp16", seed=9, q_std=4.0)
    assert q.dtype == torch.float16 and k.dtype == torch.float16
    q1, _, _ = make_qkv(1, 1, 64, 64, "fp32", seed=9, q_std=1.0)
    q4, _, _ = make_qkv(1, 1, 64, 64, "fp32", seed=9, q_std=4.0)
    assert torch.equal(q4, q1 * 4.0)   # power-of-two scaling is exact


def test_workloads_are_the_five_headline_configs():
    names = [w.name for w in WORKLOADS]
    assert len(names) == 5 and len(set(names)) == 5
    assert [w.seed for w in WORKLOADS] == [1000, 1001, 1002, 1003, 1004]
    w = WORKLOADS[2]
    assert (w.B, w.H, w.N, w.D, w.dtype, w.causal) == (4, 16, 4096, 128, "bf16", False)
    assert WORKLOADS[3].q_std == 4.0 and WORKLOADS[3].causal
    for w in WORKLOADS:
        assert abs(w.scale - w.D ** -0.5) < 1e-7
        assert w.scale == float(torch.tensor(w.D ** -0.5, dtype=torch.float32).item())


def test_small_workload_inputs_shape():
    q, k, v = workload_inputs(WORKLOADS[0])
    assert q.shape == (1, 1, 256, 64) and q.dtype == torch.float32


def test_unfused_algorithmic_bytes():
    """bench.py's byte count for the materialising comparator: non-causal, S
    (fp32) and P (16-bit) each written and read once over N x Np per head;
    causal, only the rows' 128-key tiles on or below the diagonal."""
    import bench
    from tiled_attention_forward_gb300.inputs import BY_NAME
    w = BY_NAME["bf16_B4_H16_N4096_D128"]
    assert bench.unfused_bytes(w) == bench.w_bytes(w) + 64 * 4096 * 4096 * (8 + 4)
    w = BY_NAME["fp16_B1_H16_N16000_D64_causal"]
    nt = 125  # 16000 = 125 tiles of 128
    elems = sum(128 * (qt + 1) * 128 for qt in range(nt))
    assert bench.unfused_bytes(w) == bench.w_bytes(w) + 16 * elems * (8 + 4)
    # a causal S/P triangle costs a bit over half of the square
    full = 16000 * 16000
    assert 0.5 < elems / full < 0.51


def test_recorded_traffic_follows_the_kernel_sources():
    """bench.py reports a recorded ncu DRAM figure only while the kernel
    sources it was captured on still hash the same, and null otherwise."""
    import bench
    from tiled_attention_forward_gb300.inputs import BY_NAME
    w = BY_NAME["bf16_B4_H16_N4096_D128"]
    for table, kw in ((bench.NCU_TRAFFIC, {}), (bench.NCU_TRAFFIC_BWD, {"bwd": True}),
                      (bench.NCU_TRAFFIC_UNFUSED, {"unfused": True})):
        value, tag = table[w.name]
        assert bench.ncu_traffic(w, **kw) == (value if tag == bench.kernel_source_hash(
            "bwd" if kw.get("bwd") else ("unfused" if kw.get("unfused") else "tc")) else None)
        saved = table[w.name]
        try:
            table[w.name] = (value, "0" * 16)
            assert bench.ncu_traffic(w, **kw) is None
        finally:
            table[w.name] = saved
    # every recorded figure at least covers the DRAM bytes the workload must move
    for name, (value, _) in bench.NCU_TRAFFIC.items():
        assert value >= 0.8 * bench.w_bytes(BY_NAME[name])


def test_bench_rejects_bad_hkv():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for extra in (["--hkv", "3"], ["--hkv", "16"], ["--hkv", "4", "--impl", "unfused"],
                  ["--hkv", "4", "--workload", "fp32_B4_H8_N8192_D64_causal"]):
        r = subprocess.run([sys.executable, os.path.join(root, "bench.py")] + extra,
                           capture_output=True, text=True, timeout=300)
        assert r.returncode == 2 and "--hkv needs" in r.stderr
