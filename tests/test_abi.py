"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/fattn.h declares, rejects bad arguments before touching CUDA, and
plans launches with the tile arithmetic the pages print."""
import ctypes
import json
import os
import re

import pytest
import torch

import tiled_attention_forward_gb300 as fattn
from tiled_attention_forward_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fattn.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA_ERR, TIMEOUT, NO_DEVICE = range(7)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fbuild.LIB):
        fbuild.build()
    return fattn.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FATTN_API\s+[\w\s\*]*?\b(fattn_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("fattn_fwd", "fattn_fwd_gqa", "fattn_fwd_host", "fattn_plan",
                 "fattn_get_device_status", "fattn_selftest_wait_timeout",
                 "fattn_fwd_unfused", "fattn_unfused_workspace_bytes",
                 "fattn_bwd", "fattn_bwd_gqa", "fattn_bwd_workspace_bytes",
                 "fattn_fwd_f32_rowwise", "fattn_status_string", "fattn_version"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for code, name in fattn.STATUS.items():
        assert fattn.status_string(code) == name
    assert fattn.status_string(99) == "FATTN_ERR_UNKNOWN"
    assert lib.fattn_version() == 10000


FAKE = 1 << 20  # a 16-byte aligned non-null address that is never dereferenced


def call_fwd(lib, q=FAKE, k=FAKE + (1 << 16), v=FAKE + (2 << 16), o=FAKE + (3 << 16), lse=None,
             B=1, H=1, N=16, D=64, scale=0.125, causal=0, dtype=2):
    return lib.fattn_fwd(q, k, v, o, lse, B, H, N, D, scale, causal, dtype, None)


def test_argument_errors_before_any_cuda_call(lib):
    assert call_fwd(lib, q=None) == INVALID
    assert call_fwd(lib, o=None) == INVALID
    assert call_fwd(lib, B=-1) == INVALID
    assert call_fwd(lib, N=-5) == INVALID
    assert call_fwd(lib, dtype=7) == INVALID
    assert call_fwd(lib, scale=float("nan")) == INVALID
    assert call_fwd(lib, scale=float("inf")) == INVALID
    assert call_fwd(lib, scale=-1.0) == INVALID
    assert call_fwd(lib, D=96) == UNSUPPORTED
    assert call_fwd(lib, D=256) == UNSUPPORTED
    assert call_fwd(lib, q=FAKE + 8) == MISALIGNED
    assert call_fwd(lib, o=FAKE + (3 << 16) + 2) == MISALIGNED
    assert call_fwd(lib, lse=FAKE + (4 << 16) + 1) == MISALIGNED
    # O overlapping an input, LSE overlapping O
    assert call_fwd(lib, o=FAKE + 16) == INVALID
    assert call_fwd(lib, lse=FAKE + (3 << 16) + 64) == INVALID
    # index range limits
    assert call_fwd(lib, N=(1 << 30) + 1) == UNSUPPORTED
    assert call_fwd(lib, B=1 << 16, H=1 << 16) == UNSUPPORTED
    assert call_fwd(lib, B=70000, H=1, dtype=0) == UNSUPPORTED
    # B*H*N*D past 2^52 elements (each of N and B*H within its own limit): the
    # byte counts of the overlap checks would overflow int64 otherwise
    assert call_fwd(lib, B=1 << 15, H=1 << 15, N=1 << 30, D=128) == UNSUPPORTED
    assert call_fwd(lib, B=1, H=1 << 20, N=1 << 30, D=64) == UNSUPPORTED
    # more than 2^30 tensor-core tasks (256-row Q blocks x heads), buffers far
    # apart so that no overlap check fires first
    far = dict(q=1 << 20, k=1 << 48, v=1 << 49, o=1 << 50)
    assert call_fwd(lib, B=1, H=1 << 9, N=1 << 30, D=64, **far) == UNSUPPORTED


def test_rowwise_argument_errors(lib):
    def rw(q=FAKE, k=FAKE + (1 << 16), v=FAKE + (2 << 16), o=FAKE + (3 << 16), lse=None,
           B=1, H=1, N=16, D=64, scale=0.125):
        return lib.fattn_fwd_f32_rowwise(q, k, v, o, lse, B, H, N, D, scale, 0, None)
    assert rw(q=None) == INVALID
    assert rw(N=-1) == INVALID
    assert rw(scale=float("nan")) == INVALID
    assert rw(D=96) == UNSUPPORTED
    assert rw(B=70000) == UNSUPPORTED      # grid.y limit of the fp32 launch
    assert rw(k=FAKE + (1 << 16) + 4) == MISALIGNED
    assert rw(o=FAKE + 32) == INVALID       # O over Q
    assert rw(B=0) == OK
    assert rw(N=0) == OK


def test_gqa_argument_errors(lib):
    def gqa(H=8, Hkv=2, **kw):
        args = dict(q=FAKE, k=FAKE + (1 << 16), v=FAKE + (2 << 16), o=FAKE + (3 << 16), lse=None,
                    B=1, N=16, D=64, scale=0.125, causal=0, dtype=2)
        args.update(kw)
        return lib.fattn_fwd_gqa(args["q"], args["k"], args["v"], args["o"], args["lse"],
                                 args["B"], H, Hkv, args["N"], args["D"], args["scale"],
                                 args["causal"], args["dtype"], None)
    assert gqa(Hkv=0) == INVALID
    assert gqa(Hkv=-1) == INVALID
    assert gqa(Hkv=3) == INVALID          # 8 % 3 != 0
    assert gqa(Hkv=16) == INVALID         # more K/V heads than query heads
    assert gqa(D=80) == UNSUPPORTED
    assert gqa(H=0, Hkv=0) == OK          # empty problem
    # O overlapping the (smaller) K tensor
    assert gqa(o=FAKE + (1 << 16) + 64) == INVALID


def test_unfused_workspace_bytes(lib):
    pitch = lambda n: (n + 7) // 8 * 8
    for (B, H, N) in ((1, 1, 1), (2, 3, 17), (4, 16, 4096), (1, 16, 16000), (2, 32, 8192)):
        assert lib.fattn_unfused_workspace_bytes(B, H, N) == 6 * B * H * N * pitch(N)
    for (B, H, N) in ((0, 1, 1), (1, 0, 1), (1, 1, 0), (-1, 1, 1), (1 << 31, 1, 1 << 20)):
        assert lib.fattn_unfused_workspace_bytes(B, H, N) == 0


def test_bwd_workspace_and_argument_errors(lib):
    for (B, H, N) in ((1, 1, 1), (2, 3, 129), (4, 16, 4096), (1, 16, 16000)):
        assert lib.fattn_bwd_workspace_bytes(B, H, N) == 8 * B * H * (-(-N // 128) * 128)
    assert lib.fattn_bwd_workspace_bytes(0, 1, 1) == 0
    T = 1 << 40  # far-apart fake device addresses, never dereferenced

    def bwd(q=T, k=2 * T, v=3 * T, o=4 * T, do=5 * T, lse=6 * T, dq=7 * T, dk=8 * T, dv=9 * T,
            ws=10 * T, wsb=None, B=1, H=2, N=16, D=64, dtype=2):
        if wsb is None:
            wsb = lib.fattn_bwd_workspace_bytes(B, H, N)
        return lib.fattn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, wsb, B, H, N, D, 0.125, 1,
                             dtype, None)
    assert bwd(dtype=0) == UNSUPPORTED
    assert bwd(D=96) == UNSUPPORTED
    assert bwd(do=None) == INVALID
    assert bwd(lse=None) == INVALID
    assert bwd(ws=None) == INVALID
    assert bwd(wsb=100) == INVALID
    assert bwd(dk=8 * T + 8) == MISALIGNED
    assert bwd(lse=6 * T + 2) == MISALIGNED
    assert bwd(dk=7 * T) == INVALID          # dK over dQ
    assert bwd(dv=4 * T) == INVALID          # dV over O
    assert bwd(ws=2 * T) == INVALID          # workspace over K
    assert bwd(B=0) == OK

    def bwd_gqa(Hkv, H=4, dk=8 * T, **kw):
        return lib.fattn_bwd_gqa(T, 2 * T, 3 * T, 4 * T, 5 * T, 6 * T, 7 * T, dk, 9 * T, 10 * T,
                                 1 << 30, 1, H, Hkv, 16, 64, 0.125, 0, 2, None)
    assert bwd_gqa(Hkv=3) == INVALID       # 4 % 3 != 0
    assert bwd_gqa(Hkv=0) == INVALID
    assert bwd_gqa(Hkv=8) == INVALID       # more K/V heads than query heads


def test_unfused_argument_errors(lib):
    WS = FAKE + (8 << 20)

    def unf(ws=WS, wsb=None, B=1, H=2, N=16, D=64, dtype=2, **kw):
        args = dict(q=FAKE, k=FAKE + (1 << 16), v=FAKE + (2 << 16), o=FAKE + (3 << 16), lse=None)
        args.update(kw)
        if wsb is None:
            wsb = lib.fattn_unfused_workspace_bytes(B, H, N)
        return lib.fattn_fwd_unfused(args["q"], args["k"], args["v"], args["o"], args["lse"],
                                     ws, wsb, B, H, N, D, 0.125, 0, dtype, None)
    assert unf(dtype=0) == UNSUPPORTED                  # fp32 has no comparator
    assert unf(D=96) == UNSUPPORTED
    assert unf(ws=None) == INVALID
    assert unf(wsb=100) == INVALID                      # smaller than needed
    assert unf(ws=WS + 4) == MISALIGNED
    assert unf(ws=FAKE + (2 << 16)) == INVALID          # overlaps v
    far = dict(q=1 << 40, k=2 << 40, v=3 << 40, o=4 << 40, ws=5 << 40, wsb=1 << 40)
    assert unf(B=70000, H=1, **far) == UNSUPPORTED      # grid limit on B*H
    assert unf(B=0) == OK                               # empty problem
    assert unf(q=None) == INVALID


def test_empty_problem_is_ok_and_enqueues_nothing(lib):
    for (B, H, N) in ((0, 4, 16), (2, 0, 16), (2, 4, 0)):
        assert call_fwd(lib, q=None, k=None, v=None, o=None, B=B, H=H, N=N) == OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_a_device_reports_no_device(lib):
    assert call_fwd(lib) == NO_DEVICE
    assert call_fwd(lib, dtype=0) == NO_DEVICE
    T = 1 << 40
    assert lib.fattn_bwd(T, 2 * T, 3 * T, 4 * T, 5 * T, 6 * T, 7 * T, 8 * T, 9 * T, 10 * T, 1 << 20,
                         1, 1, 16, 64, 0.125, 0, 2, None) == NO_DEVICE
    ws = FAKE + (8 << 20)
    assert lib.fattn_fwd_unfused(FAKE, FAKE + (1 << 16), FAKE + (2 << 16), FAKE + (3 << 16), None,
                                 ws, 1 << 20, 1, 1, 16, 64, 0.125, 1, 2, None) == NO_DEVICE
    assert lib.fattn_selftest_wait_timeout(1000, None) == NO_DEVICE
    assert lib.fattn_selftest_wait_timeout(0, None) == INVALID


def test_host_entry_point_argument_errors(lib):
    args = [FAKE, FAKE, FAKE, FAKE + (5 << 16), None,
            FAKE, FAKE + (1 << 16), FAKE + (2 << 16), FAKE + (3 << 16), None,
            1, 1, 16, 64, 0.125, 0, 2, None]
    bad = list(args)
    bad[0] = None
    assert lib.fattn_fwd_host(*bad) == INVALID
    bad = list(args)
    bad[8] = None
    assert lib.fattn_fwd_host(*bad) == INVALID
    bad = list(args)
    bad[13] = 80
    assert lib.fattn_fwd_host(*bad) == UNSUPPORTED


def test_plan_ffma_matches_page_tile_arithmetic(lib, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tile_arithmetic.json")))
    grid = g["cases"][0]
    # fp32 path: grid = (ceil(N/Br), B*H) with Br = 128 (the page's grid); the
    # CTA spreads its 128 rows over 256 threads, in K/V tiles of 64 keys
    p = fattn.plan(4, 8, grid["N"], 64, causal=False, dtype=torch.float32, num_sms=152)
    assert p["path"] == 1
    assert (p["grid_x"], p["grid_y"]) == (grid["grid_x"], grid["grid_y"])
    assert p["grid_x"] * p["grid_y"] == grid["blocks"]
    assert p["rows_per_task"] == grid["Br"]
    assert p["threads"] == 256 and p["keys_per_kv_tile"] == 64
    nvec = g["cases"][1]
    assert nvec["Bc"] * nvec["D"] * nvec["elem_bytes"] // 16 == nvec["nvec"]
    # non-causal: every Q block visits every K/V tile
    assert p["kv_tiles"] == 64 * 32 * (8192 // p["keys_per_kv_tile"])


def causal_tiles_per_block(N, Br, Bc):
    # Q block qb visits ceil(min((qb+1)*Br, N)/Bc) K/V tiles
    return [-(-min((qb + 1) * Br, N) // Bc) for qb in range(-(-N // Br))]


def test_plan_causal_skip_counts(lib, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tile_arithmetic.json")))["cases"][2]
    N, Br, Bc = g["N"], g["Br"], g["Bc"]
    # the page's worked numbers: with Bc = 32, block 5 visits 24 tiles and skips 40
    per_block = causal_tiles_per_block(N, Br, Bc)
    assert per_block[g["q_block"]] == g["tiles_visited"]
    assert N // Bc - per_block[g["q_block"]] == g["tiles_skipped"]
    p = fattn.plan(1, 1, N, 64, causal=True, dtype=torch.float32, num_sms=152)
    assert p["kv_tiles"] == sum(causal_tiles_per_block(N, Br, p["keys_per_kv_tile"]))
    p = fattn.plan(1, 1, 1000, 128, causal=True, dtype=torch.float32, num_sms=152)
    assert p["kv_tiles"] == sum(causal_tiles_per_block(1000, 128, p["keys_per_kv_tile"]))


def test_plan_tensor_core_path(lib):
    p = fattn.plan(4, 16, 4096, 128, causal=False, dtype=torch.bfloat16, num_sms=152)
    assert p["path"] == 2
    assert p["tasks"] == 4 * 16 * (4096 // 256)
    assert p["grid_x"] == 152 and p["grid_y"] == 1
    assert p["rows_per_task"] == 256 and p["keys_per_kv_tile"] == 128
    assert p["kv_tiles"] == p["tasks"] * (4096 // 128)
    assert p["smem_bytes"] <= 227 * 1024
    # causal N=16000: the last task's second Q tile starts at row 16000 (empty)
    p = fattn.plan(1, 16, 16000, 64, causal=True, dtype=torch.float16, num_sms=152)
    nq = -(-16000 // 256)
    assert p["tasks"] == 16 * nq
    tiles = sum(max(min(qb * 256 + 128, 16000) // 128 if qb * 256 < 16000 else 0,
                    (-(-min(qb * 256 + 256, 16000) // 128)) if qb * 256 + 128 < 16000 else 0)
                for qb in range(nq))
    assert p["kv_tiles"] == 16 * tiles
    # few tasks: one CTA per task
    p = fattn.plan(1, 1, 256, 64, causal=False, dtype=torch.bfloat16, num_sms=152)
    assert p["tasks"] == 1 and p["grid_x"] == 1


def test_plan_errors(lib):
    with pytest.raises(fattn.FattnError):
        fattn.plan(1, 1, 16, 80)
    assert fattn.plan(0, 1, 16, 64, num_sms=152)["path"] == 0


def test_product_path_does_not_touch_the_oracle():
    """The binding and the library never import or link the CPU oracle."""
    pkg = os.path.dirname(fattn.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "attn_oracle" not in text, f


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(fattn, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(fattn, "_lib", None)
    with pytest.raises(fattn.FattnLibraryMissing):
        fattn.load()


def test_plan_head_group_rules(lib):
    """The causal task order's head groups: whole K/V heads, at most about
    48 MB of 16-bit K/V per group unless a single K/V head is larger, and as
    few groups as that budget allows, as equal in size as the heads allow."""
    budget = 48 << 20
    # hand-worked cases: 64 heads of 4 MiB K/V -> 12 fit, 6 groups of <= 11
    assert fattn.plan_head_group(2, 32, 8192, 128) == 11
    # 16 heads of 4.1 MB -> 11 fit, 2 groups of 8
    assert fattn.plan_head_group(1, 16, 16000, 64) == 8
    # 8 K/V heads of 8 MiB shared by pairs of query heads -> 6 K/V heads fit
    assert fattn.plan_head_group(1, 16, 32768, 64, Hkv=8) == 8
    # everything fits: one group
    assert fattn.plan_head_group(1, 8, 1, 64) == 8
    assert fattn.plan_head_group(3, 5, 1000, 128, Hkv=1) == 15
    # one K/V head larger than the budget: groups of one K/V head
    assert fattn.plan_head_group(1, 4, 1 << 20, 128) == 1
    assert fattn.plan_head_group(1, 8, 1 << 20, 128, Hkv=2) == 4
    for B, H, Hkv, N, D in [(1, 1, 1, 64, 64), (2, 7, 7, 8192, 128), (4, 16, 4, 16384, 128),
                            (3, 24, 3, 30000, 64), (8, 32, 8, 4096, 128), (1, 40, 40, 12000, 64),
                            (2, 12, 1, 65536, 128), (5, 9, 3, 20000, 128)]:
        BH, share = B * H, H // Hkv
        kv_head = 2 * N * D * 2
        hg = fattn.plan_head_group(B, H, N, D, Hkv=Hkv)
        assert 1 <= hg <= BH and hg % share == 0
        assert (hg // share) * kv_head <= budget or hg == share
        groups = -(-BH // hg)
        # no fewer groups are possible within the budget
        cap = max(share, (budget // kv_head) * share)
        assert groups == -(-BH // min(BH, cap))
        # the groups are as equal as whole K/V heads allow
        last = BH - (groups - 1) * hg
        assert 0 < last <= hg and hg - last < groups * share


def test_plan_head_group_rejects(lib):
    import ctypes
    out = ctypes.c_int64(7)
    assert lib.fattn_plan_head_group(1, 6, 4, 128, 64, ctypes.byref(out)) == 1
    assert lib.fattn_plan_head_group(1, 4, 4, 128, 96, ctypes.byref(out)) == 1
    assert lib.fattn_plan_head_group(0, 4, 4, 128, 64, ctypes.byref(out)) == 1
    assert lib.fattn_plan_head_group(1, 4, 4, 128, 64, None) == 1
    assert lib.fattn_plan_head_group(1, 4, 4, (1 << 30) + 1, 64, ctypes.byref(out)) == 2
