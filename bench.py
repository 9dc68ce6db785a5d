"""Benchmark of the attention forward on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference|unfused|rowwise] [--pass fwd|bwd]

A step is one attention forward (the whole hot path: one kernel launch) over
the named workload's synthetic seeded inputs, already resident in HBM.
Defaults: the headline workload bf16 B=4 H=16 N=4096 D=128 non-causal; the
default run then times the causal bf16 workload (B=2 H=32 N=8192 D=128, Q
std 4) the same way and adds it as the nested record `causal_target`
(`value` and `metric` stay the headline's; `gpu_launches` counts both).

Timing: W untimed warm-up steps, then K timed steps, each bracketed by CUDA
events on the stream the kernel is launched on; L2 is flushed (a 512 MB
buffer is rewritten) before every timed step, outside the events.  A short
device-side spin and two more untimed steps before the first timed step let
the host queue the steps ahead of the GPU (no event pair includes host launch
latency) and bring the clocks back up after the idle sampler start.  The whole
timed loop is bracketed by a barrier and a device synchronise; the reported
time is the max over ranks.  Under torchrun (N > 1) every rank runs the same
workload on its own GPU (independent replicas: the method has no exchange
step), so `value` is the total FLOP of all ranks over that max time.

`e2e` is the same metric measured through the library's host-buffer entry
point (fattn_fwd_host): per step, the host->device copies of Q, K, V from
pinned memory, the kernel and the device->host copy of O and LSE.

`cpu_baseline` is the fp64 CPU oracle as it stands, timed on this host's cores
on a bounded sample of the same workload (a set of random query rows).
`--impl reference` times that oracle alone (the reference arm of this method).

`--pass bwd` times the backward pass instead (fattn_bwd: dQ, dK, dV from
Q, K, V, O, LSE and a seeded dO, three kernels per step) under the same
rules; its FLOP count is 2.5x the forward's (five products of the size of
the forward's two), and its cpu_baseline / reference arm is the oracle's
backward on whole heads of the workload.

`--impl unfused` times the library's materialising comparator
(fattn_fwd_unfused: S and P written to HBM, three kernels per step) on the
same workload, inputs and timing rules, for the HBM-traffic comparison; its
roofline is the HBM bound of the whole three-kernel step.

`--impl rowwise` (fp32 workloads) times fattn_fwd_f32_rowwise, the fp32
kernel with one query row per thread, under the same rules (no e2e leg).

`--hkv G` times the grouped-query form of a 16-bit workload (forward or
backward): K and V are the workload's first G heads, shared by H/G query
heads each; FLOP as for the multi-head workload; device buffers only.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from tiled_attention_forward_gb300.inputs import BY_NAME, HEADLINE, workload_inputs  # noqa: E402

# The causal half of the target (bf16, N >= 4096): timed beside the headline.
CAUSAL_TARGET = BY_NAME["bf16_B2_H32_N8192_D128_causal_qstd4"]

METRIC = "attn fwd TFLOP/s (B=4,H=16,N=4096,D=128 bf16) and % of GB300 BF16 peak"
METRIC_BWD = "attn bwd TFLOP/s (5-product convention, 2.5x fwd FLOP) and % of GB300 BF16 peak"
BWD_FLOP_FACTOR = 2.5

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the forward kernel on each workload, from an ncu capture (summaries under
# profiles/), tagged with the hash of that kernel's device sources when it
# was taken.  Reported only while those sources still hash the same; null
# once the kernel has changed.
KERNEL_SOURCES = {"tc": ["fwd_tc.cu", "sm103_ptx.cuh"], "ffma": ["fwd_ffma.cu"],
                  "unfused": ["fwd_unfused.cu", "sm103_ptx.cuh"],
                  "bwd": ["bwd_tc.cu", "sm103_ptx.cuh"]}
NCU_TRAFFIC = {
    "bf16_B4_H16_N4096_D128": (201829632 + 39738624, "3a3002c616902885"),
    "bf16_B2_H32_N8192_D128_causal_qstd4": (410912768 + 111794176, "3a3002c616902885"),
    "fp16_B1_H16_N16000_D64_causal": (98407936 + 10369024, "3a3002c616902885"),
    "fp32_B4_H8_N8192_D64_causal": (201639936 + 51146240, "61c5185890f7842f"),
}


# The materialising comparator: DRAM bytes of one step (its three kernels).
NCU_TRAFFIC_UNFUSED = {
    "bf16_B4_H16_N4096_D128": (6653218560 + 6403927040, "ab7c710081d7976f"),
    "bf16_B2_H32_N8192_D128_causal_qstd4": (13389131008 + 13121990912, "ab7c710081d7976f"),
    "fp16_B1_H16_N16000_D64_causal": (12437732864 + 12321522432, "ab7c710081d7976f"),
}


# The backward: DRAM bytes of one step (statistics, dK/dV and dQ kernels).
NCU_TRAFFIC_BWD = {
    "bf16_B4_H16_N4096_D128": (676513536 + 154105856, "77268889cef676d6"),
    "bf16_B2_H32_N8192_D128_causal_qstd4": (7977567744 + 355400704, "77268889cef676d6"),
    "fp16_B1_H16_N16000_D64_causal": (463855360 + 51330816, "77268889cef676d6"),
}


def kernel_family(w):
    return "ffma" if w.dtype == "fp32" else "tc"


def kernel_source_hash(family):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tiled_attention_forward_gb300", "csrc")
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(w, unfused=False, bwd=False):
    table = NCU_TRAFFIC_BWD if bwd else (NCU_TRAFFIC_UNFUSED if unfused else NCU_TRAFFIC)
    family = "bwd" if bwd else ("unfused" if unfused else kernel_family(w))
    entry = table.get(w.name)
    if entry is None or entry[1] != kernel_source_hash(family):
        return None
    return entry[0]


UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20
PRIME_CYCLES = 20_000_000  # about 10 ms of device-side spin before the timed steps
DTYPE_NAMES = {"bf16": "bf16", "fp16": "f16", "fp32": "f32"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings (a no-op without a process group)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tflops(flops_per_step, n_ranks, steps, ms_total_max):
    """Work of every rank (weak scaling: each rank runs the full workload) over
    the slowest rank's time."""
    return flops_per_step * n_ranks * steps / (ms_total_max * 1e-3) / 1e12


def w_bytes(w):
    """Compulsory HBM bytes of one forward: read Q, K, V once, write O and LSE once."""
    e = {"fp32": 4, "fp16": 2, "bf16": 2}[w.dtype]
    return 4 * w.B * w.H * w.N * w.D * e + 4 * w.B * w.H * w.N


def unfused_bytes(w):
    """Algorithmic HBM bytes of one materialising forward: Q, K, V read and O,
    LSE written once, plus every computed S element written (fp32) and read
    once and every P element the P V product reads written and read once
    (16-bit).  Computed elements: 128 x 128 score tiles on or below the
    diagonal under causal masking, all N x N otherwise."""
    e = {"fp16": 2, "bf16": 2}[w.dtype]
    nt = -(-w.N // 128)
    npitch = -(-w.N // 8) * 8
    if w.causal:
        s_elems = 0
        p_elems = 0
        for qt in range(nt):
            rows = min(128, w.N - qt * 128)
            s_elems += rows * min(npitch, (qt + 1) * 128)
            p_elems += rows * min(npitch, (qt + 1) * 128)
    else:
        s_elems = p_elems = w.N * npitch
    bh = w.B * w.H
    return w_bytes(w) + bh * (2 * 4 * s_elems + 2 * e * p_elems)


def config_of(w, n_gpus, hkv=0):
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": hkv or w.H, "N": w.N, "D": w.D, "dtype": w.dtype,
            "causal": w.causal, "q_std": w.q_std, "scale": w.scale, "seed": w.seed,
            "l2": "flushed before every timed step (512 MB rewrite outside the events)",
            "parallelism": "replicas x%d (no exchange step)" % n_gpus}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for (t, s) in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not inside:  # region shorter than the sampling period: nearest samples
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[:3]
            inside = [s for (_, s) in near]
            window = "nearest samples to a timed region shorter than the 25 ms sampling period"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        sm = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        smax = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 5 + i and s[5 + i].lower() == "active"})
        power = [float(s[3]) for s in inside if s[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (the cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_rows_rate(w, q64, k64, v64, target_s, seed):
    """Times the oracle on random query rows of the workload; returns
    (FLOP done in the method's convention, seconds, rows, threads)."""
    import oracle
    rng = np.random.default_rng(seed)
    BH = w.B * w.H

    def flops_of(rows):
        keys = (rows + 1) if w.causal else np.full_like(rows, w.N)
        return float(np.sum(4.0 * keys * w.D))  # 2 FLOP for q.k and 2 for p.v per key and dim

    def run(nrows):
        bh = rng.integers(0, BH, nrows)
        rows = rng.integers(0, w.N, nrows)
        t = time.perf_counter()
        oracle.attention_rows(q64, k64, v64, w.scale, w.causal, bh, rows)
        return time.perf_counter() - t, flops_of(rows)

    nrows = 256
    dt, fl = run(nrows)
    while dt < 0.5 and nrows < (1 << 22):
        nrows *= 4
        dt, fl = run(nrows)
    nrows = max(1, int(nrows * target_s / max(dt, 1e-9)))
    dt, fl = run(nrows)
    return fl, dt, nrows, oracle.default_threads()


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, w, ws, rank, local):
    import tiled_attention_forward_gb300 as fattn

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    q, k, v = workload_inputs(w)
    if args.hkv:  # grouped-query heads: the first Hkv heads of the workload's K and V
        k, v = k[:, :args.hkv].contiguous(), v[:, :args.hkv].contiguous()
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    unfused = args.impl == "unfused"
    rowwise = args.impl == "rowwise"
    if rowwise and w.dtype != "fp32":
        raise SystemExit("--impl rowwise covers fp32 workloads only")
    if unfused:
        if w.dtype == "fp32":
            raise SystemExit("--impl unfused covers bf16 / fp16 workloads only")
        wsp = torch.empty(fattn.unfused_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)

    def step():
        if unfused:
            fattn.fwd_unfused(qd, kd, vd, causal=w.causal, scale=w.scale, out=o, lse=lse,
                              workspace=wsp, stream=stream)
        elif rowwise:
            fattn.fwd_f32_rowwise(qd, kd, vd, causal=w.causal, scale=w.scale, out=o, lse=lse,
                                  stream=stream)
        else:
            fattn.fwd(qd, kd, vd, causal=w.causal, scale=w.scale, out=o, lse=lse, stream=stream)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fattn.get_device_status(stream) != 0:
        raise RuntimeError("device status after warm-up")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    # A short device-side spin (outside every event pair) lets the host queue
    # the timed steps ahead of the GPU, so that no step's events include the
    # host's launch latency; two more untimed steps right before the timed
    # ones bring the clocks back up after the idle time around the sampler
    # start (the first step after an idle GPU ran about 10 % slower).
    torch.cuda._sleep(PRIME_CYCLES)
    for _ in range(2):
        flush.zero_()
        step()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t1 = time.time()
    time.sleep(0.15)
    sampler.stop()
    status = fattn.get_device_status(stream)
    if status != 0:
        raise RuntimeError("device status %s during the timed region" % fattn.status_string(status))
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms
    ms_total = float(sum(per))
    # fattn_fwd launches exactly one kernel per call, fattn_fwd_unfused three
    launches = args.steps * (3 if unfused else 1)

    # end to end through the host-buffer entry point
    e2e_ms, h2d, d2h = float("nan"), 0, 0
    if not args.no_e2e and not unfused and not rowwise:
        e2e_ms, h2d, d2h = run_e2e(fattn, w, q, k, v, qd, kd, vd, o, lse, stream, dev, args.steps, barrier)
    ms_total, e2e_ms = max_over_ranks([ms_total, e2e_ms], device=dev)
    clocks = sampler.summary(t0, t1)
    if rank != 0:
        return None

    flops = w.flops()
    ms_per_step = ms_total / args.steps
    value = whole_job_tflops(flops, ws, args.steps, ms_total)
    achieved = flops / (ms_per_step * 1e-3) / 1e12  # one launch = one step on this GPU
    peaks, peak_src = load_peaks()
    peak_key = "bf16_tflops"
    if unfused:
        gbs = unfused_bytes(w) / (ms_per_step * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                "traffic": ncu_traffic(w, unfused=True),
                "scope": "the whole three-kernel step (S, softmax, P V)",
                "peak_source": "hbm_gbs (STREAM-style copy) of %s" % peak_src,
                "algorithmic_bytes": unfused_bytes(w),
                "tensor_tflops": achieved}
    elif w.dtype == "fp32":
        sm_mhz = peaks.get("sm_max_mhz", 2070.0)
        peak = torch.cuda.get_device_properties(dev).multi_processor_count * 128 * 2 * sm_mhz * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "traffic": ncu_traffic(w) if not (rowwise or args.hkv) else None,
                "peak_source": "FP32 FFMA: SMs x 128 lanes x 2 FLOP x max SM clock (%s clock)" % peak_src}
    else:
        peak = float(peaks[peak_key])
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "traffic": ncu_traffic(w) if not (rowwise or args.hkv) else None,
                "peak_source": "%s dense bf16 (cuBLAS burst) of %s; fp16 taken at the same rate"
                               % (peak_key, peak_src),
                "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak))}
    roof["traffic_note"] = ("DRAM bytes per step, summed over its three kernels (ncu "
                            "dram__bytes_read.sum + dram__bytes_write.sum)") if unfused else ("DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum); "
                            "algorithmic compulsory bytes (Q+K+V read, O+LSE write): %d" % w_bytes(w))
    if unfused or rowwise:
        line_extra = {"impl": args.impl}
    else:
        line_extra = {}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_median": statistics.median(per),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_NAMES[w.dtype], "data": "synthetic (seeded iid normal Q, K, V)",
        "config": config_of(w, ws, args.hkv), "pct_of_peak": 100.0 * roof["frac"], "roofline": roof,
        "e2e": ({"value": flops * ws / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                 "ms_per_step": e2e_ms, "api": "fattn_fwd_host (pinned host buffers)"}
                if not (args.no_e2e or unfused or rowwise) else None),
        "gpu_launches": launches, "clocks": clocks,
    }
    line.update(line_extra)
    if not args.no_cpu_baseline and not unfused and not rowwise:
        q64, k64, v64 = (t.to(torch.float64).numpy() for t in (q, k, v))
        fl, secs, nrows, threads = oracle_rows_rate(w, q64, k64, v64, args.cpu_seconds, 1)
        line["cpu_baseline"] = {"value": fl / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": "%d random query rows of the workload (%.1f s, fp64 C "
                                          "oracle, one thread per CPU)" % (nrows, secs)}
    return line


def oracle_bwd_rate(w, q, k, v, do, target_s):
    """Times the oracle's backward on whole heads of the workload (as many as
    fit in about target_s seconds); returns (FLOP in the backward convention,
    seconds, heads, threads)."""
    import oracle
    heads_total = w.B * w.H
    qh, kh, vh, dh = (t.reshape(1, heads_total, w.N, w.D) for t in (q, k, v, do))
    done, secs, n = 0, 0.0, 1
    while done < heads_total:
        n = min(n, heads_total - done)
        sl = slice(done, done + n)
        args = [t[:, sl].to(torch.float64).numpy() for t in (qh, kh, vh, dh)]
        t0 = time.perf_counter()
        oracle.backward(*args, w.scale, w.causal)
        dt = time.perf_counter() - t0
        secs += dt
        done += n
        if secs >= target_s:
            break
        n = max(1, min(2 * n, int(n * (target_s - secs) / max(dt, 1e-3))))
    per_head = w.flops() / heads_total
    return BWD_FLOP_FACTOR * per_head * done, secs, done, oracle.default_threads()


def bwd_inputs(w):
    q, k, v = workload_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 50)
    do = torch.randn(q.shape, generator=g).to(q.dtype)
    return q, k, v, do


def run_ours_bwd(args, w, ws, rank, local):
    """The backward pass: one step = fattn_bwd over the workload (statistics,
    dK/dV and dQ kernels), inputs (Q, K, V, O, LSE, dO) resident in HBM."""
    import tiled_attention_forward_gb300 as fattn

    if w.dtype == "fp32":
        raise SystemExit("--pass bwd covers bf16 / fp16 workloads only")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    q, k, v, do = bwd_inputs(w)
    if args.hkv:  # grouped-query heads: the first Hkv heads of the workload's K and V
        k, v = k[:, :args.hkv].contiguous(), v[:, :args.hkv].contiguous()
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fattn.fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    wsp = torch.empty(fattn.bwd_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fattn.bwd(qd, kd, vd, o, lse, dod, causal=w.causal, scale=w.scale, dq=dq, dk=dk, dv=dv,
                  workspace=wsp, stream=stream)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fattn.get_device_status(stream) != 0:
        raise RuntimeError("device status after warm-up")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    # A short device-side spin (outside every event pair) lets the host queue
    # the timed steps ahead of the GPU, so that no step's events include the
    # host's launch latency; two more untimed steps right before the timed
    # ones bring the clocks back up after the idle time around the sampler
    # start (the first step after an idle GPU ran about 10 % slower).
    torch.cuda._sleep(PRIME_CYCLES)
    for _ in range(2):
        flush.zero_()
        step()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t1 = time.time()
    time.sleep(0.15)
    sampler.stop()
    status = fattn.get_device_status(stream)
    if status != 0:
        raise RuntimeError("device status %s during the timed region" % fattn.status_string(status))
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_total = float(sum(per))

    # end to end through the library's host-buffer entry point: per step the
    # six inputs copied in from pinned memory, the backward and the three
    # gradients copied back, in groups of heads that overlap
    e2e_ms, h2d, d2h = float("nan"), 0, 0
    if not args.no_e2e:
        hosts = [t.pin_memory() for t in (q, k, v)] + [o.cpu().pin_memory(), do.pin_memory(),
                                                       lse.cpu().pin_memory()]
        devs = [qd, kd, vd, o, dod, lse]
        outs_h = [torch.empty_like(q).pin_memory() for _ in range(3)]
        n_e2e = max(3, min(args.steps, 20))

        def e2e_step():
            fattn.bwd_host(hosts, devs, outs_h, [dq, dk, dv], wsp, causal=w.causal, scale=w.scale,
                           stream=stream)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        es.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        ee.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = es.elapsed_time(ee) / n_e2e
        h2d = sum(t.numel() * t.element_size() for t in hosts)
        d2h = sum(t.numel() * t.element_size() for t in outs_h)
    ms_total, e2e_ms = max_over_ranks([ms_total, e2e_ms], device=dev)
    clocks = sampler.summary(t0, t1)
    if rank != 0:
        return None
    flops = BWD_FLOP_FACTOR * w.flops()
    ms_per_step = ms_total / args.steps
    value = whole_job_tflops(flops, ws, args.steps, ms_total)
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
            "traffic": ncu_traffic(w, bwd=True) if not args.hkv else None,
            "scope": "the whole three-kernel step (statistics, dK/dV, dQ)",
            "traffic_note": "DRAM bytes per step, summed over its three kernels (ncu "
                            "dram__bytes_read.sum + dram__bytes_write.sum)",
            "peak_source": "bf16_tflops dense bf16 (cuBLAS burst) of %s; fp16 taken at the same rate" % peak_src,
            "frac_of_sustained": achieved / float(peaks.get("bf16_tflops_sustained", peak)),
            "executed_tensor_tflops": achieved * 7.0 / 5.0,
            "note": "algorithmic FLOP = 5 products of 128x128xD per tile pair; the kernels execute 7 "
                    "(S and dP are formed once for dK/dV and once for dQ)"}
    line = {
        "metric": METRIC_BWD, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "ms_per_step_median": statistics.median(per),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_NAMES[w.dtype], "data": "synthetic (seeded iid normal Q, K, V, dO)",
        "config": dict(config_of(w, ws, args.hkv), **{"pass": "bwd"}), "pct_of_peak": 100.0 * roof["frac"],
        "roofline": roof,
        "e2e": ({"value": flops * ws / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                 "api": "fattn_bwd_host (pinned host buffers)"}
                if not args.no_e2e else None),
        "gpu_launches": 3 * args.steps, "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        fl, secs, heads, threads = oracle_bwd_rate(w, q, k, v, do, args.cpu_seconds)
        line["cpu_baseline"] = {"value": fl / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": "fp64 C oracle backward on %d whole head(s) of the workload "
                                          "(%.1f s)" % (heads, secs)}
    return line


def run_reference_bwd(args, w, ws, rank):
    if rank != 0:
        return None
    q, k, v, do = bwd_inputs(w)
    per_step_s = max(0.5, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_bwd_rate(w, q, k, v, do, min(per_step_s, 1.0))
    fl_tot, secs_tot, heads_tot, threads = 0.0, 0.0, 0, 1
    for _ in range(args.steps):
        fl, s, h, threads = oracle_bwd_rate(w, q, k, v, do, per_step_s)
        fl_tot += fl
        secs_tot += s
        heads_tot += h
    value = fl_tot / secs_tot / 1e12 if secs_tot > 0 else 0.0
    sample = "%d whole heads over %d steps (%.1f s), fp64 C oracle backward" % (heads_tot, args.steps, secs_tot)
    return {
        "impl": "reference", "metric": METRIC_BWD, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs_tot / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded iid normal Q, K, V, dO)",
        "config": dict(config_of(w, 1), **{"pass": "bwd"}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_e2e(fattn, w, q, k, v, qd, kd, vd, o, lse, stream, dev, steps, barrier):
    """Per step: H2D of Q, K, V from pinned memory, the kernel, D2H of O and LSE,
    all enqueued by the library's host-buffer entry point."""
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty_like(q).pin_memory()
    lh = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(steps, 20))
    for _ in range(2):
        fattn.fwd_host(qh, kh, vh, qd, kd, vd, o, oh, lse, lh, causal=w.causal, scale=w.scale,
                       stream=stream)
    torch.cuda.synchronize(dev)
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    es.record(stream)
    for _ in range(e2e_steps):
        fattn.fwd_host(qh, kh, vh, qd, kd, vd, o, oh, lse, lh, causal=w.causal, scale=w.scale,
                       stream=stream)
    ee.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = es.elapsed_time(ee) / e2e_steps
    elem = q.element_size()
    return e2e_ms, 3 * q.numel() * elem, o.numel() * elem + lse.numel() * 4


def run_reference(args, w, ws, rank):
    if rank != 0:
        return None
    q, k, v = workload_inputs(w)
    q64, k64, v64 = (t.to(torch.float64).numpy() for t in (q, k, v))
    per_step_s = max(0.5, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_rows_rate(w, q64, k64, v64, min(per_step_s, 1.0), 100 + i)
    flops_tot, rows_tot, secs_tot, threads = 0.0, 0, 0.0, 1
    for i in range(args.steps):
        fl, s, n, threads = oracle_rows_rate(w, q64, k64, v64, per_step_s, 1000 + i)
        flops_tot += fl
        rows_tot += n
        secs_tot += s
    value = flops_tot / secs_tot / 1e12 if secs_tot > 0 else 0.0
    sample = "%d random query rows over %d steps (%.1f s), fp64 C oracle" % (rows_tot, args.steps, secs_tot)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs_tot / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded iid normal Q, K, V)",
        "config": config_of(w, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE.name, choices=sorted(BY_NAME))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference", "unfused", "rowwise"])
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd"])
    ap.add_argument("--hkv", type=int, default=0,
                    help="grouped-query K/V heads (0: as many as query heads); 16-bit workloads, "
                         "device-buffer timing only")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall time of the CPU oracle sample (cpu_baseline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--no-causal-target", action="store_true",
                    help="on the default workload, skip the nested causal bf16 record")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl != "reference":
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    w = BY_NAME[args.workload]
    if args.hkv:
        if args.impl != "ours" or w.dtype == "fp32" or w.H % args.hkv != 0 or args.hkv >= w.H:
            ap.error("--hkv needs --impl ours, a 16-bit workload and 0 < Hkv < H dividing H")
        args.no_e2e = True           # the host-buffer entry points take H == Hkv
        args.no_cpu_baseline = True
    if args.pass_ == "bwd" and args.impl in ("unfused", "rowwise"):
        ap.error("--impl %s is a forward variant" % args.impl)
    if args.impl == "reference":
        line = run_reference_bwd(args, w, ws, rank) if args.pass_ == "bwd" else run_reference(args, w, ws, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        if args.pass_ == "bwd":
            line = run_ours_bwd(args, w, ws, rank, local)
        else:
            line = run_ours(args, w, ws, rank, local)
            # The target has a causal half: on the default run the causal bf16
            # workload is timed too, after the headline and under the same
            # rules, and reported as a nested record (value and metric stay
            # the headline's).
            if (w is HEADLINE and args.impl == "ours" and not args.hkv and not args.no_causal_target):
                cargs = argparse.Namespace(**vars(args))
                cargs.no_e2e = True
                cargs.no_cpu_baseline = True
                sub = run_ours(cargs, CAUSAL_TARGET, ws, rank, local)
                if line is not None and sub is not None:
                    line["causal_target"] = {
                        key: sub[key] for key in ("value", "unit", "ms_per_step", "ms_per_step_median",
                                                  "steps", "warmup", "dtype", "config", "pct_of_peak",
                                                  "roofline", "clocks", "gpu_launches")}
                    line["causal_target"]["metric"] = "attn fwd TFLOP/s (B=2,H=32,N=8192,D=128 bf16 causal, Q std 4)"
                    line["gpu_launches"] += sub["gpu_launches"]
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
