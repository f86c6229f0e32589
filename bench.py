#!/usr/bin/env python3
"""Benchmark of exact softmax attention (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step is one pass of the whole hot path over one batch of synthetic input:
fa_fwd, then fa_bwd, which runs three backward phases for this head dimension
(d = 128: preprocess, dK/dV, per-query-tile dQ, the dQ kernel taking the SMs
the dK/dV pass leaves idle in its last round; d = 64, 256: preprocess, main
with atomic dQ, postprocess), all through the C ABI. The headline pass times
K such steps; a second pass of K steps runs the same kernels with events
between the backward's phases (which serialises them) for each kernel's own
time, used by the rooflines. The default workload is the pages' microbenchmark shape at
hidden size 2048 with d = 128 and N = 8192 (B = 16384 / N = 2, H = 16),
non-causal: the configuration the headline "fwd+bwd TFLOP/s" figures are
quoted on. FLOPs follow the pages' convention: forward 4 B H N^2 d (halved
when causal), backward 2.5x forward.

Rank 0 prints one JSON line. `value` is fwd+bwd TFLOP/s over all ranks with
inputs resident in HBM; `e2e` is the same metric through the host-buffer
entry point fa_fwd_bwd_host, with the host->device copies of Q, K, V, dO and
the device->host copies of O, L, dQ, dK, dV (pinned host memory) inside the
timed region, overlapped with the kernels by the library; `roofline` is the dominant kernel against the measured dense bf16
peak, with that kernel's own algorithmic FLOPs; `cpu_baseline` is the float64 CPU oracle timed on
a bounded sample. `--impl reference` times that oracle alone as the reference
arm (rank 0 only).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attn_inputs import WORKLOADS, sweep_points, seed_for, make_inputs  # noqa: E402

METRIC = "attention fwd and fwd+bwd TFLOP/s (bf16, 1 GB300) and % of dense BF16 peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "sweep_d128_N8192_full"
# Pages' fwd+bwd number for this exact workload (A100 80GB, d=128, N=8k,
# non-causal, 16k tokens, hidden 2048): context only, another machine.
PAGES_FWD_BWD_TFLOPS = {"sweep_d128_N8192_full": 201.0}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_BF16_TFLOPS = 2250.0  # GB300 datasheet dense bf16 (without 2:4 sparsity), for context
_CSRC = "exact_softmax_attention_fa_gb300/csrc/"
_COMMON = [_CSRC + "sm103_ptx.cuh", _CSRC + "fa_kernel_common.cuh"]
# Source files of each kernel: a committed ncu summary carries their hash,
# and its DRAM traffic is reported only while the hash still matches.
KERNEL_SOURCES = {
    "fa_bwd_main": [_CSRC + "fa_bwd.cu"] + _COMMON,
    "fa_bwd_dkdv": [_CSRC + "fa_bwd.cu"] + _COMMON,
    "fa_bwd_dq": [_CSRC + "fa_bwd_dq.cu"] + _COMMON,
    "fa_fwd": [_CSRC + "fa_fwd_kernel.cuh"] + _COMMON,
    "fa_bwd256": [_CSRC + "fa_bwd256.cu"] + _COMMON,
    "fa_bwd_dq256": [_CSRC + "fa_bwd_dq256.cu"] + _COMMON,
    "bwd_pre": [_CSRC + "fa_bwd.cu"] + _COMMON,
}


def all_workloads() -> dict:
    w = {name: dict(p) for name, p in sweep_points()}
    for name, p in WORKLOADS.items():
        w[name] = dict(p)
    return w


def flops(p: dict, mode: str) -> float:
    f = 4.0 * p["B"] * p["H"] * p["N"] * p["N"] * p["d"]
    if p["causal"]:
        f *= 0.5
    return f * {"fwd": 1.0, "bwd": 2.5, "fwd_bwd": 3.5}[mode]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    if not m_bytes or not m_hash or m_hash.group(1) != source_hash(kernel):
        return None
    return int(m_bytes.group(1))


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,power.limit")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        self.out.close()
        os.unlink(self.out.name)
        sm, mx, pw, lim, reasons = [], [], [], [], set()
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for lst, idx in ((pw, 3), (lim, 9)):
                try:
                    lst.append(float(r[idx]))
                except (ValueError, IndexError):
                    pass
            for name, val in zip(self.REASONS, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w": statistics.median(pw) if pw else None, "power_limit_w": max(lim) if lim else None}


# ---------------------------------------------------------------------------
# distributed helpers (one process per GPU; gloo works on CPU for tests)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and getattr(device, "type", "cpu") == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate_value(per_rank_flops: float, world: int, max_time_s: float) -> float:
    """Whole-job TFLOP/s: every rank processes its own copy of the workload."""
    return per_rank_flops * world / max_time_s / 1e12


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------
def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(p: dict, x: dict, rows_per_call: int, calls: int):
    """Run the float64 oracle's row-block fwd+bwd `calls` times; return (seconds, flops)."""
    import numpy as np
    import oracle
    from attn_inputs import bf16_bits_to_f64
    scale = float(np.float32(1.0 / np.sqrt(p["d"])))
    N = p["N"]
    f64 = {k: bf16_bits_to_f64(v[0, 0]) for k, v in x.items()}
    t0 = time.perf_counter()
    fl = 0.0
    for c in range(calls):
        r0 = (c * rows_per_call) % max(1, N - rows_per_call + 1)
        rows = np.arange(r0, min(N, r0 + rows_per_call))
        oracle.attention_fwd_bwd_rows(f64["q"], f64["k"], f64["v"], f64["do"], rows, p["causal"], scale)
        keys = (rows + 1).sum() if p["causal"] else len(rows) * N
        fl += 3.5 * 4.0 * keys * p["d"]  # same convention: causal counts only unmasked entries
    return time.perf_counter() - t0, fl


def calibrate_rows(p: dict, x: dict, target_s: float) -> int:
    rows = 64
    t, _ = oracle_sample(p, x, rows, 1)
    per_row = max(t / rows, 1e-7)
    return int(max(16, min(p["N"], target_s / per_row)))


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def host_inputs(p: dict, rank: int):
    return make_inputs(p["B"], p["H"], p["N"], p["d"], seed_for(p) + rank, peaked_frac=p.get("peaked_frac", 0.0))


def backward_phases(fa, d, t, causal, scale, ws, stream):
    """The backward phases fa_bwd runs for this head dimension (include/fa.h):
    names and calls, in order."""
    q, k, v, o, lse, do, dq, dk, dv = (t[n] for n in ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv"))
    if d == 128:
        return (("bwd_pre", "bwd_dkdv", "bwd_dq"),
                (lambda: fa.fa_bwd_preprocess_stats(o, lse, do, ws, stream),
                 lambda: fa.fa_bwd_dkdv(q, k, v, do, dk, dv, causal, scale, ws, stream),
                 lambda: fa.fa_bwd_dq(q, k, v, do, dq, causal, scale, ws, stream)))
    return (("bwd_pre", "bwd_main", "bwd_post"),
            (lambda: fa.fa_bwd_preprocess(o, lse, do, ws, stream),
             lambda: fa.fa_bwd_main(q, k, v, do, dk, dv, causal, scale, ws, stream),
             lambda: fa.fa_bwd_postprocess(dq, ws, stream)))


def device_buffers(fa, p: dict, x: dict, device):
    """Device copies of the inputs and the outputs and workspace of one step."""
    import numpy as np
    import torch
    B, H, N, d = p["B"], p["H"], p["N"], p["d"]
    t = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(device) for k, v in x.items()}
    t["o"] = torch.empty_like(t["q"])
    t["lse"] = torch.empty((B, H, N), dtype=torch.float32, device=device)
    for n in ("dq", "dk", "dv"):
        t[n] = torch.empty_like(t["q"])
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=device)
    return t, ws


def time_device_step(fa, p: dict, t: dict, ws, stream, steps: int, warmup: int, on_timed=None):
    """Time `steps` back-to-back steps (fa_fwd, then the backward phases) with
    CUDA events on `stream`; returns (total ms, per-phase mean ms, phase names).
    `on_timed` = (start, stop) callbacks bracketing the timed region."""
    import numpy as np
    import torch
    causal, d = p["causal"], p["d"]
    scale = float(np.float32(1.0 / np.sqrt(d)))
    names, calls = backward_phases(fa, d, t, causal, scale, ws, stream)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(t["q"], t["k"], t["v"], t["o"], t["lse"], causal, scale, stream)
        for i, call in enumerate(calls):
            if ev is not None:
                ev[1 + i].record(stream)
            call()
        if ev is not None:
            ev[4].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(stream.device)
    if fa.fa_get_device_status(stream) != 0:
        raise RuntimeError("device status reports a timed-out pipeline wait during warm-up")
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    if on_timed:
        on_timed[0]()
    for s_ in range(steps):
        step(events[s_])
    torch.cuda.synchronize(stream.device)
    if on_timed:
        on_timed[1]()
    status = fa.fa_get_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    total_ms = events[0][0].elapsed_time(events[-1][4])
    phase_ms = [sum(e[i].elapsed_time(e[i + 1]) for e in events) / steps for i in range(4)]
    return total_ms, phase_ms, ("fwd",) + names


def time_api_step(fa, p: dict, t: dict, ws, stream, steps: int, warmup: int, on_timed=None):
    """Time `steps` back-to-back steps as a user makes them: fa_fwd, then
    fa_bwd, which queues the backward's kernels with the overlap it gives
    them (at d = 128 the dQ kernel takes the SMs the dK/dV pass leaves idle
    in its last round; events between the phases would serialise them).
    CUDA events on `stream` at the step and pass boundaries only; returns
    (total ms, mean forward ms, mean backward ms)."""
    import numpy as np
    import torch
    causal, d = p["causal"], p["d"]
    scale = float(np.float32(1.0 / np.sqrt(d)))
    q, k, v, o, lse, do, dq, dk, dv = (t[n] for n in ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv"))

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(q, k, v, o, lse, causal, scale, stream)
        if ev is not None:
            ev[1].record(stream)
        fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal, scale, ws, stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(stream.device)
    if fa.fa_get_device_status(stream) != 0:
        raise RuntimeError("device status reports a timed-out pipeline wait during warm-up")
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    if on_timed:
        on_timed[0]()
    for s_ in range(steps):
        step(events[s_])
    torch.cuda.synchronize(stream.device)
    if on_timed:
        on_timed[1]()
    status = fa.fa_get_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    total_ms = events[0][0].elapsed_time(events[-1][2])
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in events) / steps
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in events) / steps
    return total_ms, fwd_ms, bwd_ms


EXTRA_WORKLOADS = ("long_causal_peaked", "wide_head_d256")
EXTRA_STEPS = 10


def time_workload(fa, name: str, device, stream, steps: int, warmup: int) -> dict:
    """Device-resident timing of one named workload (fa_fwd + the backward
    phases fa_bwd runs), as a dict of sizes, per-phase ms and TFLOP/s."""
    import torch
    p = all_workloads()[name]
    t, ws = device_buffers(fa, p, host_inputs(p, 0), device)
    total_ms, fwd_ms, bwd_ms = time_api_step(fa, p, t, ws, stream, steps, warmup)
    _total, phase_ms, names = time_device_step(fa, p, t, ws, stream, steps, warmup)
    del t, ws
    torch.cuda.empty_cache()
    return {"workload": name, **{kk: p[kk] for kk in ("B", "H", "N", "d", "causal")},
            **({"peaked_frac": p["peaked_frac"]} if "peaked_frac" in p else {}),
            "steps": steps, "warmup": warmup, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            **workload_rates(p, fwd_ms, bwd_ms, total_ms / steps),
            "phase_ms": dict(zip(names, phase_ms))}


def run_sweep(args) -> int:
    """One JSON line per point of the pages' microbenchmark grid (hidden 2048:
    d = 64 x 32 heads and d = 128 x 16 heads, N = 512 .. 16k, B = 16384 / N,
    causal and not), then the long-context and d = 256 configurations."""
    import torch
    import exact_softmax_attention_fa_gb300 as fa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    names = [n for n, _ in sweep_points()] + list(EXTRA_WORKLOADS)
    for name in names:
        print(json.dumps(time_workload(fa, name, device, stream, args.steps, args.warmup)), flush=True)
    return 0


def workload_rates(p: dict, fwd_ms: float, bwd_ms: float, step_ms: float) -> dict:
    """TFLOP/s by the pages' convention from the mean forward, backward and
    step times (ms) of the user-call pass."""
    f_fwd, f_bwd, f_step = flops(p, "fwd"), flops(p, "bwd"), flops(p, "fwd_bwd")
    return {"fwd_tflops": f_fwd / (fwd_ms / 1e3) / 1e12,
            "bwd_tflops": f_bwd / (bwd_ms / 1e3) / 1e12,
            "fwd_bwd_tflops": f_step / (step_ms / 1e3) / 1e12}


def run_reference(args, p: dict, name: str) -> dict:
    """The float64 CPU oracle as the reference arm (rank 0 only)."""
    x = make_inputs(1, 1, p["N"], p["d"], seed_for(p))
    budget_s = 100.0
    rows = calibrate_rows(p, x, budget_s / max(1, args.steps + args.warmup))
    oracle_sample(p, x, rows, args.warmup)
    t, fl = oracle_sample(p, x, rows, args.steps)
    value = fl / t / 1e12
    cores = cpu_threads()
    sample = (f"per step: float64 oracle forward+backward of {rows} query rows x all {p['N']} keys of one head "
              f"(d={p['d']}, causal={p['causal']}), i.e. {rows / p['N'] / (p['B'] * p['H']):.2e} of one "
              f"workload step")
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, **{k: p[k] for k in ("B", "H", "N", "d", "causal")}},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_ours(args, p: dict, name: str, world: int, rank: int, local: int) -> dict | None:
    import numpy as np
    import torch
    import exact_softmax_attention_fa_gb300 as fa

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    B, H, N, d, causal = p["B"], p["H"], p["N"], p["d"], p["causal"]
    scale = float(np.float32(1.0 / np.sqrt(d)))
    x = host_inputs(p, rank)
    pinned = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory() for k, v in x.items()}
    t, ws = device_buffers(fa, p, x, device)
    q, k, v, do = t["q"], t["k"], t["v"], t["do"]
    o, lse, dq, dk, dv = t["o"], t["lse"], t["dq"], t["dk"], t["dv"]
    stream = torch.cuda.current_stream(device)

    clocks = ClockSampler(local)

    def start_timed():
        barrier(device)
        torch.cuda.synchronize(device)
        clocks.start()

    def start_phases():
        barrier(device)
        torch.cuda.synchronize(device)

    def stop_timed():
        barrier(device)

    # The headline pass: K steps of fa_fwd + fa_bwd as a user calls them. Then
    # K steps of the same kernels with events between the backward's phases
    # (which serialises them) for each kernel's own time: the rooflines.
    # The clock sampler runs through both.
    total_ms, api_fwd_ms, api_bwd_ms = time_api_step(fa, p, t, ws, stream, args.steps, args.warmup,
                                                     (start_timed, stop_timed))
    _phase_total_ms, phase_ms, phase_names = time_device_step(fa, p, t, ws, stream, args.steps, args.warmup,
                                                              (start_phases, stop_timed))
    clk = clocks.stop()
    bwd_names = phase_names[1:]
    max_s = max_over_ranks(total_ms / 1e3, device if world > 1 else None)

    # End to end through the C ABI's host-buffer entry point (fa_fwd_bwd_host):
    # every step uploads Q, K, V, dO from pinned host memory and reads O, L,
    # dQ, dK, dV back into it; the library overlaps those copies with its
    # kernels on two copy streams of its own.
    e2e_steps = max(1, min(args.steps, 20))
    out_host = {kk: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for kk, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    host_buf = torch.empty(fa.fa_fwd_bwd_host_device_bytes(B, H, N, d), dtype=torch.uint8, device=device)

    def e2e_step():
        fa.fa_fwd_bwd_host(pinned["q"], pinned["k"], pinned["v"], pinned["do"], out_host["o"], out_host["lse"],
                           out_host["dq"], out_host["dk"], out_host["dv"], causal, scale, host_buf, stream)

    for _ in range(max(3, min(args.warmup, 5))):
        e2e_step()
    torch.cuda.synchronize(device)
    barrier(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3 / e2e_steps, device if world > 1 else None)
    # The forward alone through fa_fwd_host (inference callers): Q, K, V up,
    # O and L back, pipelined over head chunks.
    fwd_buf = torch.empty(fa.fa_fwd_host_device_bytes(B, H, N, d), dtype=torch.uint8, device=device)

    def e2e_fwd_step():
        fa.fa_fwd_host(pinned["q"], pinned["k"], pinned["v"], out_host["o"], out_host["lse"], causal, scale, fwd_buf,
                       stream)

    for _ in range(max(3, min(args.warmup, 5))):
        e2e_fwd_step()
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_fwd_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_fwd_s = max_over_ranks(e0.elapsed_time(e1) / 1e3 / e2e_steps, device if world > 1 else None)
    del fwd_buf
    h2d = sum(a.numel() * a.element_size() for a in (q, k, v, do))
    d2h = sum(a.numel() * a.element_size() for a in (o, lse, dq, dk, dv))
    q_bytes, o_bytes, lse_bytes = (a.numel() * a.element_size() for a in (q, o, lse))
    del host_buf, out_host

    # The other single-GPU configurations of the pages' workloads (the
    # longest causal sequence with peaked rows, and the d = 256 head), timed
    # the same way as the headline step on their own device-resident inputs.
    extra = {}
    if world == 1 and not args.no_extra_configs:
        del t, ws, q, k, v, do, o, lse, dq, dk, dv
        torch.cuda.empty_cache()
        for wname in EXTRA_WORKLOADS:
            extra[wname] = time_workload(fa, wname, device, stream, EXTRA_STEPS, 3)

    if rank != 0:
        return None

    peaks, peak_kind = load_peaks()
    burst, sustained = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    f_fwd, f_bwd, f_step = flops(p, "fwd"), flops(p, "bwd"), flops(p, "fwd_bwd")
    n_pad = (N + 127) // 128 * 128
    clock_mhz = clk.get("sm_mhz") or clk.get("sm_max_mhz") or 2070.0
    num_sms = torch.cuda.get_device_properties(device).multi_processor_count
    pre_bytes = B * H * (2 * N * d * 2 + N * 4 + 2 * n_pad * 4 + (0 if bwd_names[1] == "bwd_dkdv" else n_pad * d * 4))
    value = aggregate_value(f_step * args.steps, world, max_s)
    rates = workload_rates(p, api_fwd_ms, api_bwd_ms, total_ms / args.steps)
    fwd_tf, bwd_tf, fwd_bwd_tf = rates["fwd_tflops"], rates["bwd_tflops"], rates["fwd_bwd_tflops"]
    # Per kernel: its phase time and its own share of the method's FLOPs. The
    # backward's 10 N^2 d per head (2.5x forward) are five 128x128xd products
    # per tile pair: the dK/dV kernel computes four of them (S, dP, dV, dK);
    # the dQ kernel recomputes S and dP, which the method needs only once, so
    # it is credited with its dQ product alone.
    if bwd_names[1] == "bwd_dkdv":
        kernels = {"fa_fwd": (phase_ms[0], f_fwd), "fa_bwd_dkdv": (phase_ms[2], 0.8 * f_bwd),
                   "fa_bwd_dq": (phase_ms[3], 0.2 * f_bwd)}
    else:  # the atomic main kernel: fa_bwd.cu at d = 64, fa_bwd256.cu at d = 256
        kernels = {"fa_fwd": (phase_ms[0], f_fwd), ("fa_bwd256" if d == 256 else "fa_bwd_main"): (phase_ms[2], f_bwd)}
    # The denominator: the burst bf16 peak for kernels timed in a short
    # region that the power cap did not throttle, the sustained one when the
    # clock sampler saw the power cap active. Both fractions are reported.
    capped = "sw_power_cap" in (clk.get("reasons") or [])
    peak = sustained if capped else burst
    peak_desc = (f"{peak_kind} {'sustained' if capped else 'burst'} dense bf16 (MEASURED_PEAKS.json); "
                 f"{'sw_power_cap seen' if capped else 'no power cap seen'} during the timed region")

    def roof(name):
        ms, fl = kernels[name]
        ach = fl / (ms / 1e3) / 1e12
        return {"bound": "tensor", "kernel": name, "achieved": ach, "peak": peak, "unit": UNIT,
                "frac": ach / peak, "frac_vs_burst": ach / burst, "frac_vs_sustained": ach / sustained,
                "traffic": profiled_traffic(name, name_workload), "avg_launch_ms": ms}

    name_workload = name
    ranked = sorted(kernels, key=lambda kk: -kernels[kk][0])  # the dominant kernel has the largest share
    roofline = {**roof(ranked[0]), "peak_kind": peak_desc}
    roofline_other = roof(ranked[1])

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / PAGES_FWD_BWD_TFLOPS[name]) if name in PAGES_FWD_BWD_TFLOPS else None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": B, "H": H, "N": N, "d": d, "causal": causal,
                   "l2": "inputs larger than L2 (Q, K, V, dO and outputs exceed 129 MB per step)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf, "fwd_bwd_tflops": fwd_bwd_tf,
        "kernel_tflops": {kk: fl / (ms / 1e3) / 1e12 for kk, (ms, fl) in kernels.items()},
        "pct_of_peak": {"fwd": fwd_tf / burst, "fwd_bwd": fwd_bwd_tf / burst, "peak_tflops": burst,
                        "peak_kind": f"{peak_kind} burst dense bf16 (MEASURED_PEAKS.json)",
                        "vs_sustained": {"fwd": fwd_tf / sustained, "fwd_bwd": fwd_bwd_tf / sustained,
                                         "peak_tflops": sustained},
                        "vs_nominal": {"fwd": fwd_tf / NOMINAL_BF16_TFLOPS, "fwd_bwd": fwd_bwd_tf / NOMINAL_BF16_TFLOPS,
                                       "peak_tflops": NOMINAL_BF16_TFLOPS}},
        "phase_ms": {"fwd": phase_ms[0], bwd_names[0]: phase_ms[1], bwd_names[1]: phase_ms[2],
                     bwd_names[2]: phase_ms[3]},
        "phase_ms_source": "second timed pass, events between the phases (no overlap); value, ms_per_step and "
                           "the fwd/bwd rates come from the fa_fwd + fa_bwd pass",
        "roofline": roofline, "roofline_secondary": roofline_other,
        # The whole backward (all its kernels) against the same peak, with
        # the method's FLOPs (2.5x forward), not the kernels' executed ones.
        "bwd_algorithmic_frac": {"value": f_bwd / (api_bwd_ms / 1e3) / 1e12 / peak, "peak": peak,
                                 "bwd_ms": api_bwd_ms, "bwd_ms_phases_serialised": sum(phase_ms[1:])},
        # The preprocess kernel is HBM-bound: it reads O, dO (bf16) and L,
        # writes D and the base-2 L (fp32) per padded row, and on the atomic
        # path zeroes the fp32 dQ accumulator.
        # The forward's second bound: one 2^x per score on the special-function
        # unit, measured at 4 cycles per warp instruction per sub-partition
        # (32 results per clock per SM) on this GPU; peak at the sampled clock.
        "roofline_exp": {"bound": "alu", "kernel": "fa_fwd", "unit": "Gexp/s",
                         "achieved": f_fwd / (4 * d) / (phase_ms[0] / 1e3) / 1e9,
                         "peak": 32 * num_sms * clock_mhz * 1e6 / 1e9,
                         "frac": (f_fwd / (4 * d) / (phase_ms[0] / 1e3)) / (32 * num_sms * clock_mhz * 1e6)},
        "roofline_hbm": {"bound": "hbm", "kernel": "bwd_pre", "unit": "GB/s", "peak": peaks["hbm_gbs"],
                         "achieved": pre_bytes / (phase_ms[1] / 1e3) / 1e9,
                         "frac": pre_bytes / (phase_ms[1] / 1e3) / 1e9 / peaks["hbm_gbs"],
                         "bytes": pre_bytes, "avg_launch_ms": phase_ms[1]},
        "e2e": {"value": aggregate_value(f_step, world, e2e_s), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "e2e_fwd": {"value": aggregate_value(f_fwd, world, e2e_fwd_s), "unit": UNIT,
                    "h2d_bytes_per_step": 3 * q_bytes, "d2h_bytes_per_step": o_bytes + lse_bytes,
                    "steps": e2e_steps, "entry": "fa_fwd_host"},
        "gpu_launches": 4 * args.steps,
        "clocks": clk,
        "other_configs": extra,
    }
    if not args.no_cpu_baseline and world == 1:
        xs = make_inputs(1, 1, N, d, seed_for(p))
        rows = calibrate_rows(p, xs, 4.0)
        t1, _ = oracle_sample(p, xs, rows, 1)
        calls = max(1, int(round(12.0 / max(t1, 1e-3))))  # about 12 s of CPU work
        t_cpu, fl = oracle_sample(p, xs, rows, calls)
        result["cpu_baseline"] = {
            "value": fl / t_cpu / 1e12, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": (f"{calls} x float64 oracle forward+backward of {rows} query rows x all {N} keys of one head "
                       f"({t_cpu:.1f} s); FLOPs by the same convention as the GPU number")}
    return result


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(all_workloads()))
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle sample (profiling runs)")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="skip timing the long-context and d = 256 configurations after the headline step")
    ap.add_argument("--sweep", action="store_true",
                    help="print one line per point of the microbenchmark grid and the other configurations "
                         "(1 GPU, device-resident inputs) instead of the benchmark line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.sweep:
        return run_sweep(args)
    p = all_workloads()[args.workload]
    world, rank, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, p, args.workload)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        res = run_ours(args, p, args.workload, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if res is not None:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
