#!/usr/bin/env python
"""Decode-step benchmark: the 197 NF4 GEMVs of one Qwen2.5-1.5B-shaped decode step at batch 1.

One step = one replay of the step's CUDA graph: one persistent launch running all 197 GEMVs, where
each dependency level (q,k,v / o / gate,up / down / lm_head) reads x only after every GEMV of the
previous level completed.  value = algorithmic HBM bytes of the step (packed weights + scales +
x + y) / device time, in GB/s; the step's weights (871 MB) exceed the 129 MB L2, so no flush is
needed between steps.  Rank 0 prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain float64 restatement of the method) on the same
workload, a bounded row sample per step, on this machine's host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-step 4-bit GEMV µs and achieved HBM GB/s (% of GB300 roofline)"
WORKLOAD = ("Qwen2.5-1.5B-shaped decode step, batch 1: 197 NF4 GEMVs (28 layers x q 1536x1536, "
            "k 256x1536, v 256x1536, o 1536x1536, gate 8960x1536, up 8960x1536, down 1536x8960, "
            "+ lm_head 151936x1536), blocksize 64, FP32 absmax, weights N(0,0.02), x N(0,1) FP16")
FALLBACK_HBM_GBS = 6800.0
BLOCK = {"nf4": 64, "int4": 128, "fp4": 32}          # default block / group size per format
FORMAT_ID = {"nf4": 0, "int4": 1, "fp4": 2}          # w4_format of include/w4.h


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Measured dense bf16 TFLOP/s (burst), the denominator for batch >= 32 contractions (FP16
    operands have the same tensor rate)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def run_sweep(args):
    """The batch sweep of the pages' small-batch configurations: every decode shape alone at batch
    1, 8, 32 and 128, NF4, INT4 and FP4, weights N(0, 0.02) with 0.1 % outliers at 10 sigma.  One
    JSON line; not part of the default run."""
    import torch
    from weight_only_bit_gb300 import build as _b
    _b.build()
    dev = torch.device("cuda:0")
    hbm, _ = peaks()
    tfp, tsrc = bf16_peak()
    res = {}
    only = set(args.sweep_shapes.split(",")) if args.sweep_shapes else None
    for fmt in args.sweep_formats.split(","):
        for M in (int(b) for b in args.sweep_batches.split(",")):
            shapes, weighted = per_shape(fmt, dev, torch, hbm, M=M, tflops_peak=tfp, outlier_frac=0.001, only=only)
            res[f"{fmt}_b{M}"] = {"shapes": shapes, "weighted_step_us": round(weighted, 2) if only is None else None}
    print(json.dumps({"sweep": res, "hbm_peak_GB_s": hbm, "bf16_peak_TFLOP_s": tfp, "peak_source": tsrc}), flush=True)


def kernel_sha() -> str:
    h = hashlib.sha256()
    for f in ("w4_persist.cu", "w4_mma_unit.cuh", "w4_decode.cuh", "w4_common.cuh"):
        h.update(open(os.path.join(ROOT, "weight_only_bit_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic():
    """Per-launch DRAM bytes of the GEMV kernel from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "gemv_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_sha") != kernel_sha():
        return None
    return d.get("dram_bytes_per_launch_full_step")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------- oracle timing
def oracle_sample_rate(budget_s: float, fmt: str = "nf4"):
    """The oracle (as it stands) on a row sample of the step's GEMVs, for about budget_s seconds.
    Returns (GB/s of algorithmic bytes, cores, description)."""
    import numpy as np
    import oracle
    from weight_only_bit_gb300 import synth
    bs = 64 if fmt == "nf4" else 128
    code = oracle.nf4_codebook()
    pool = []
    for proj in ("q", "k", "v", "o", "gate", "up", "down"):
        n, k = synth.shape_of(proj)
        rows = min(n, 512)
        w = synth.weights(synth.weight_seed(0, proj), n, k)[:rows]
        x = synth.activations(synth.x_seed(0, synth.X_SLOT[proj], 1), 1, k)
        if fmt == "nf4":
            p, s = oracle.quantize_nf4(w, code, bs)
        else:
            p, s = oracle.quantize_int4(w, bs)
        sbytes = 4 if fmt == "nf4" else 2
        nbytes = rows * k // 2 + rows * (k // bs) * sbytes + 2 * k + 2 * rows
        pool.append((p, s, x, nbytes))
    t0 = time.perf_counter()
    done = 0
    i = 0
    while time.perf_counter() - t0 < budget_s:
        p, s, x, nb = pool[i % len(pool)]
        if fmt == "nf4":
            oracle.gemv_nf4(p, s, code, x, bs)
        else:
            oracle.gemv_int4(p, s, x, bs)
        done += nb
        i += 1
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"oracle.gemv_{fmt} (numpy float64 dequantise + BLAS matmul) over the first 512 rows of layer 0's "
            f"seven projections, {i} GEMVs in {dt:.1f} s")
    return done / dt / 1e9, cores, desc


def cpu_practical_rate(budget_s: float):
    """A practical CPU path beside the oracle (not the oracle, and not reachable from the library):
    FP32 NumPy, nibbles unpacked and decoded per weight (code-book lookup times block absmax),
    one BLAS matrix-vector product per GEMV on all cores, over the same row sample as the oracle
    baseline, for about budget_s seconds.  Returns (GB/s of algorithmic bytes, cores, description)."""
    import numpy as np
    import oracle
    from weight_only_bit_gb300 import synth
    bs = 64
    code64 = oracle.nf4_codebook()
    code = np.asarray(code64, dtype=np.float32)
    pool = []
    for proj in ("q", "k", "v", "o", "gate", "up", "down"):
        n, k = synth.shape_of(proj)
        rows = min(n, 512)
        w = synth.weights(synth.weight_seed(0, proj), n, k)[:rows]
        x = synth.activations(synth.x_seed(0, synth.X_SLOT[proj], 1), 1, k)
        p, s = oracle.quantize_nf4(w, code64, bs)
        nbytes = rows * k // 2 + rows * (k // bs) * 4 + 2 * k + 2 * rows
        pool.append((p, np.asarray(s, dtype=np.float32), x.astype(np.float32).reshape(-1), nbytes))
    t0 = time.perf_counter()
    done = 0
    i = 0
    while time.perf_counter() - t0 < budget_s:
        p, s, x, nb = pool[i % len(pool)]
        codes = np.empty((p.shape[0], 2 * p.shape[1]), dtype=np.uint8)
        codes[:, 0::2] = p >> 4
        codes[:, 1::2] = p & 15
        w = code[codes] * np.repeat(s, bs, axis=1)
        (w @ x).astype(np.float16)
        done += nb
        i += 1
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"NumPy FP32 dequantise + BLAS sgemv over the first 512 rows of layer 0's seven projections, "
            f"{i} GEMVs in {dt:.1f} s")
    return done / dt / 1e9, cores, desc


def run_reference(args):
    """The oracle timed as the reference arm: each step a bounded row sample of the workload."""
    import numpy as np
    import oracle
    from weight_only_bit_gb300 import synth
    budget = float(os.environ.get("W4_REFERENCE_BUDGET_S", "60"))
    per_step = budget / max(1, args.steps + args.warmup)
    code = oracle.nf4_codebook()
    shapes = [(proj,) + synth.shape_of(proj) for proj in ("q", "k", "v", "o", "gate", "up", "down", "lm_head")]
    mats = {}
    for proj, n, k in shapes:
        rows = min(n, 256)
        w = synth.weights(synth.weight_seed(28 if proj == "lm_head" else 0, proj), n, k)[:rows] \
            if proj != "lm_head" else synth.weights(synth.weight_seed(28, proj), rows, k)
        p, s = oracle.quantize_nf4(w, code, 64)
        x = synth.activations(synth.x_seed(0, synth.X_SLOT[proj], 1), 1, k)
        mats[proj] = (p, s, x, k)
    # rows per step from a calibration call
    p, s, x, k = mats["gate"]
    t0 = time.perf_counter()
    oracle.gemv_nf4(p, s, code, x, 64)
    per_row = (time.perf_counter() - t0) / p.shape[0]
    rows_per_step = max(1, min(256, int(per_step / max(per_row, 1e-9))))
    order = [proj for _, proj, _, _ in synth.decode_step_gemvs()]
    total_b, total_t = 0, 0.0
    for it in range(args.warmup + args.steps):
        proj = order[it % len(order)]
        p, s, x, k = mats[proj]
        r = min(rows_per_step, p.shape[0])
        t0 = time.perf_counter()
        oracle.gemv_nf4(p[:r], s[:r], code, x, 64)
        dt = time.perf_counter() - t0
        if it >= args.warmup:
            total_t += dt
            total_b += r * k // 2 + r * (k // 64) * 4 + 2 * k + 2 * r
    gbs = total_b / total_t / 1e9
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"oracle.gemv_nf4 on {rows_per_step} rows per step of the step's GEMVs in order "
              f"(float64 numpy), {args.steps} timed steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_t / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "format": "nf4"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------- GPU arm
def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time per step (replicas: every rank times the same workload)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: the bytes every rank moved in one step over the slowest rank's time."""
    return bytes_per_rank * world / (ms_max * 1e-3) / 1e9


def time_graph(step, stream, steps, warmup, torch):
    for _ in range(warmup):
        step.launch(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step.launch(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


class _GraphRunner:
    """A torch CUDA graph around libw4 calls (used for chains of separate launches)."""

    def __init__(self, torch, stream, fn):
        self.g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()                       # warm (lazy init outside capture)
        torch.cuda.synchronize()
        with torch.cuda.graph(self.g, stream=stream):
            fn()

    def launch(self, stream):
        import torch
        with torch.cuda.stream(stream):     # replay on the stream the timing events are recorded on
            self.g.replay()
        return 0


def per_shape(fmt, dev, torch, hbm, M=1, tflops_peak=None, outlier_frac=0.0, only=None):
    """Each decode shape alone at batch M: a chain of back-to-back launches (one per weight copy,
    distinct copies totalling > 4x L2, so every launch streams from HBM) replayed as a graph; the
    time per launch is what one such GEMV costs inside a launch-per-GEMV decode step."""
    import weight_only_bit_gb300 as w4
    from weight_only_bit_gb300 import synth
    from weight_only_bit_gb300 import _lib
    bs = BLOCK[fmt]
    out = {}
    code = None
    if fmt == "nf4":
        st, c = w4.w4_nf4_codebook()
        code = torch.tensor(c, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    for name, n, k, _ in synth.DECODE_SHAPES:
        if only is not None and name not in only:
            continue
        w = synth.weights(synth.weight_seed(0 if name != "lm_head" else 28, name), n, k, outlier_frac=outlier_frac)
        W = torch.from_numpy(w).to(dev)
        packed = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
        sdt = torch.float32 if fmt == "nf4" else torch.float16
        sc = torch.empty((n, k // bs), dtype=sdt, device=dev)
        if fmt == "nf4":
            w4.check(w4.w4_quantize_nf4(W, packed, sc, code, n, k, bs))
        elif fmt == "int4":
            w4.check(w4.w4_quantize_int4(W, packed, sc, n, k, bs))
        else:
            w4.check(w4.w4_quantize_fp4(W, packed, sc, n, k, bs))
        del W
        per = n * k // 2 + sc.numel() * sc.element_size()
        copies = max(2, min(4096, (4 * 129 * 2 ** 20) // per + 1))
        P = packed.reshape(1, -1).repeat(copies, 1)
        S = sc.reshape(1, -1).repeat(copies, 1)
        x = torch.from_numpy(synth.activations(synth.x_seed(0, synth.X_SLOT[name], M), M, k)).to(dev)
        y = torch.empty((M, n), dtype=torch.float16, device=dev)
        descs = [dict(format=FORMAT_ID[fmt], packed=P[i], scales=S[i],
                      codebook=code, x=x, y=y, M=M, N=n, K=k, blocksize=bs) for i in range(copies)]
        arr = w4._descs(descs)
        lib = w4.lib()
        runner = _GraphRunner(torch, stream, lambda: w4.check(lib.w4_gemv_sequence(arr, len(descs),
                                                                                  stream.cuda_stream)))
        ms = time_graph(runner, stream, 5, 2, torch) / copies
        nbytes = per + 2 * M * k + 2 * M * n
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"N": n, "K": k, "us": round(ms * 1e3, 3), "GB_s": round(gbs, 1),
                     "frac_of_measured": round(gbs / hbm, 4), "launches_timed": copies * 5}
        if M >= 32:
            tf = 2.0 * M * n * k / (ms * 1e-3) / 1e12
            out[name]["TFLOP_s"] = round(tf, 1)
            if tflops_peak:
                out[name]["frac_of_bf16_peak"] = round(tf / tflops_peak, 4)
        del runner, P, S
        torch.cuda.empty_cache()
    # the pages' "weighted" step: sum over shapes of count x per-launch time
    weighted_us = sum(out[nm]["us"] * c for nm, _, _, c in synth.DECODE_SHAPES if nm in out)
    return out, weighted_us


def run_ours(args):
    import torch
    import torch.distributed as dist
    import weight_only_bit_gb300 as w4
    from weight_only_bit_gb300 import build as _b
    from weight_only_bit_gb300.step import DecodeStep

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    if rank == 0 or world == 1:
        _b.build()
    if world > 1:
        dist.barrier()
    hbm, peak_src = peaks()

    step = DecodeStep("nf4", batch=1, device=str(dev), levels="grouped").build().capture()
    nbytes = step.bytes_per_step()
    nlaunch = len(step.gemvs)
    stream = torch.cuda.Stream(dev)

    # warm-up, then the timed region bracketed by barrier + synchronize, clocks sampled inside
    for _ in range(args.warmup):
        step.launch(stream)
    torch.cuda.synchronize()
    w4.check(w4.w4_device_check(stream), "warm-up")
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    l0 = w4.w4_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        w4.check(step.launch(stream))
    e1.record(stream)
    torch.cuda.synchronize()
    launches = w4.w4_launch_count() - l0
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    w4.check(w4.w4_device_check(stream), "timed region")
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    value = job_gbs(nbytes, world, ms_max)

    # distribution of single steps (each bracketed by its own events, back to back, after the
    # timed region): p10 / median / p90
    nlat = 200
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nlat)]
    for a, b in evs:
        a.record(stream)
        step.launch(stream)
        b.record(stream)
    torch.cuda.synchronize()
    lat = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    step_us_pct = {"p10": round(lat[nlat // 10], 2), "p50": round(lat[nlat // 2], 2), "p90": round(lat[9 * nlat // 10], 2),
                   "steps": nlat}

    # end to end through the public API with host buffers: w4_step_run_host copies every x in from
    # pinned host memory, runs the step and copies every y out, all on the stream
    x_pin = torch.from_numpy(step.x_host).pin_memory()
    y_pin = torch.empty(step.y_elems, dtype=torch.float16).pin_memory()
    e2e_steps = max(20, args.steps // 10)
    for _ in range(3):
        w4.check(step.run_host(x_pin, y_pin, stream))
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        w4.check(step.run_host(x_pin, y_pin, stream))
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = f0.elapsed_time(f1) / e2e_steps
    e2e = {"value": round(nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": int(step.x_elems * 2), "d2h_bytes_per_step": int(step.y_elems * 2),
           "ms_per_step": round(e2e_ms, 5), "call": "w4_step_run_host (H2D of x, the step's graph, D2H of y)"}

    extra = {}
    if rank == 0 and not args.quick:
        # the same step with a level per GEMV, and as 197 separate back-to-back launches
        nrep = max(100, args.steps // 4)
        ss = DecodeStep("nf4", batch=1, device=str(dev), levels="strict")
        ss.packed, ss.scales, ss.code, ss.x, ss.y, ss.x_host = step.packed, step.scales, step.code, step.x, step.y, \
            step.x_host
        ss.capture()
        ms_s = time_graph(ss, stream, nrep, args.warmup, torch)
        ss.close()
        extra["strict_levels_step"] = {"us": round(ms_s * 1e3, 2), "GB_s": round(nbytes / (ms_s * 1e-3) / 1e9, 1),
                                       "frac_of_measured": round(nbytes / (ms_s * 1e-3) / 1e9 / hbm, 4),
                                       "levels": 197, "launches_per_step": 1}
        arr = w4._descs(step.descriptors())
        lib = w4.lib()
        chain = _GraphRunner(torch, stream, lambda: w4.check(lib.w4_gemv_sequence(arr, nlaunch, stream.cuda_stream)))
        ms_c = time_graph(chain, stream, nrep, args.warmup, torch)
        del chain
        extra["launch_per_gemv_step"] = {"us": round(ms_c * 1e3, 2),
                                         "GB_s": round(nbytes / (ms_c * 1e-3) / 1e9, 1),
                                         "frac_of_measured": round(nbytes / (ms_c * 1e-3) / 1e9 / hbm, 4),
                                         "launches_per_step": nlaunch}
        # the other formats' steps at batch 1, and the small batches of the decode step (same
        # shapes, grouped levels, one persistent launch each)
        for tag, fmt, batch in (("int4_step", "int4", 1), ("fp4_step", "fp4", 1), ("nf4_step_b4", "nf4", 4),
                                ("nf4_step_b8", "nf4", 8), ("int4_step_b8", "int4", 8)):
            s4 = DecodeStep(fmt, batch=batch, device=str(dev), levels="grouped").build().capture()
            ms4 = time_graph(s4, stream, nrep, args.warmup, torch)
            b4 = s4.bytes_per_step()
            extra[tag] = {"us": round(ms4 * 1e3, 2), "GB_s": round(b4 / (ms4 * 1e-3) / 1e9, 1),
                          "frac_of_measured": round(b4 / (ms4 * 1e-3) / 1e9 / hbm, 4), "bytes": b4,
                          "batch": batch, "format": fmt, "group": BLOCK[fmt]}
            s4.close()
            del s4
            torch.cuda.empty_cache()
        shapes, weighted = per_shape("nf4", dev, torch, hbm)
        extra["per_shape_nf4"] = shapes
        extra["weighted_step_us_nf4"] = round(weighted, 2)
        # the small-shape configuration: NF4 256 x 1536 at batch 1 (the k / v projection)
        extra["c1_nf4_256x1536_b1"] = shapes["k"]
        # small batches on gate, down and q (NF4 and INT4, batch 8 and 32)
        c4 = {}
        tfp, _ = bf16_peak()
        for fmt in ("nf4", "int4"):
            for M in (8, 32):
                sh, _ = per_shape(fmt, dev, torch, hbm, M=M, tflops_peak=tfp, only={"gate", "down", "q"})
                c4[f"{fmt}_b{M}"] = sh
        extra["c4_small_batches"] = c4
        # prefill-sized batches on the lm_head: 256-row batch tiles (one pass over the weights per
        # 256 rows)
        pre = {}
        for M in (256, 512):
            sh, _ = per_shape("nf4", dev, torch, hbm, M=M, tflops_peak=tfp, only={"lm_head"})
            pre[f"nf4_b{M}"] = sh["lm_head"]
        extra["prefill_lm_head"] = pre
        # read-only streaming ceiling: a library reduction reading a 2 GiB buffer once per pass
        buf = torch.ones(1 << 29, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(3):
                torch.amax(buf)
            r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            r0.record(stream)
            for _ in range(10):
                torch.amax(buf)
            r1.record(stream)
        torch.cuda.synchronize()
        ro = 10 * buf.numel() * 4 / (r0.elapsed_time(r1) * 1e-3) / 1e9
        extra["read_only_ceiling"] = {"GB_s": round(ro, 1), "frac_of_measured": round(ro / hbm, 4),
                                      "kernel": "torch.amax over a 2 GiB FP32 buffer (library reduction, "
                                                "every byte read once per pass)"}
        del buf
        torch.cuda.empty_cache()
    step.close()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs_cpu, cores, desc = oracle_sample_rate(float(os.environ.get("W4_CPU_BASELINE_S", "12")))
        cpu = {"value": round(gbs_cpu, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}
        gbs_p, cores_p, desc_p = cpu_practical_rate(float(os.environ.get("W4_CPU_PRACTICAL_S", "8")))
        extra["cpu_practical"] = {"value": round(gbs_p, 4), "unit": "GB/s", "cores": cores_p,
                                  "kind": "numpy FP32 dequantise-on-the-fly", "sample": desc_p}

    if rank == 0:
        achieved = nbytes / (ms_max * 1e-3) / 1e9     # one launch per step
        traffic = ncu_traffic()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "us_per_step": round(ms_max * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": 1, "format": "nf4", "gemvs": nlaunch,
                       "bytes_per_step": nbytes, "parallelism": "replicas" if world > 1 else "single",
                       "l2": "no flush: 871 MB of distinct weights per step > 129 MB L2",
                       "launch": "one persistent launch per step (113 dependency levels), replayed as a CUDA graph"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "traffic": traffic,
                         "peak_source": peak_src, "kernel": "w4_persistent_kernel<NF4,1> (the whole step)"},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches), "clocks": clocks,
            "frac_of_nominal_8TBs": round(value / world / 8000.0, 4),
            "step_us_percentiles": step_us_pct,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="skip the INT4 step and the per-shape table")
    ap.add_argument("--sweep", action="store_true", help="only the per-shape batch sweep (1, 8, 32, 128; NF4, INT4)")
    ap.add_argument("--sweep-batches", default="1,8,32,128", help="batches of the sweep, comma-separated")
    ap.add_argument("--sweep-formats", default="nf4,int4,fp4", help="formats of the sweep, comma-separated")
    ap.add_argument("--sweep-shapes", default="", help="decode shapes of the sweep (default: all), comma-separated")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
