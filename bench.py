#!/usr/bin/env python
"""Throughput of the batched power-of-two C2C FFT on one GB300 (or N, one
process per GPU, each with its own full batch: weak scaling).

Default workload (``--config c2``): 16384 transforms of 4096 fp32 complex
points (512 MiB), a step = forward then inverse (1/N).  Inputs are larger
than L2 (129 MB), so no flush between steps is needed.

Metric: effective GB/s = algorithmic HBM bytes of the step / step time,
where the algorithmic bytes of one transform call are (HBM passes of the
chosen plan) x 2 x (bytes of the complex array); the on-chip path makes one
pass.  Also reported: 5 N log2 N GFLOP/s, transforms/s, the roofline of
the dominant kernel against the measured HBM copy bandwidth, the fp64 CPU
oracle on a bounded sample, an end-to-end figure with host buffers, and
the SM clocks sampled during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c1..c5]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed alone
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

GIB = float(1 << 30)


def log2i(n: int) -> int:
    return int(n).bit_length() - 1


# ---------------------------------------------------------------------------
# Workload descriptions (bytes / flops / units per step)
# ---------------------------------------------------------------------------

SIZE_OVERRIDE = {}


def config_of(name: str) -> dict:
    """The workload's sizes, with any --n / --batch override applied."""
    c = dict(workloads.CONFIGS[name])
    c.update(SIZE_OVERRIDE)
    return c


def smooth_2357(n: int) -> bool:
    for f in (2, 3, 5, 7):
        while n % f == 0:
            n //= f
    return n == 1


def planned_passes(logn: int, pass_log: int) -> int:
    """HBM passes the library plans for a 2^logn-point transform beyond the
    on-chip length: the FFT_GB300_PASS_SPLIT / FFT_GB300_PASS_LOG tuning
    overrides when set (as the planner reads them), else factors of at most
    pass_log bits."""
    split = os.environ.get("FFT_GB300_PASS_SPLIT", "")
    try:
        parts = [int(v) for v in split.split(",")] if split else []
    except ValueError:
        parts = []
    if len(parts) >= 2 and sum(parts) == logn and all(1 <= v <= 14 for v in parts):
        return len(parts)
    env_log = os.environ.get("FFT_GB300_PASS_LOG", "")
    if env_log.isdigit() and int(env_log) >= 4:
        pass_log = min(int(env_log), 14)
    return max(2, math.ceil(logn / pass_log))


def workload_info(name: str, pass_log: int = 9):
    c = config_of(name)
    n, batch = c["n"], c["batch"]
    if c["kind"] == "fft1d":
        elem = 8
        arr = n * batch * elem
        directions = 1 if name in ("c1", "c3") else 2
        info = dict(kind="fft1d", n=n, batch=batch, directions=directions, array_bytes=arr,
                    transforms_per_step=directions * batch, h2d=arr, d2h=arr,
                    flops_per_step=directions * 5.0 * n * math.log2(max(n, 2)) * batch)
        if n & (n - 1) == 0:
            passes = 1 if log2i(n) <= 14 else planned_passes(log2i(n), pass_log)
        elif smooth_2357(n) and 64 < n <= 12288:
            passes = 1    # mixed radix on chip: one read, one write
            info.update(mixed=True)
        elif smooth_2357(n):
            passes = 5    # four-step: 3 transposes + 2 on-chip mixed-radix passes
            info.update(four_step=True)
        else:
            # Bluestein: a length-M cyclic convolution per row, M = 2^ceil(log2(2n - 1));
            # fused on chip (one read, one write) while M <= 2^14.
            M = 1 << (2 * n - 2).bit_length()
            passes = 1 if M <= 1 << 14 else None
            info.update(bluestein_m=M, alu_flops_per_row=2 * 5.0 * M * log2i(M) + 6.0 * M
                        + 12.0 * n)
        info.update(passes=passes, bytes_per_step=directions * (passes or 1) * 2 * arr,
                    ideal_bytes_per_step=directions * 2 * arr)
        return info
    if c["kind"] == "real":
        # R2C then C2R: samples (4 B) read and bins (8 B, n/2 + 1 per row)
        # written, then the reverse.
        H = n // 2
        pw2 = H > 0 and H & (H - 1) == 0 and n % 2 == 0
        passes = 1 if pw2 and log2i(H) <= 14 else None
        rb, cb = n * 4 * batch, (H + 1) * 8 * batch
        return dict(
            kind="real", n=n, batch=batch, passes=passes, directions=2, array_bytes=rb,
            bytes_per_step=2 * (rb + cb), ideal_bytes_per_step=2 * (rb + cb),
            flops_per_step=2 * 2.5 * n * math.log2(max(n, 2)) * batch,
            transforms_per_step=2 * batch, h2d=rb, d2h=rb)
    if c["kind"] == "fftnd":
        npts = 1
        for v in c["shape"]:
            npts *= v
        arr = npts * batch * 8
        passes = sum(1 for v in c["shape"] if v > 1)
        return dict(
            kind="fftnd", n=n, batch=batch, passes=passes, directions=2, array_bytes=arr,
            bytes_per_step=2 * passes * 2 * arr, ideal_bytes_per_step=2 * 2 * arr,
            flops_per_step=2 * 5.0 * npts * log2i(npts) * batch,
            transforms_per_step=2 * batch, h2d=arr, d2h=arr)
    if c["kind"] == "fft2d":
        arr = n * n * batch * 8
        return dict(
            kind="fft2d", n=n, batch=batch, passes=2, directions=2, array_bytes=arr,
            bytes_per_step=2 * 2 * 2 * arr, ideal_bytes_per_step=2 * 2 * arr,
            flops_per_step=2 * 5.0 * n * n * log2i(n * n) * batch,
            transforms_per_step=2 * batch, h2d=arr, d2h=arr)
    if c["kind"] == "conv":
        nh = c["nh"]
        ny = n + nh - 1
        L = 1 << (ny - 1).bit_length()
        return dict(
            kind="conv", n=n, nh=nh, batch=batch, L=L, passes=1, directions=2,
            array_bytes=batch * n * 4,
            bytes_per_step=batch * n * 4 + nh * 4 + batch * ny * 4,   # x, h read; y written
            ideal_bytes_per_step=batch * n * 4 + nh * 4 + batch * ny * 4,
            flops_per_step=2 * 5.0 * L * log2i(L) * ((batch + 1) // 2),
            transforms_per_step=2 * ((batch + 1) // 2), h2d=batch * n * 4 + nh * 4,
            d2h=batch * ny * 4)
    # polymul: fused ideal = int64 inputs read once + int64 output written once
    nc = 2 * n - 1
    L = 1 << (nc - 1).bit_length()
    return dict(
        kind="polymul", n=n, batch=batch, L=L, passes=None, directions=3,
        array_bytes=batch * L * 16,
        bytes_per_step=batch * (2 * n * 8 + nc * 8),
        ideal_bytes_per_step=batch * (2 * n * 8 + nc * 8),
        flops_per_step=3 * 5.0 * L * log2i(L) * batch,
        # the transforms the pipeline actually runs: one of length L (both
        # inputs packed as a + ib) and one of length L/2 (the real product)
        fp64_flops_per_step=(5.0 * L * log2i(L) + 5.0 * (L // 2) * log2i(L // 2)) * batch,
        transforms_per_step=3 * batch, h2d=batch * 2 * n * 8, d2h=batch * nc * 8)


# ---------------------------------------------------------------------------
# Clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Committed ncu traffic summary (null once the kernels have changed)
# ---------------------------------------------------------------------------

# Sources of the kernels each workload's roofline entry measures.
KERNEL_SOURCES = {
    "c1": ["fft_device.cuh", "fft_rows.cuh", "fft_rows_f32.cu"],
    "c2": ["fft_device.cuh", "fft_rows.cuh", "fft_rows_f32.cu"],
    "c3": ["fft_device.cuh", "fft_pass.cuh", "fft_pass_tma.cuh", "fft_pass_cluster.cuh",
           "fft_pass_f32.cu", "fft_plan.cu", "fft_exec.cu", "plan.h"],
    "c4": ["fft_device.cuh", "fft_rows.cuh", "fft_rows_f32.cu", "fft_pass.cuh",
           "fft_pass_tma.cuh", "fft_pass_cluster.cuh", "fft_pass_f32.cu", "fft_plan.cu",
           "fft_exec.cu", "plan.h"],
    "c5": ["fft_device.cuh", "fft_pass.cuh", "fft_pass_tma.cuh", "fft_pass_cluster.cuh",
           "fft_pass_f64.cu", "polymul.cu"],
    "conv1": ["fft_device.cuh", "fft_rows.cuh", "conv.cuh", "conv_f32.cu"],
    "any1": ["fft_device.cuh", "mixed.cuh", "mixed_f32.cu", "fft_plan.cu", "fft_exec.cu", "plan.h"],
    "any2": ["fft_device.cuh", "fft_rows.cuh", "conv.cuh", "anylen.cuh", "anylen_f32.cu"],
    "any3": ["fft_device.cuh", "mixed.cuh", "mixed_f32.cu", "transpose.cu", "fft_plan.cu", "fft_exec.cu", "plan.h"],
    "real1": ["fft_device.cuh", "fft_rows.cuh", "real.cuh", "real_f32.cu"],
    "nd1": ["fft_device.cuh", "fft_rows.cuh", "fft_rows_t.cuh", "rows_t_f32.cu", "fft_plan.cu", "fft_exec.cu", "plan.h"],
}


def kernel_source_hash(config: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fft_convolution_gb300", "csrc")
    for fn in sorted(KERNEL_SOURCES[config]):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(config: str):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    ent = data.get(config)
    if not ent or ent.get("source_hash") != kernel_source_hash(config):
        return None
    return ent


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------

def cpu_oracle_sample(name: str, budget_s: float = 12.0):
    """Times the fp64 oracle (recursive Cooley-Tukey; schoolbook-free fp64
    pipeline for polymul) on a bounded sample of the workload and scales to
    the metric's unit.  Single-threaded."""
    import oracle
    info = workload_info(name)
    c = config_of(name)
    t0 = time.perf_counter()
    done_units = 0.0  # fraction of one step's work
    sample = ""
    if info["kind"] == "fft1d":
        n = c["n"]
        if n <= 1 << 16:
            x = workloads.config_input(name, scale_batch=min(c["batch"], 64)).astype(np.complex128)
            pow2 = n & (n - 1) == 0
            fwd = oracle.fft if pow2 else oracle.dft          # any length: the direct DFT
            k = 0
            while time.perf_counter() - t0 < budget_s and k < x.shape[0] * 64:
                r = x[k % x.shape[0]]
                y = fwd(r)
                if info["directions"] == 2:
                    oracle.ifft(y) if pow2 else oracle.dft(y, +1)
                k += 1
            done_units = k / c["batch"]
            sample = f"{k} of {c['batch']} transforms of N={n}" + \
                (" (forward+inverse)" if info["directions"] == 2 else "")
        elif n & (n - 1):
            # a long length that is not a power of two: the oracle is the direct
            # DFT; time bins of one row (O(N) each) and scale by the bins of the step
            x = workloads.config_input(name, scale_batch=1)[0].astype(np.complex128)
            bins = 0
            while time.perf_counter() - t0 < budget_s and bins < n:
                oracle.dft_bins(x, np.arange(bins, bins + 64, dtype=np.int64) % n)
                bins += 64
            done_units = bins / (n * c["batch"] * info["directions"])
            sample = f"{bins} bins of one N={n} row by the direct sum, scaled to the step"
        else:
            # one long transform: time a 2^20 transform and scale by N log N
            m = 1 << 20
            x = workloads.normal_complex(m, 99, np.complex128)
            k = 0
            while time.perf_counter() - t0 < budget_s and k < 64:
                oracle.fft(x)
                k += 1
            done_units = k * (m * log2i(m)) / (n * log2i(n))
            sample = f"{k} transforms of N=2^20 scaled by N log2 N to N={n}"
    elif info["kind"] == "fft2d":
        n = c["n"]
        img = workloads.normal_complex((1, n, n), 4, np.complex128)[0]
        k = 0
        while time.perf_counter() - t0 < budget_s and k < 8:
            X = oracle.fft2d(img)
            oracle.fft2d(X, +1)
            k += 1
        done_units = k / c["batch"]
        sample = f"{k} of {c['batch']} images {n}x{n} (forward+inverse)"
    elif info["kind"] == "fftnd":
        vol = workloads.normal_complex((1,) + tuple(c["shape"]), c["seed"], np.complex128)
        k = 0
        while time.perf_counter() - t0 < budget_s and k < 4:
            Y = oracle.fftn(vol, len(c["shape"]))
            oracle.fftn(Y, len(c["shape"]), +1)
            k += 1
        done_units = k / c["batch"]
        sample = f"{k} of {c['batch']} volumes {c['shape']} (forward+inverse)"
    elif info["kind"] == "real":
        x = workloads.normal_real((64, c["n"]), c["seed"], np.float64)
        k = 0
        while time.perf_counter() - t0 < budget_s and k < 64 * 64:
            oracle.irfft(oracle.rfft(x[k % 64]), c["n"])
            k += 1
        done_units = k / c["batch"]
        sample = f"{k} of {c['batch']} real rows of N={c['n']} (forward+inverse)"
    elif info["kind"] == "conv":
        x, h = workloads.conv_signals(64, c["n"], c["nh"], c["seed"])
        k = 0
        while time.perf_counter() - t0 < budget_s and k < 64:
            oracle.convolve(x[k].astype(np.complex128), h.astype(np.complex128))
            k += 1
        done_units = k / c["batch"]
        sample = f"{k} of {c['batch']} signals (direct sum, {c['n']} x {c['nh']} taps)"
    else:
        n = c["n"]
        m = 1 << 16
        a, b = workloads.poly_coeffs(m, 5)
        k = 0
        while time.perf_counter() - t0 < budget_s and k < 64:
            oracle.polymul_fft(a, b)
            k += 1
        L, Lm = info["L"], 1 << (2 * m - 1 - 1).bit_length()
        done_units = k * (Lm * log2i(Lm)) / (L * log2i(L)) / c["batch"]
        sample = f"{k} fp64 products of 2^16-coefficient pairs, scaled by L log2 L"
    el = time.perf_counter() - t0
    gbs = info["bytes_per_step"] * done_units / el / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
            "seconds": round(el, 3)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def max_over_ranks(value: float, world: int, device=None) -> float:
    """The maximum of `value` over all ranks (the job's time is its slowest
    rank's); the identity when world == 1."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_host_steps(step, stream, steps: int, warmup: int = 2) -> dict:
    """Times `step` (host buffers in, host buffers out, asynchronous on
    `stream`) with CUDA events around each step after `warmup` untimed ones;
    the median step is the figure (host-memory effects make single steps
    noisy)."""
    import torch
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return {"median_ms": statistics.median(times), "mean_ms": statistics.mean(times),
            "min_ms": min(times), "steps": steps}


def whole_job_value(bytes_per_step: float, world: int, ms_step: float) -> float:
    """Weak scaling: every rank moves bytes_per_step per step; the job's GB/s
    is all ranks' bytes over the slowest rank's step time."""
    return bytes_per_step * world / (ms_step * 1e-3) / 1e9


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import fft_convolution_gb300 as fg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    name = args.config
    c = config_of(name)
    info = workload_info(name)
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)

    # Inputs: seeded on the host, resident in HBM before timing.
    if info["kind"] == "conv":
        xc_h, hc_h = workloads.conv_signals(c["batch"], c["n"], c["nh"], c["seed"])
        xc_d, hc_d = torch.from_numpy(xc_h).to(dev), torch.from_numpy(hc_h).to(dev)
        ny = c["n"] + c["nh"] - 1
        yc_d = torch.empty(c["batch"], ny, dtype=torch.float32, device=dev)
        plans = []

        def step(events=None):
            if events is not None:
                events[0].record(stream)
            rc = fg.fft_convolve(xc_d.data_ptr(), c["n"], hc_d.data_ptr(), c["nh"],
                                 yc_d.data_ptr(), c["batch"], 0, fg.FFT_CONV_REAL,
                                 fg.FFT_C2C_F32, sh)
            if events is not None:
                events[1].record(stream)
            assert rc == 0, fg.fft_status_string(rc)
        kernels_per_step = fg.fft_convolve_num_kernels(c["n"], c["nh"], c["batch"], 0,
                                                       fg.FFT_CONV_REAL, fg.FFT_C2C_F32)
    elif info["kind"] == "polymul":
        a_h, b_h = workloads.poly_coeffs((c["batch"], c["n"]), c["seed"])
        a_d, b_d = torch.from_numpy(a_h).to(dev), torch.from_numpy(b_h).to(dev)
        c_d = torch.empty(c["batch"], 2 * c["n"] - 1, dtype=torch.int64, device=dev)
        plans = []

        def step(events=None):
            with torch.cuda.stream(stream):
                if events is not None:
                    events[0].record(stream)
                rc = fg.polymul_batched(a_d.data_ptr(), c["n"], b_d.data_ptr(), c["n"],
                                        c_d.data_ptr(), c["batch"], sh)
                if events is not None:
                    events[1].record(stream)
            assert rc == 0, fg.fft_status_string(rc)
        kernels_per_step = fg.polymul_num_kernels(c["n"], c["n"])
    elif info["kind"] == "real":
        x_h = sized_input(name, c)
        x_d = torch.from_numpy(x_h).to(dev)
        n, batch = c["n"], c["batch"]
        X_d = torch.empty(batch, n // 2 + 1, dtype=torch.complex64, device=dev)
        y_d = torch.empty_like(x_d)
        pf = fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_REAL_F32)
        pi = fg.Plan(n, batch, 1, fg.FFT_INVERSE, fg.FFT_REAL_F32)
        plans = [pf, pi]

        def step(events=None):
            if events is not None:
                events[0].record(stream)
            r0 = fg.fft_exec(pf.handle, x_d.data_ptr(), X_d.data_ptr(), sh)
            if events is not None:
                events[1].record(stream)
            r1 = fg.fft_exec(pi.handle, X_d.data_ptr(), y_d.data_ptr(), sh)
            if events is not None:
                events[2].record(stream)
            assert r0 == 0 and r1 == 0, (fg.fft_status_string(r0), fg.fft_status_string(r1))
        kernels_per_step = pf.num_kernels + pi.num_kernels
    else:
        x_h = sized_input(name, c)
        x_d = torch.from_numpy(x_h).to(dev)
        y_d = torch.empty_like(x_d)
        z_d = torch.empty_like(x_d)
        dims = 2 if info["kind"] == "fft2d" else 1
        n, batch = c["n"], c["batch"]
        shape = tuple(c["shape"]) if info["kind"] == "fftnd" else None
        pf = fg.Plan(n, batch, dims, fg.FFT_FORWARD, fg.FFT_C2C_F32, shape=shape)
        plans = [pf]
        if info["directions"] == 2:
            pi = fg.Plan(n, batch, dims, fg.FFT_INVERSE, fg.FFT_C2C_F32, shape=shape)
            plans.append(pi)

        def step(events=None):
            rcs = []
            if events is not None:
                events[0].record(stream)
            rcs.append(fg.fft_exec(pf.handle, x_d.data_ptr(), y_d.data_ptr(), sh))
            if events is not None:
                events[1].record(stream)
            if len(plans) == 2:
                rcs.append(fg.fft_exec(plans[1].handle, y_d.data_ptr(), z_d.data_ptr(), sh))
                if events is not None:
                    events[2].record(stream)
            assert all(r == 0 for r in rcs), [fg.fft_status_string(r) for r in rcs]
        kernels_per_step = sum(p.num_kernels for p in plans)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # Clock sampling: nvidia-smi samples every 100 ms, longer than most timed
    # regions here, so the sampler runs over an untimed soak of the same
    # steps (>= args.clock_soak seconds of load) that leads straight into
    # the timed region; the clocks reported are those of the GPU under this
    # load.
    nev = 3
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.clock_soak:
        for _ in range(4):
            step()
        torch.cuda.synchronize(dev)

    # Timed region.
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        step(ev[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    ms_step = ms_total / args.steps

    # Per-launch durations of the dominant kernel (the forward transform;
    # for 1-kernel plans that is one launch per exec).
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    inv_ms = [e[1].elapsed_time(e[2]) for e in ev] if info["kind"] in ("fft1d", "fft2d", "fftnd",
                                                                        "real") and \
        info["directions"] == 2 else []

    # End-to-end through the host-buffer entry point: pinned host input ->
    # device, transforms, device -> pinned host output, every step.
    e2e = None
    if info["kind"] in ("fft1d", "fft2d", "fftnd", "real") and not args.no_e2e:
        h_in = torch.from_numpy(x_h).pin_memory()
        h_out = torch.empty_like(h_in).pin_memory()
        e2e_steps = max(5, min(args.steps, 10))
        # Chunks of the batch stream through the device: uploads, transforms
        # and downloads of different chunks overlap (fft_exec_host_chain).
        chunk = max(1, c["batch"] // args.e2e_chunks)
        # Samples in x_d, spectra in X_d for the real round trip.
        dev_b = X_d if info["kind"] == "real" else y_d

        def e2e_step():
            plans[0].chain_host(plans[1:], h_in, h_out, x_d, dev_b, chunk, stream)
        t = time_host_steps(e2e_step, stream, e2e_steps)
        e2e_ms = t["median_ms"]
        e2e = {"value": info["bytes_per_step"] * world / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": info["h2d"], "d2h_bytes_per_step": info["d2h"],
               "ms_per_step": round(e2e_ms, 4), "ms_mean": round(t["mean_ms"], 4),
               "ms_min": round(t["min_ms"], 4), "timed_steps": e2e_steps,
               "chunk_transforms": chunk}
    elif info["kind"] == "conv" and not args.no_e2e:
        hx = torch.from_numpy(xc_h).pin_memory()
        hy = torch.empty(yc_d.shape, dtype=torch.float32).pin_memory()
        chunk = max(1, c["batch"] // args.e2e_chunks)

        def e2e_step():
            # Chunks of rows stream through the device (fft_convolve_host).
            rc = fg.fft_convolve_host(hx.data_ptr(), c["n"], hc_d.data_ptr(), c["nh"],
                                      hy.data_ptr(), c["batch"], 0, fg.FFT_CONV_REAL,
                                      fg.FFT_C2C_F32, xc_d.data_ptr(), yc_d.data_ptr(), chunk, sh)
            assert rc == 0, fg.fft_status_string(rc)
        t = time_host_steps(e2e_step, stream, max(5, min(args.steps, 10)))
        e2e_ms = t["median_ms"]
        e2e = {"value": info["bytes_per_step"] * world / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": info["h2d"], "d2h_bytes_per_step": info["d2h"],
               "ms_per_step": round(e2e_ms, 4), "ms_mean": round(t["mean_ms"], 4),
               "ms_min": round(t["min_ms"], 4), "timed_steps": t["steps"]}
    elif info["kind"] == "polymul" and not args.no_e2e:
        ha, hb = torch.from_numpy(a_h).pin_memory(), torch.from_numpy(b_h).pin_memory()
        hc = torch.empty(c_d.shape, dtype=torch.int64).pin_memory()

        chunk = max(1, c["batch"] // args.e2e_chunks)

        def e2e_step():
            # Chunks of pairs stream through the device (polymul_batched_host).
            rc = fg.polymul_batched_host(ha.data_ptr(), c["n"], hb.data_ptr(), c["n"],
                                         hc.data_ptr(), c["batch"], a_d.data_ptr(),
                                         b_d.data_ptr(), c_d.data_ptr(), chunk, sh)
            assert rc == 0, fg.fft_status_string(rc)
        t = time_host_steps(e2e_step, stream, 5, warmup=2)
        e2e_ms = t["median_ms"]
        e2e = {"value": info["bytes_per_step"] * world / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": info["h2d"], "d2h_bytes_per_step": info["d2h"],
               "ms_per_step": round(e2e_ms, 4), "ms_mean": round(t["mean_ms"], 4),
               "ms_min": round(t["min_ms"], 4), "timed_steps": t["steps"]}

    peak, peak_kind = measured_peaks()
    value = whole_job_value(info["bytes_per_step"], world, ms_step)

    if info["kind"] == "conv":
        dom_ms = statistics.mean(fwd_ms)
        per_launch_bytes = info["bytes_per_step"]
        dom_name = "fft_convolve (filter spectrum + fused convolution, %d kernels)" % kernels_per_step
    elif info["kind"] == "polymul":
        dom_ms = statistics.mean(fwd_ms)
        per_launch_bytes = info["bytes_per_step"]
        dom_name = "polymul (whole fused pipeline, %d kernels)" % kernels_per_step
    elif info["kind"] == "real":
        dom_ms = statistics.mean(fwd_ms)
        per_launch_bytes = info["bytes_per_step"] / 2
        dom_name = ("r2c_rows_kernel<float,%d>" % log2i(c["n"] // 2)) if info["passes"] == 1 \
            else "forward real plan (%d kernels)" % plans[0].num_kernels
    else:
        dom_ms = statistics.mean(fwd_ms)
        per_launch_bytes = info["bytes_per_step"] / info["directions"]
        dom_name = ("fft_rows_kernel<float,%d,-1>" % log2i(c["n"])) if info["passes"] == 1 and \
            info["kind"] == "fft1d" else "forward plan (%d kernels)" % plans[0].num_kernels
        if info.get("mixed"):
            dom_name = "mixed_rows_kernel<float,-1> (N=%d)" % c["n"]
        if info.get("four_step"):
            dom_name = "forward four-step plan (%d kernels, N=%d)" % (plans[0].num_kernels, c["n"])
    achieved = per_launch_bytes / (dom_ms * 1e-3) / 1e9
    tr = committed_traffic(name)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": tr["traffic_bytes_per_launch"] if tr else None,
                "kernel": dom_name, "peak_source": peak_kind,
                "launch_ms": round(dom_ms, 4),
                "inverse_launch_ms": round(statistics.mean(inv_ms), 4) if inv_ms else None}
    if info["kind"] == "polymul":
        # Bound by the FP64 pipe: flops of the transforms run (5 M log2 M each) per pipeline
        # launch against the GB300's nominal 1.25 TFLOP/s FP64 (an FMA probe measured 1.19).
        fl = info["fp64_flops_per_step"]
        tf = fl / (dom_ms * 1e-3) / 1e12
        roofline.update(bound="alu", achieved=round(tf, 4), peak=1.25, unit="TFLOP/s",
                        frac=round(tf / 1.25, 4), flops_per_launch=fl,
                        peak_source="nominal FP64 (1.25 TFLOP/s); measured FMA probe 1.19",
                        hbm_achieved_gbs=round(achieved, 1))
    if info.get("bluestein_m") and info["passes"] == 1:
        # Two length-M transforms per row of n points: the fused Bluestein kernel is bound by
        # on-chip arithmetic, not HBM.  Peak: 152 SMs x 128 fp32 lanes x 2 flop (FMA) x 2070 MHz.
        alu_peak = 152 * 128 * 2 * 2.070e9 / 1e12
        flops = info["alu_flops_per_row"] * c["batch"]
        alu = flops / (dom_ms * 1e-3) / 1e12
        roofline.update(bound="alu", achieved=round(alu, 2), peak=round(alu_peak, 1),
                        unit="TFLOP/s", frac=round(alu / alu_peak, 4),
                        peak_source="derived (152 SM x 128 fp32 lanes x 2 x 2070 MHz)",
                        kernel="conv_rows_kernel<float,%d,COMPLEX,1> (Bluestein, M=%d)"
                        % (log2i(info["bluestein_m"]), info["bluestein_m"]),
                        hbm_achieved_gbs=round(achieved, 1),
                        flops_per_launch=flops)

    line = {
        "metric": metric_name(info["kind"]),
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64" if info["kind"] == "polymul" else "f32",
        "data": "synthetic (seeded)",
        "config": {"workload": workload_label(name), "l2": "inputs larger than L2, no flush",
                   "hbm_passes": info["passes"], "parallelism": f"replicas x{world}"},
        "hbm_frac": round(value / world / peak, 4),
        "ideal_1pass_frac": round(info["ideal_bytes_per_step"] / (ms_step * 1e-3) / 1e9 / peak, 4),
        "gflops": round(info["flops_per_step"] * world / (ms_step * 1e-3) / 1e9, 1),
        "transforms_per_s": round(info["transforms_per_step"] * world / (ms_step * 1e-3), 1),
        "gpu_launches": kernels_per_step * args.steps,
        "roofline": roofline,
        "e2e": e2e,
        "clocks": clk,
        "clock_soak_s": args.clock_soak,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(name)
    if rank == 0:
        print(json.dumps(line), flush=True)
    for p in plans:
        p.close()
    if world > 1:
        dist.destroy_process_group()


def sized_input(name: str, c: dict):
    if not SIZE_OVERRIDE:
        return workloads.config_input(name)
    if c["kind"] == "fftnd":
        return workloads.normal_complex((c["batch"],) + tuple(c["shape"]), c["seed"])
    if c["kind"] == "real":
        return workloads.normal_real((c["batch"], c["n"]), c["seed"])
    if c["kind"] == "fft2d":
        return workloads.normal_complex((c["batch"], c["n"], c["n"]), c["seed"])
    if name == "c3":
        return workloads.tones_plus_noise(c["n"], c["seed"]).reshape(1, -1)
    return workloads.normal_complex((c["batch"], c["n"]), c["seed"])


def metric_name(kind: str) -> str:
    if kind == "conv":
        return "batched FFT convolution effective GB/s"
    if kind == "real":
        return "batched real FFT (R2C + C2R) effective GB/s"
    return "batched C2C FFT effective GB/s"


def workload_label(name: str) -> str:
    if SIZE_OVERRIDE:
        c = config_of(name)
        return f"{name} reduced for profiling: n={c['n']}, batch={c['batch']}"
    c = workloads.CONFIGS[name]
    if name == "c1":
        return "1D C2C forward, N=1024, batch 1, fp32"
    if name == "c2":
        return "1D C2C forward+inverse, N=4096, batch 16384, fp32 (512 MiB)"
    if name == "c3":
        return "1D C2C forward, N=2^26, batch 1, fp32 (512 MiB), multi-pass"
    if name == "c4":
        return "2D C2C forward+inverse, 2048x2048, batch 8, fp32"
    if name == "conv1":
        return ("real fp32 convolution, 32768 signals x 3072 samples with one 1025-tap filter "
                "(transform length 4096)")
    if name == "real1":
        return "1D real R2C+C2R, N=8192, batch 32768, fp32 (1 GiB of samples)"
    if name == "any1":
        return "1D C2C forward+inverse, N=3000 = 2^3 3 5^3 (mixed radix on chip), batch 16384, fp32"
    if name == "any3":
        return ("1D C2C forward+inverse, N=100000 = 2^5 5^5 (four-step: 2 mixed-radix passes, "
                "3 transposes), batch 1024, fp32")
    if name == "any2":
        return "1D C2C forward+inverse, N=3001 prime (Bluestein, M=8192 on chip), batch 16384, fp32"
    if name == "nd1":
        return "3D C2C forward+inverse, 128x256x256, batch 4, fp32 (256 MiB)"
    return f"polymul, {c['batch']} pairs of 2^20 int64 coefficients, fp64 transforms of 2^21"


# ---------------------------------------------------------------------------
# Reference arm: the fp64 CPU oracle as it stands
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    name = args.config
    info = workload_info(name)

    def one_step():
        return cpu_oracle_sample(name, budget_s=args.ref_step_seconds)
    for _ in range(args.warmup):
        one_step()
    vals, secs, last = [], 0.0, None
    for _ in range(args.steps):
        last = one_step()
        vals.append(last["value"])
        secs += last["seconds"]
    value = statistics.mean(vals)
    ms_step = 1e3 * info["bytes_per_step"] / (value * 1e9)
    line = {
        "impl": "reference",
        "metric": metric_name(info["kind"]),
        "value": float(f"{value:.4g}"),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": workload_label(name), "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": float(f"{value:.4g}"), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": last["sample"] + " per step"},
        "e2e": {"value": float(f"{value:.4g}"), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(workloads.CONFIGS), default="c2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=16,
                    help="batch chunks streamed through the device by the end-to-end pipeline")
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    ap.add_argument("--clock-soak", type=float, default=0.6,
                    help="seconds of untimed load sampled for clocks before the timed region")
    ap.add_argument("--n", type=int, default=None,
                    help="override the transform length (small profiling cases)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch (small profiling cases)")
    args = ap.parse_args()
    if args.n is not None:
        SIZE_OVERRIDE["n"] = args.n
    if args.batch is not None:
        SIZE_OVERRIDE["batch"] = args.batch
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
