#!/usr/bin/env python
"""Throughput of the batched power-of-two C2C FFT on one GB300 (or N, one
process per GPU, each with its own full batch: weak scaling).

Default workload (``--config c2``): 16384 transforms of 4096 fp32 complex
points (512 MiB), a step = forward then inverse (1/N).  Inputs are larger
than L2 (129 MB), so no flush between steps is needed.  The default run also
times the other four configurations of the same method -- one 1024-point
transform (c1, latency), one 2^26-point transform (c3, multi-pass), 8 images
of 2048 x 2048 (c4, 2D) and 64 polynomial products of 2^20 coefficients (c5,
fp64) -- each in its own timed region, reported under ``configs``.

Metric: effective GB/s = algorithmic HBM bytes of the step / step time,
where the algorithmic bytes of one transform call are (HBM passes of the
chosen plan) x 2 x (bytes of the complex array); the on-chip path makes one
pass.  Also reported: 5 N log2 N GFLOP/s, transforms/s, the roofline of
the dominant kernel against the measured HBM copy bandwidth, the fp64 CPU
oracle on a bounded sample (one core and all cores), an end-to-end figure
with host buffers, and the SM clocks sampled during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed alone
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import itertools
import json
import math
import os
import platform
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
    on-chip length with factors of at most pass_log bits (its own rule; the
    bench reads the real count from the plan it builds)."""
    return max(2, math.ceil(logn / pass_log))


def workload_info(name: str, pass_log: int = 9, passes=None):
    """Bytes, flops and units of one step.  `passes`: the HBM passes of the
    plan actually built (its kernel count), for the multi-pass 1D kind."""
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
            if log2i(n) <= 14:
                passes = 1
            elif passes is None:
                passes = planned_passes(log2i(n), pass_log)
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
        if n & (n - 1) == 0 and log2i(n) > 14:
            # the least HBM traffic for a transform beyond one block: a
            # 2-pass four-step (every element read and written twice)
            info.update(min_passes=2, min_bytes_per_step=directions * 2 * 2 * arr)
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
    "c4": ["fft_device.cuh", "fft_rows.cuh", "fft_rows_f32.cu", "fft_rows_col.cuh",
           "rows_col_f32.cu", "fft_pass.cuh", "fft_pass_tma.cuh", "fft_pass_cluster.cuh",
           "fft_pass_f32.cu", "fft_plan.cu", "fft_exec.cu", "plan.h"],
    "c5": ["fft_device.cuh", "fft_pass.cuh", "fft_pass_tma.cuh", "fft_pass_cluster.cuh",
           "fft_pass_f64.cu", "polymul.cu"],
    "conv1": ["fft_device.cuh", "fft_rows.cuh", "conv.cuh", "conv_f32.cu"],
    "any1": ["fft_device.cuh", "mixed.cuh", "mixed_f32.cu", "fft_plan.cu", "fft_exec.cu", "plan.h"],
    "any2": ["fft_device.cuh", "fft_rows.cuh", "conv.cuh", "anylen.cuh", "anylen_f32.cu"],
    "any3": ["fft_device.cuh", "mixed.cuh", "mixed_f32.cu", "transpose.cu", "fft_plan.cu", "fft_exec.cu", "plan.h"],
    "real1": ["fft_device.cuh", "fft_rows.cuh", "real.cuh", "real_f32.cu"],
    "nd1": ["fft_device.cuh", "fft_rows.cuh", "fft_rows_t.cuh", "rows_t_f32.cu", "fft_plan.cu", "fft_exec.cu", "plan.h"],
    "rows512": ["fft_device.cuh", "fft_rows.cuh", "fft_warp.cuh", "fft_rows_f32.cu"],
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
    # The counters belong to the workload as captured: none for a resized
    # workload (--n / --batch) or one run with forced library choices.
    if SIZE_OVERRIDE or OPTIONS:
        return None
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

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_units(name: str):
    """(unit, fraction of one step's work per unit, sample description) for
    the oracle's timed sample of a workload: `unit(k)` runs the k-th unit of
    work on the oracle as it stands."""
    import oracle
    info = workload_info(name)
    c = config_of(name)
    if info["kind"] == "fft1d":
        n = c["n"]
        two = info["directions"] == 2
        if n <= 1 << 16:
            x = workloads.config_input(name, scale_batch=min(c["batch"], 64)).astype(np.complex128)
            pow2 = n & (n - 1) == 0

            def unit(k):
                y = oracle.fft(x[k % x.shape[0]]) if pow2 else oracle.dft(x[k % x.shape[0]])
                if two:
                    oracle.ifft(y) if pow2 else oracle.dft(y, +1)
            how = "recursive CT" if pow2 else "direct DFT"
            return unit, 1.0 / c["batch"], \
                f"transforms of N={n} ({how}{', forward+inverse' if two else ''}) of {c['batch']}"
        if n & (n - 1):
            # a long length that is not a power of two: the oracle is the direct
            # DFT; units of 64 bins of one row (O(N) each)
            x = workloads.config_input(name, scale_batch=1)[0].astype(np.complex128)

            def unit(k):
                oracle.dft_bins(x, (np.arange(64, dtype=np.int64) + 64 * k) % n)
            return unit, 64.0 / (n * c["batch"] * info["directions"]), \
                f"blocks of 64 direct-DFT bins of one N={n} row, scaled to the step"
        # one long transform: 2^20-point transforms scaled by N log N
        m = 1 << 20
        x = workloads.normal_complex(m, 99, np.complex128)

        def unit(k):
            oracle.fft(x)
        return unit, (m * log2i(m)) / (n * log2i(n)), \
            f"transforms of N=2^20 (recursive CT) scaled by N log2 N to N={n}"
    if info["kind"] == "fft2d":
        n = c["n"]
        img = workloads.normal_complex((1, n, n), 4, np.complex128)[0]

        def unit(k):
            oracle.fft2d(oracle.fft2d(img), +1)
        return unit, 1.0 / c["batch"], f"images {n}x{n} (forward+inverse) of {c['batch']}"
    if info["kind"] == "fftnd":
        vol = workloads.normal_complex((1,) + tuple(c["shape"]), c["seed"], np.complex128)

        def unit(k):
            oracle.fftn(oracle.fftn(vol, len(c["shape"])), len(c["shape"]), +1)
        return unit, 1.0 / c["batch"], f"volumes {c['shape']} (forward+inverse) of {c['batch']}"
    if info["kind"] == "real":
        x = workloads.normal_real((64, c["n"]), c["seed"], np.float64)

        def unit(k):
            oracle.irfft(oracle.rfft(x[k % 64]), c["n"])
        return unit, 1.0 / c["batch"], f"real rows of N={c['n']} (forward+inverse) of {c['batch']}"
    if info["kind"] == "conv":
        x, h = workloads.conv_signals(64, c["n"], c["nh"], c["seed"])
        h = h.astype(np.complex128)

        def unit(k):
            oracle.convolve(x[k % 64].astype(np.complex128), h)
        return unit, 1.0 / c["batch"], \
            f"signals (direct sum, {c['n']} x {c['nh']} taps) of {c['batch']}"
    m = 1 << 16
    a, b = workloads.poly_coeffs(m, 5)
    L, Lm = info["L"], 1 << (2 * m - 1 - 1).bit_length()

    def unit(k):
        oracle.polymul_fft(a, b)
    return unit, (Lm * log2i(Lm)) / (L * log2i(L)) / c["batch"], \
        "fp64 FFT products of 2^16-coefficient pairs, scaled by L log2 L to 2^20"


def cpu_oracle_sample(name: str, budget_s: float = 6.0, threads: int = 1,
                      max_fraction: float = None):
    """Times the fp64 oracle as it stands on a bounded sample of the
    workload (about `budget_s` seconds, and at most `max_fraction` of one
    step's work when given) on `threads` host threads -- units of work run
    concurrently, each a plain call into the oracle's C code, which releases
    the interpreter lock -- and scales to the metric's unit."""
    info = workload_info(name)
    unit, frac, what = _oracle_units(name)
    unit(0)  # first-call set-up (library load) outside the timed sample
    limit = None if max_fraction is None else max(1, int(round(max_fraction / frac)))
    done = [0] * threads
    next_unit = itertools.count()  # shared by the workers (atomic under the GIL)
    t0 = time.perf_counter()
    deadline = t0 + budget_s

    def worker(w):
        while True:
            k = next(next_unit)
            if limit is not None and k >= limit:
                return
            unit(k)
            done[w] += 1
            if time.perf_counter() >= deadline:
                return
    if threads == 1:
        worker(0)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(worker, range(threads)))
    el = time.perf_counter() - t0
    units = sum(done)
    step_fraction = units * frac
    gbs = info["bytes_per_step"] * step_fraction / el / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{units} {what}", "seconds": round(el, 3),
            "step_fraction": step_fraction}


def cpu_baselines(name: str, budget_s: float):
    """The oracle on one core and on every core of the host, with the CPU
    model; the one-core figure is the headline baseline."""
    one = cpu_oracle_sample(name, budget_s, 1)
    n = host_cores()
    if n > 1:
        allc = cpu_oracle_sample(name, budget_s, n)
        one["all_cores"] = {k: allc[k] for k in ("value", "unit", "cores", "sample", "seconds")}
    one["cpu_model"] = cpu_model()
    return one


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


class Workload:
    """Device buffers, plans and one step of a workload, on `stream`."""

    def __init__(self, name, fg, torch, dev, stream):
        self.name = name
        c = self.c = config_of(name)
        info = workload_info(name)
        self.kind = info["kind"]
        self.stream = stream
        sh = self.sh = int(stream.cuda_stream)
        self.plans = []
        self.fg = fg
        self.torch = torch
        # Inputs smaller than L2 (129 MB): a 256 MiB buffer written before
        # every step evicts them, so every timed call starts from HBM.
        self.flush = torch.empty(1 << 26, dtype=torch.float32, device=dev) \
            if info["array_bytes"] <= L2_BYTES else None
        if info["kind"] == "conv":
            self.xc_h, self.hc_h = workloads.conv_signals(c["batch"], c["n"], c["nh"], c["seed"])
            self.xc_d = torch.from_numpy(self.xc_h).to(dev)
            self.hc_d = torch.from_numpy(self.hc_h).to(dev)
            ny = c["n"] + c["nh"] - 1
            self.yc_d = torch.empty(c["batch"], ny, dtype=torch.float32, device=dev)
            self.kernels_per_step = fg.fft_convolve_num_kernels(
                c["n"], c["nh"], c["batch"], 0, fg.FFT_CONV_REAL, fg.FFT_C2C_F32)
        elif info["kind"] == "polymul":
            self.a_h, self.b_h = workloads.poly_coeffs((c["batch"], c["n"]), c["seed"])
            self.a_d, self.b_d = torch.from_numpy(self.a_h).to(dev), torch.from_numpy(self.b_h).to(dev)
            self.c_d = torch.empty(c["batch"], 2 * c["n"] - 1, dtype=torch.int64, device=dev)
            self.kernels_per_step = fg.polymul_num_kernels(c["n"], c["n"])
        elif info["kind"] == "real":
            self.x_h = sized_input(name, c)
            self.x_d = torch.from_numpy(self.x_h).to(dev)
            n, batch = c["n"], c["batch"]
            self.X_d = torch.empty(batch, n // 2 + 1, dtype=torch.complex64, device=dev)
            self.y_d = torch.empty_like(self.x_d)
            self.plans = [fg.Plan(n, batch, 1, fg.FFT_FORWARD, fg.FFT_REAL_F32),
                          fg.Plan(n, batch, 1, fg.FFT_INVERSE, fg.FFT_REAL_F32)]
            self.kernels_per_step = sum(p.num_kernels for p in self.plans)
        else:
            self.x_h = sized_input(name, c)
            self.x_d = torch.from_numpy(self.x_h).to(dev)
            self.y_d = torch.empty_like(self.x_d)
            self.z_d = torch.empty_like(self.x_d)
            dims = 2 if info["kind"] == "fft2d" else 1
            shape = tuple(c["shape"]) if info["kind"] == "fftnd" else None
            self.plans = [fg.Plan(c["n"], c["batch"], dims, fg.FFT_FORWARD, fg.FFT_C2C_F32,
                                  shape=shape)]
            if info["directions"] == 2:
                self.plans.append(fg.Plan(c["n"], c["batch"], dims, fg.FFT_INVERSE,
                                          fg.FFT_C2C_F32, shape=shape))
            self.kernels_per_step = sum(p.num_kernels for p in self.plans)
        self.check_shapes()
        # The HBM passes of the plan actually built (multi-pass 1D: one per kernel).
        passes = None
        if info["kind"] == "fft1d" and c["n"] & (c["n"] - 1) == 0 and log2i(c["n"]) > 14:
            passes = self.plans[0].num_kernels
        self.info = workload_info(name, passes=passes)

    def check_shapes(self):
        """Host-side check, before any launch, that every device buffer holds
        what the plans and calls of this workload read and write."""
        c = self.c
        if self.kind == "conv":
            ok = tuple(self.xc_d.shape) == (c["batch"], c["n"]) and \
                tuple(self.yc_d.shape) == (c["batch"], c["n"] + c["nh"] - 1)
        elif self.kind == "polymul":
            ok = tuple(self.a_d.shape) == (c["batch"], c["n"]) == tuple(self.b_d.shape) and \
                tuple(self.c_d.shape) == (c["batch"], 2 * c["n"] - 1)
        elif self.kind == "real":
            ok = tuple(self.x_d.shape) == (c["batch"], c["n"]) and \
                tuple(self.X_d.shape) == (c["batch"], c["n"] // 2 + 1)
        else:
            per = c["n"] * c["n"] if self.kind == "fft2d" else \
                int(np.prod(c["shape"])) if self.kind == "fftnd" else c["n"]
            ok = self.x_d.numel() == c["batch"] * per and \
                self.y_d.numel() == self.x_d.numel() == self.z_d.numel()
        if not ok:
            raise ValueError(f"{self.name}: input buffers do not match the plan's sizes")

    def call(self, which: int):
        """The step's first (0: the dominant forward call) or second (1:
        the inverse, where the workload has one) library call."""
        fg, sh = self.fg, self.sh
        if which == 0:
            if self.kind == "conv":
                rc = fg.fft_convolve(self.xc_d.data_ptr(), self.c["n"], self.hc_d.data_ptr(),
                                     self.c["nh"], self.yc_d.data_ptr(), self.c["batch"], 0,
                                     fg.FFT_CONV_REAL, fg.FFT_C2C_F32, sh)
            elif self.kind == "polymul":
                rc = fg.polymul_batched(self.a_d.data_ptr(), self.c["n"], self.b_d.data_ptr(),
                                        self.c["n"], self.c_d.data_ptr(), self.c["batch"], sh)
            elif self.kind == "real":
                rc = fg.fft_exec(self.plans[0].handle, self.x_d.data_ptr(), self.X_d.data_ptr(), sh)
            else:
                rc = fg.fft_exec(self.plans[0].handle, self.x_d.data_ptr(), self.y_d.data_ptr(), sh)
        elif self.kind == "real":
            rc = fg.fft_exec(self.plans[1].handle, self.X_d.data_ptr(), self.y_d.data_ptr(), sh)
        else:
            rc = fg.fft_exec(self.plans[1].handle, self.y_d.data_ptr(), self.z_d.data_ptr(), sh)
        assert rc == 0, fg.fft_status_string(rc)

    def has_second(self) -> bool:
        return self.kind == "real" or (self.kind not in ("conv", "polymul") and len(self.plans) == 2)

    def step(self, events=None):
        """One step.  Inputs smaller than L2 are preceded by an L2 flush,
        and then events[0..2] (which such workloads pass) bracket the calls:
        [0]..[1] the first, [1]..[2] the second.  Other workloads are timed
        without events between their calls (an event recorded between two
        launches keeps the second from starting while the first drains)."""
        st = self.stream
        if self.flush is not None:
            with self.torch.cuda.stream(st):
                self.flush.zero_()
        if events is not None:
            events[0].record(st)
        self.call(0)
        if events is not None:
            events[1].record(st)
        if self.has_second():
            self.call(1)
        if events is not None:
            events[2].record(st)

    def e2e_step_fn(self, torch, chunks):
        """One end-to-end step through the host-buffer entry points (pinned
        host input -> device, the transforms, device -> pinned host output),
        and the number of chunks the batch streams through in."""
        fg, sh, c = self.fg, self.sh, self.c
        chunk = max(1, c["batch"] // chunks)
        if self.kind in ("fft1d", "fft2d", "fftnd", "real"):
            h_in = torch.from_numpy(self.x_h).pin_memory()
            h_out = torch.empty_like(h_in).pin_memory()
            dev_b = self.X_d if self.kind == "real" else self.y_d
            plans = self.plans

            def f():
                plans[0].chain_host(plans[1:], h_in, h_out, self.x_d, dev_b, chunk, self.stream)
            return f, chunk
        if self.kind == "conv":
            hx = torch.from_numpy(self.xc_h).pin_memory()
            hy = torch.empty(self.yc_d.shape, dtype=torch.float32).pin_memory()

            def f():
                rc = fg.fft_convolve_host(hx.data_ptr(), c["n"], self.hc_d.data_ptr(), c["nh"],
                                          hy.data_ptr(), c["batch"], 0, fg.FFT_CONV_REAL,
                                          fg.FFT_C2C_F32, self.xc_d.data_ptr(),
                                          self.yc_d.data_ptr(), chunk, sh)
                assert rc == 0, fg.fft_status_string(rc)
            return f, chunk
        ha, hb = torch.from_numpy(self.a_h).pin_memory(), torch.from_numpy(self.b_h).pin_memory()
        hc = torch.empty(self.c_d.shape, dtype=torch.int64).pin_memory()

        def f():
            rc = fg.polymul_batched_host(ha.data_ptr(), c["n"], hb.data_ptr(), c["n"],
                                         hc.data_ptr(), c["batch"], self.a_d.data_ptr(),
                                         self.b_d.data_ptr(), self.c_d.data_ptr(), chunk, sh)
            assert rc == 0, fg.fft_status_string(rc)
        return f, chunk

    def close(self):
        for p in self.plans:
            p.close()


def graph_latency_us(w: Workload, torch, replays: int = 20, per_graph: int = 256) -> float:
    """Device time per transform of `per_graph` back-to-back forward calls
    captured in one CUDA graph (no host enqueue between them), averaged over
    `replays` replays timed with one pair of events."""
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device=w.x_d.device)
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cap):
        sh = int(torch.cuda.current_stream().cuda_stream)
        for _ in range(per_graph):
            rc = w.fg.fft_exec(w.plans[0].handle, w.x_d.data_ptr(), w.y_d.data_ptr(), sh)
            assert rc == 0, w.fg.fft_status_string(rc)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (replays * per_graph)
    del g
    return us


def measure(name, args, fg, torch, dev, world, barrier, with_cpu):
    """Times `args.steps` steps of workload `name` after `args.warmup`
    untimed ones (clocks sampled over an untimed soak that runs straight
    into the timed region) and returns the JSON fields of its line."""
    stream = torch.cuda.Stream(device=dev)
    w = Workload(name, fg, torch, dev, stream)
    info, c = w.info, w.c
    for _ in range(args.warmup):
        w.step()
    torch.cuda.synchronize(dev)

    # Clock sampling: nvidia-smi samples every 100 ms, longer than most timed
    # regions here, so the sampler runs over an untimed soak of the same
    # steps (>= args.clock_soak seconds of load) that leads straight into
    # the timed region; the clocks reported are those of the GPU under this
    # load.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.clock_soak:
        for _ in range(4):
            w.step()
        torch.cuda.synchronize(dev)

    # Timed region: the steps alone between one pair of events (workloads
    # smaller than L2 flush it before each step, outside per-call events).
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        w.step(ev[k] if w.flush is not None else None)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    ms_step = ms_total / args.steps
    if w.flush is not None:
        # The step's own time, without the L2 flush before it.
        ms_step = max_over_ranks(statistics.mean(e[0].elapsed_time(e[2]) for e in ev), world,
                                 dev)
        fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
        inv_ms = [e[1].elapsed_time(e[2]) for e in ev] if w.has_second() else []
    else:
        # Average duration of each call of the step: the same number of
        # back-to-back launches of that call alone, between one pair of
        # events on the launching stream.
        def timed_calls(which):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                w.call(which)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            return [e0.elapsed_time(e1) / args.steps]
        fwd_ms = timed_calls(0)
        inv_ms = timed_calls(1) if w.has_second() else []

    # End-to-end through the host-buffer entry points, every step.
    e2e = None
    if not args.no_e2e:
        f, chunk = w.e2e_step_fn(torch, args.e2e_chunks)
        nsteps = 5 if info["kind"] == "polymul" else max(5, min(args.steps, 10))
        t = time_host_steps(f, stream, nsteps)
        e2e_ms = t["median_ms"]
        e2e = {"value": round(info["bytes_per_step"] * world / (e2e_ms * 1e-3) / 1e9, 2),
               "unit": "GB/s", "h2d_bytes_per_step": info["h2d"],
               "d2h_bytes_per_step": info["d2h"], "ms_per_step": round(e2e_ms, 4),
               "ms_mean": round(t["mean_ms"], 4), "ms_min": round(t["min_ms"], 4),
               "timed_steps": t["steps"], "chunk": chunk}

    peak, peak_kind = measured_peaks()
    value = whole_job_value(info["bytes_per_step"], world, ms_step)
    dom_ms = statistics.mean(fwd_ms)
    kps = w.kernels_per_step
    if info["kind"] == "conv":
        per_launch_bytes = info["bytes_per_step"]
        dom_name = "fft_convolve (filter spectrum + fused convolution, %d kernels)" % kps
    elif info["kind"] == "polymul":
        per_launch_bytes = info["bytes_per_step"]
        dom_name = "polymul (whole fused pipeline, %d kernels)" % kps
    elif info["kind"] == "real":
        per_launch_bytes = info["bytes_per_step"] / 2
        dom_name = ("r2c_rows_kernel<float,%d>" % log2i(c["n"] // 2)) if info["passes"] == 1 \
            else "forward real plan (%d kernels)" % w.plans[0].num_kernels
    else:
        per_launch_bytes = info["bytes_per_step"] / info["directions"]
        dom_name = ("fft_rows_kernel<float,%d,-1>" % log2i(c["n"])) if info["passes"] == 1 and \
            info["kind"] == "fft1d" else "forward plan (%d kernels)" % w.plans[0].num_kernels
        if info.get("mixed"):
            dom_name = "mixed_rows_kernel<float,-1> (N=%d)" % c["n"]
        if info.get("four_step"):
            dom_name = "forward four-step plan (%d kernels, N=%d)" % (w.plans[0].num_kernels,
                                                                      c["n"])
    achieved = per_launch_bytes / (dom_ms * 1e-3) / 1e9
    tr = committed_traffic(name)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": tr["traffic_bytes_per_launch"] if tr else None,
                "kernel": dom_name, "peak_source": peak_kind,
                "bytes_per_launch": per_launch_bytes,
                "launch_ms": round(dom_ms, 4),
                "inverse_launch_ms": round(statistics.mean(inv_ms), 4) if inv_ms else None}
    if info.get("min_bytes_per_step"):
        # Against the 2-pass four-step minimum for this length, next to the
        # chosen plan's own pass count.
        mb = info["min_bytes_per_step"] / info["directions"]
        roofline.update(min_passes=info["min_passes"], min_bytes_per_launch=mb,
                        frac_vs_min_passes=round(mb / (dom_ms * 1e-3) / 1e9 / peak, 4))
    if info["kind"] == "polymul":
        # Bound by the FP64 pipe.  Two flop counts per pipeline launch: the
        # transforms the pipeline runs (one of length L for a + ib, one of
        # length L/2 for the real product: 5 M log2 M each) and the method's
        # count (three length-L transforms), against the GB300's nominal
        # 1.25 TFLOP/s FP64 (an FMA probe on this part measured 1.19).
        fl = info["fp64_flops_per_step"]
        tf = fl / (dom_ms * 1e-3) / 1e12
        mfl = info["flops_per_step"]
        mtf = mfl / (dom_ms * 1e-3) / 1e12
        roofline.update(bound="alu", achieved=round(tf, 4), peak=1.25, unit="TFLOP/s",
                        frac=round(tf / 1.25, 4), flops_per_launch=fl,
                        method_flops_per_launch=mfl, method_achieved=round(mtf, 4),
                        method_frac=round(mtf / 1.25, 4),
                        peak_source="nominal FP64 (1.25 TFLOP/s); FMA probe measured 1.19",
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
    fields = {
        "metric": metric_name(info["kind"]),
        "value": round(value, 2),
        "unit": "GB/s",
        "ms_per_step": round(ms_step, 4),
        "steps": args.steps,
        "warmup": args.warmup,
        "dtype": "f64" if info["kind"] == "polymul" else "f32",
        "config": config_dict(name, info, world),
        "hbm_frac": round(value / world / peak, 4),
        "ideal_1pass_frac": round(info["ideal_bytes_per_step"] / (ms_step * 1e-3) / 1e9 / peak, 4),
        "gflops": round(info["flops_per_step"] * world / (ms_step * 1e-3) / 1e9, 1),
        "transforms_per_s": round(info["transforms_per_step"] * world / (ms_step * 1e-3), 1),
        "gpu_launches": kps * args.steps,
        "roofline": roofline,
        "e2e": e2e,
        "clocks": clk,
    }
    if name == "c1" and not SIZE_OVERRIDE:
        # Latency of one 1024-point transform: the step time above brackets
        # the host's enqueue of each call (ctypes + launch); the device time
        # per transform comes from back-to-back calls replayed from a graph.
        dev_us = graph_latency_us(w, torch)
        fields["latency"] = {"cold_l2_call_us": round(ms_step * 1e3, 3),
                             "cold_l2_call_how": "events around each call (host enqueue "
                                                 "included), L2 flushed before it",
                             "device_us_per_transform": round(dev_us, 3),
                             "device_how": "256 back-to-back forward calls captured in one CUDA "
                                           "graph, 20 replays between one pair of events (warm "
                                           "L2)"}
    if with_cpu:
        fields["cpu_baseline"] = cpu_baselines(name, args.cpu_seconds)
    w.close()
    return fields


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import fft_convolution_gb300 as fg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    for item in args.option:
        name, _, value = item.partition("=")
        name = name.strip().upper()
        code = getattr(fg, "FFT_OPT_" + name)
        # PASS_SPLIT takes the per-pass factors, first pass first: 13,13
        v = fg.pass_split_value(int(f) for f in value.split(",")) \
            if name == "PASS_SPLIT" and "," in value else int(value)
        rc = fg.fft_debug_set_option(code, v)
        assert rc == 0, f"option {item}: {fg.fft_status_string(rc)}"

    def barrier():
        if world > 1:
            dist.barrier()

    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    head = measure(args.config, args, fg, torch, dev, world, barrier, with_cpu)
    line = {
        "metric": head["metric"],
        "value": head["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": head["dtype"],
        "data": "synthetic (seeded)",
    }
    line.update({k: v for k, v in head.items() if k not in line})
    line["clock_soak_s"] = args.clock_soak
    extras = [] if args.no_extra_configs or args.config != "c2" or SIZE_OVERRIDE else \
        [c for c in EXTRA_CONFIGS if c != args.config]
    if extras:
        line["configs"] = {}
        for nm in extras:
            line["configs"][nm] = measure(nm, args, fg, torch, dev, world, barrier, with_cpu)
        # Launches of every timed region of this run (headline and configs).
        line["gpu_launches_all_configs"] = line["gpu_launches"] + sum(
            e["gpu_launches"] for e in line["configs"].values())
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# The other configurations of the method, timed by the default run beside
# the c2 headline.
EXTRA_CONFIGS = ("c1", "c3", "c4", "c5")


L2_BYTES = 129e6


OPTIONS = []  # --option NAME=VALUE items of this run


def config_dict(name: str, info: dict, world: int) -> dict:
    d = {"workload": workload_label(name), "l2": "inputs larger than L2, no flush"
         if info["array_bytes"] > L2_BYTES else "L2 flushed (256 MiB written) before every "
         "timed step", "hbm_passes": info["passes"], "parallelism": f"replicas x{world}"}
    if OPTIONS:
        d["library_options"] = list(OPTIONS)
    return d


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
        # one tones-plus-noise row per transform of the (possibly reduced) batch
        return np.stack([workloads.tones_plus_noise(c["n"], c["seed"] + r)
                         for r in range(c["batch"])])
    return workloads.normal_complex((c["batch"], c["n"]), c["seed"])


def metric_name(kind: str) -> str:
    if kind == "conv":
        return "batched FFT convolution effective GB/s"
    if kind == "real":
        return "batched real FFT (R2C + C2R) effective GB/s"
    if kind == "polymul":
        return "batched FFT polynomial multiplication effective GB/s (int64 in and out)"
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
    if name == "rows512":
        return "1D C2C forward+inverse, N=512, batch 131072, fp32 (512 MiB)"
    return f"polymul, {c['batch']} pairs of 2^20 int64 coefficients, fp64 transforms of 2^21"


# ---------------------------------------------------------------------------
# Reference arm: the fp64 CPU oracle as it stands
# ---------------------------------------------------------------------------

def run_reference(args):
    """The fp64 CPU oracle as it stands, on every host core: each step runs
    the workload's work, or a bounded sample of it (about --ref-step-seconds)
    when the whole step would take longer; the line reports the rate over
    the work done, the fraction of a full step each timed step covered, and
    the wall time actually spent."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    name = args.config
    info = workload_info(name)
    cores = host_cores()

    def one_step():
        return cpu_oracle_sample(name, budget_s=args.ref_step_seconds, threads=cores,
                                 max_fraction=1.0)
    t_all = time.perf_counter()
    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    done, secs, last = 0.0, 0.0, None
    for _ in range(args.steps):
        last = one_step()
        done += last["step_fraction"]
        secs += last["seconds"]
    wall = time.perf_counter() - t0
    value = info["bytes_per_step"] * done / secs / 1e9
    ms_step = 1e3 * secs / args.steps
    line = {
        "impl": "reference",
        "metric": metric_name(info["kind"]),
        "value": float(f"{value:.4g}"),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        # Wall time of one timed step; its work is `sample_fraction` of a
        # full step (1 when the whole step ran), the full-step time
        # extrapolated only when it is less.
        "ms_per_step": round(ms_step, 2),
        "sample_fraction": float(f"{done / args.steps:.4g}"),
        "extrapolated": ({"ms_per_full_step": round(ms_step * args.steps / done, 2)}
                         if 0 < done < args.steps * 0.9999 else None),
        "wall_s": {"timed": round(wall, 2), "total": round(time.perf_counter() - t_all, 2)},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": config_dict(name, info, world),
        "cpu_baseline": {"value": float(f"{value:.4g}"), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "cpu_model": cpu_model(),
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
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="time only --config (the default c2 run also times c1, c3, c4, c5)")
    ap.add_argument("--cpu-seconds", type=float, default=5.0,
                    help="seconds of oracle work per CPU-baseline sample (one core, all cores)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=16,
                    help="batch chunks streamed through the device by the end-to-end pipeline")
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    ap.add_argument("--clock-soak", type=float, default=0.6,
                    help="seconds of untimed load sampled for clocks before the timed region")
    ap.add_argument("--option", action="append", default=[], metavar="NAME=VALUE",
                    help="force a library choice through its test hook before planning, e.g. "
                         "ROWS_SHFL=1, COL_RADIX_LOG=0 or PASS_SPLIT=13,13 (kernel comparisons; "
                         "recorded in config)")
    ap.add_argument("--n", type=int, default=None,
                    help="override the transform length (small profiling cases)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch (small profiling cases)")
    args = ap.parse_args()
    OPTIONS.extend(args.option)
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
