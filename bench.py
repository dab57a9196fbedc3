#!/usr/bin/env python3
"""Benchmark of the shard-reduction GEMM on GB300; prints ONE JSON line.

A step is one call of the fused projection on one batch of synthetic input.
The headline workload is the AG mode of the KDA-like projection at its largest
global M: R = 8 activation shards of 4096 rows, K = 7168, N = 6288 (AG-GEMM
page, microbenchmark table, last KDA row). Inputs (561 MB per step) are larger
than the 126 MB L2 and resident in HBM before the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-sweep] [--no-e2e] [--no-cpu-baseline]

--impl reference times the CPU oracle (the only baseline this path has) on the
box's host cores, each step a bounded sample of the same workload. Under
torchrun (N > 1) every rank runs an independent replica of the workload on its
own GPU (no collective on the data path); the JSON value is the work of all
ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BF16 TFLOP/s per mode vs M on 1 GB300; % of dense BF16 peak; oracle time"
ROW_PAUSE_S = 0.3   # idle pause before each per-workload row (see sweep)
L2_BYTES = 126 * 1024 * 1024
DECODE_LAYERS = 4   # o_proj weight sets of the decode-step rows: 4 x 103 MB, more than L2
# GB300 datasheet figures (dense bf16 tensor throughput, HBM3e bandwidth). The
# roofline's `peak` is the measured one (a cuBLAS GEMM and a device copy on
# this machine); these give the second fraction, against the nominal part.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_burst": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def kernel_source_hash() -> str:
    """Hash of the sources the main kernel (the headline workload's) is built from."""
    h = hashlib.sha256()
    for f in ("gsr_kernel.cu", "gsr_device.cuh", "gsr_params.h"):
        with open(os.path.join(ROOT, "tensor_gemm_reduction_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class NvmlField(ctypes.Structure):
    """nvmlFieldValue_t: one field query and its 8-byte value."""
    _fields_ = [("fieldId", ctypes.c_uint), ("scopeId", ctypes.c_uint),
                ("timestamp", ctypes.c_longlong), ("latencyUsec", ctypes.c_longlong),
                ("valueType", ctypes.c_int), ("nvmlReturn", ctypes.c_int),
                ("value", ctypes.c_ulonglong)]


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read in-process through NVML
    (read-only queries; no setting is touched) every ~1 ms on a background
    thread, so that a timed region of a few tens of milliseconds still holds
    tens of samples. Only samples taken between mark_start() and mark_end()
    enter the summary. NVML is loaded with ctypes from the driver's own
    library; where it is missing, start() returns False."""
    SM = 1                      # NVML_CLOCK_SM
    POWER_INSTANT = 186         # NVML_FI_DEV_POWER_INSTANT
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, cuda_index: int, interval_s: float = 0.001):
        self.cuda_index = cuda_index
        self.interval = interval_s
        self.samples = []          # (t, sm_mhz, power_w, reasons_mask)
        self.t0 = self.t1 = None
        self._stop = False
        self._thread = None
        self.nvml = None
        self.handle = None
        self.max_mhz = None

    def _open(self) -> bool:
        import torch
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if nv.nvmlInit_v2() != 0:
            return False
        self.nvml = nv
        h = ctypes.c_void_p()
        pr = torch.cuda.get_device_properties(self.cuda_index)
        bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0 and \
                nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.cuda_index), ctypes.byref(h)) != 0:
            return False
        self.handle = h
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, self.SM, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        return True

    def _read(self):
        nv, h = self.nvml, self.handle
        mhz, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        f = NvmlField(fieldId=self.POWER_INSTANT)
        sm = float(mhz.value) if nv.nvmlDeviceGetClockInfo(h, self.SM, ctypes.byref(mhz)) == 0 else None
        if nv.nvmlDeviceGetFieldValues(h, 1, ctypes.byref(f)) == 0 and f.nvmlReturn == 0:
            watts = f.value / 1000.0
        elif nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0:
            watts = mw.value / 1000.0
        else:
            watts = None
        mask = int(rs.value) if self._reasons(h, ctypes.byref(rs)) == 0 else 0
        return sm, watts, mask

    def _loop(self):
        while not self._stop:
            t = time.perf_counter()
            self.samples.append((t,) + self._read())
            time.sleep(self.interval)

    def start(self) -> bool:
        import threading
        if not self._open():
            return False
        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()
        time.sleep(0.02)
        return True

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self._thread is not None:
            time.sleep(0.005)
            self._stop = True
            self._thread.join(timeout=5)
        if self.nvml is not None:
            self.nvml.nvmlShutdown()

    def summary(self):
        inside = [x for x in self.samples if self.t0 is not None and self.t0 <= x[0] <= self.t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"],
                    "source": "nvml"}
        sm = [x[1] for x in inside if x[1] is not None]
        pw = [x[2] for x in inside if x[2] is not None]
        reasons = sorted({name for x in inside for bit, name in self.REASONS.items() if x[3] & bit})
        span = (self.t1 - self.t0) * 1e3
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_mhz_min": min(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "power_w_median": statistics.median(pw) if pw else None,
                "power_w_max": max(pw) if pw else None, "samples": len(inside),
                "region_ms_host": span, "reasons": reasons,
                "source": "nvml, in-process, ~%g ms apart, samples inside the timed region only"
                          % (self.interval * 1e3)}


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"gsr_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        maxp = max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= 0.5 * maxp] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": maxp, "samples": len(loaded), "reasons": reasons}


def init_replicas():
    """World size, rank and local rank from the launcher's environment; with
    more than one rank, a gloo process group for the barriers and the max over
    ranks (nothing on the data path)."""
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="gloo")
    return world, rank, local


def replica_region(step, steps: int, warmup: int, world: int, sync, time_fn):
    """One rank's timed region: `warmup` untimed steps, a synchronise and a
    barrier, `steps` steps timed by time_fn(step, steps) -> (per-step ms,
    region ms), then a barrier, so every rank's region spans the same moment."""
    for _ in range(warmup):
        step()
    sync()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    times, region_ms = time_fn(step, steps)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    return times, region_ms


def finish_replicas(world: int) -> None:
    """Every rank waits for rank 0's output, then the process group ends."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def replica_value(local_seconds: float, flops_per_rank: float, world: int):
    """Whole-job TFLOP/s of `world` independent replicas: all ranks' flops over
    the slowest rank's timed region (max over ranks through the process group)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_seconds], dtype=torch.float64)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    slowest = float(t.item())
    return flops_per_rank * world / slowest / 1e12, slowest


def workload_by_name(name: str):
    from tensor_gemm_reduction_gb300 import inputs as gi
    for w in gi.ALL_WORKLOADS:
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}; choose from {[w.name for w in gi.ALL_WORKLOADS]}")


def describe_workload(w) -> dict:
    sizes = w.shard_sizes()
    d = {"workload": w.name, "mode": w.mode, "R": w.R, "M": w.M, "N": w.N, "K": w.K}
    d["M_r" if w.mode == "ag" else "K_r"] = sizes[0] if len(set(sizes)) == 1 else sizes
    return d


def parse_options(items) -> dict:
    """--option NAME=VALUE pairs -> {GSR_OPT_* constant name: int}. NAME is the
    option's name in gsr.h without the prefix, in any case (split_k, block_n,
    schedule, raster_m, small_m, ...)."""
    from tensor_gemm_reduction_gb300 import binding as B
    out = {}
    for item in items or ():
        name, sep, value = item.partition("=")
        key = "GSR_OPT_" + name.strip().upper()
        if not sep or not hasattr(B, key):
            known = sorted(k[8:].lower() for k in dir(B) if k.startswith("GSR_OPT_"))
            raise SystemExit(f"--option {item!r}: expected NAME=VALUE with NAME one of {known}")
        try:
            out[key] = int(value, 0)
        except ValueError:
            raise SystemExit(f"--option {item!r}: the value must be an integer") from None
    return out


def bench_config(w, world: int, options: dict | None = None) -> dict:
    """The `config` object of the JSON line (the same for both arms; the seed of
    the workload's generator, 2000 + M + K unless the workload fixes another;
    plan options only when some were given)."""
    from tensor_gemm_reduction_gb300 import inputs as gi
    read = w.bytes - 2 * w.M * w.N
    l2 = ("inputs larger than L2: %.0f MB read per step" % (read / 1e6) if read > L2_BYTES else
          "inputs fit in L2 (%.1f MB per step): timed back to back without a flush" % (read / 1e6))
    cfg = dict(describe_workload(w), l2=l2,
               parallelism="replicas" if world > 1 else "single",
               seed=w.seed if w.seed is not None else gi.default_seed(w.M, w.K))
    if options:
        cfg["options"] = {k[len("GSR_OPT_"):].lower(): v for k, v in options.items()}
    return cfg


class Runner:
    """Device-resident inputs and outputs of one workload plus its call."""

    def __init__(self, w, plan, ws, dev):
        import torch
        from tensor_gemm_reduction_gb300 import binding as B
        from tensor_gemm_reduction_gb300 import inputs as gi
        self.w, self.plan, self.ws, self.B = w, plan, ws, B
        inp = gi.make_inputs(w, device=dev)     # seeded on the device: fast at full size
        self.inp = inp
        if w.mode in ("ag", "ar"):
            self.Y = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
        else:
            rps = -(-w.M // w.R)
            self.Y_r = [torch.empty(rps, w.N, dtype=torch.bfloat16, device=dev) for _ in range(w.R)]

    def inputs(self):
        return (self.inp.A_r + [self.inp.W]) if self.w.mode == "ag" else (self.inp.X_r + self.inp.W_r)

    def outputs(self):
        return [self.Y] if self.w.mode != "rs" else self.Y_r

    def _prepare(self):
        B, inp = self.B, self.inp
        if self.w.mode == "ag":
            return B.prepare_ag(self.plan, inp.A_r, inp.W, self.Y, self.ws)
        if self.w.mode == "ar":
            return B.prepare_ar(self.plan, inp.X_r, inp.W_r, self.Y, self.ws)
        return B.prepare_rs(self.plan, inp.X_r, inp.W_r, self.Y_r, self.ws, M=self.w.M)

    def __call__(self):
        # One validated, marshalled call per (plan, workspace); re-prepared when
        # a sweep swaps them.
        key = (id(self.plan), id(self.ws))
        if getattr(self, "_key", None) != key:
            self._call, self._key = self._prepare(), key
        self._call()


def trimmed_mean(xs, cut: float = 0.25):
    """Mean of the middle of the sorted samples (a `cut` fraction dropped at each
    end): robust to the odd slow launch, and unlike the median it averages out
    the clustering of single flushed launches at values about a microsecond apart."""
    s = sorted(xs)
    k = int(len(s) * cut)
    mid = s[k:len(s) - k] or s
    return sum(mid) / len(mid)


def time_launches(fn, steps: int, warmup: int, flush=None, marks=None):
    """Per-launch CUDA-event durations (ms) on the current stream, plus the
    elapsed time of the whole region (ms). `marks` (a clock sampler) is told
    when the region starts and when the synchronise after it returns."""
    import torch
    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if marks is not None:
        marks.mark_start()
    t0.record()
    for s, e in ev:
        if flush is not None:
            flush()
        s.record()
        fn()
        e.record()
    t1.record()
    torch.cuda.synchronize()
    if marks is not None:
        marks.mark_end()
    return [s.elapsed_time(e) for s, e in ev], t0.elapsed_time(t1)


def cpu_oracle_rate(w, host_inp, target_s: float, max_rows: int | None = None):
    """Time the oracle on whole output rows of `w` (TFLOP/s), bounded to about
    target_s seconds of CPU work. Returns (rate, rows, seconds, threads)."""
    import numpy as np
    import oracle
    oracle.build()
    M, N = w.M, w.N
    rng = np.random.default_rng(0)

    def run(rows):
        r = np.repeat(rows, N)
        c = np.tile(np.arange(N), len(rows))
        t = time.perf_counter()
        if w.mode == "ag":
            oracle.ag_at(host_inp.A_r, host_inp.W, r, c)
        else:
            oracle.ar_at(host_inp.X_r, host_inp.W_r, r, c)
        return time.perf_counter() - t

    probe = rng.integers(0, M, 8)
    dt = run(probe)
    n = max(8, int(len(probe) * target_s / max(dt, 1e-3)))
    if max_rows:
        n = min(n, max_rows)
    rows = rng.integers(0, M, n)
    dt = run(rows)
    flops = 2.0 * len(rows) * N * w.K
    return flops / dt / 1e12, len(rows), dt, oracle.threads()


def host_copy(inp, w):
    """CPU copies (bf16) of device inputs for the oracle."""
    if w.mode == "ag":
        from tensor_gemm_reduction_gb300.inputs import AGInputs
        return AGInputs(inp.N, inp.K, inp.M_r, [a.cpu() for a in inp.A_r], inp.W.cpu())
    from tensor_gemm_reduction_gb300.inputs import ARInputs
    return ARInputs(inp.M, inp.N, inp.K_r, [x.cpu() for x in inp.X_r], [x.cpu() for x in inp.W_r])


def run_reference(args, w):
    """The oracle, as it stands, on host cores: each step computes a bounded
    sample (a few whole output rows) of the same workload."""
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from tensor_gemm_reduction_gb300 import inputs as gi
    oracle.build()
    # Inputs from the CPU generator (same recipe; no GPU needed on this arm).
    inp = gi.make_inputs(w, device="cpu")
    rows_per_step = args.ref_rows
    rng = np.random.default_rng(1)
    N = w.N

    def step():
        rows = rng.integers(0, w.M, rows_per_step)
        r = np.repeat(rows, N)
        c = np.tile(np.arange(N), rows_per_step)
        if w.mode == "ag":
            oracle.ag_at(inp.A_r, inp.W, r, c)
        else:
            oracle.ar_at(inp.X_r, inp.W_r, r, c)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    flops = 2.0 * rows_per_step * N * w.K * args.steps
    value = flops / dt / 1e12
    sample = f"{rows_per_step} whole output rows ({rows_per_step * N} outputs) of {w.name} per step"
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, ws_, parse_options(args.option)), "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def sweep(plan, ws, dev, pk, names):
    """Per-workload kernel time with an L2 flush before every launch: the
    trimmed mean of 20 launches. Each row starts after a short idle pause, so
    that a short kernel is not timed while the GPU is still held at the power
    limit by the previous row (after the M = 32768 rows the SM clock stays near
    1.4 GHz for a while, which slowed the next mid-M rows by up to 25 %)."""
    import torch
    from tensor_gemm_reduction_gb300 import inputs as gi
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    rows = []
    for w in gi.ALL_WORKLOADS:
        if names and w.name not in names:
            continue
        try:
            r = Runner(w, plan, ws, dev)
        except torch.OutOfMemoryError:
            continue
        torch.cuda.synchronize()
        time.sleep(ROW_PAUSE_S)
        times, _ = time_launches(r, steps=20, warmup=3, flush=lambda: flush_buf.fill_(1))
        r.B.gemm_shard_check_status(plan, ws)    # raises if an in-kernel wait ran out
        t = trimmed_mean(times) * 1e-3
        t_roof = max(w.flops / (pk["bf16_burst"] * 1e12), w.bytes / (pk["hbm_gbs"] * 1e9))
        d = B_describe(plan, w)
        rows.append({"workload": w.name, "mode": w.mode, "M": w.M, "N": w.N, "K": w.K, "R": w.R,
                     "us": round(t * 1e6, 2), "tflops": round(w.flops / t / 1e12, 1),
                     "hbm_gbs": round(w.bytes / t / 1e9, 1),
                     "roofline_frac": round(t_roof / t, 3),
                     "roofline_frac_nominal": round(
                         max(w.flops / (NOMINAL_BF16_TFLOPS * 1e12),
                             w.bytes / (NOMINAL_HBM_GBS * 1e9)) / t, 3),
                     "bound": "tensor" if w.flops / (pk["bf16_burst"] * 1e12) >= w.bytes / (pk["hbm_gbs"] * 1e9) else "hbm",
                     "split": d["split"], "block_n": d["block_n"],
                     "kernel": "small_m" if d["schedule"] == 3 else "main",
                     "timing": "single launches, L2 flushed before each"})
        del r
        torch.cuda.empty_cache()
    return rows


def decode_layer_workloads(names=()):
    """The workloads of the decode-step rows: the o_proj shapes in the small-M
    kernel's range (M <= 256), all of them, or those named (by workload or by
    row name)."""
    from tensor_gemm_reduction_gb300 import inputs as gi
    return [w for w in gi.ALL_WORKLOADS
            if w.name.startswith("ar_oproj_m") and w.M <= 256
            and (not names or w.name in names or f"{w.name}_layers{DECODE_LAYERS}" in names)]


def sweep_decode_layers(plan, ws, dev, pk, names):
    """Decode-size AR as a decode step runs it: calls back to back, each on the
    next of DECODE_LAYERS o_proj weight sets (a model's successive layers), so
    that W always streams from HBM with no L2 flush (the weight sets together
    are larger than the L2). Time per call: CUDA-event time of a region of
    20 x DECODE_LAYERS calls over their number, the median of five regions.
    Programmatic dependent launch lets each call start while the previous one
    ends, as in a decode step; the flushed rows time single launches instead."""
    import statistics
    import torch
    from tensor_gemm_reduction_gb300 import binding as B
    from tensor_gemm_reduction_gb300 import inputs as gi
    ws_list = decode_layer_workloads(names)
    if not ws_list:
        return []
    w0 = ws_list[0]
    layers = [gi.gaussian_ar(1, w0.N, w0.shard_sizes(), seed=1000 + l, device=dev).W_r
              for l in range(DECODE_LAYERS)]
    rows = []
    for w in ws_list:
        assert (w.N, w.shard_sizes()) == (w0.N, w0.shard_sizes())
        X_r = gi.make_inputs(w, device=dev).X_r
        Y = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
        calls = [B.prepare_ar(plan, X_r, W_r, Y, ws) for W_r in layers]
        n = 20 * DECODE_LAYERS
        torch.cuda.synchronize()
        time.sleep(ROW_PAUSE_S)
        for i in range(2 * DECODE_LAYERS):
            calls[i % DECODE_LAYERS]()
        per_call = []
        for _ in range(5):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for i in range(n):
                calls[i % DECODE_LAYERS]()
            e.record()
            torch.cuda.synchronize()
            per_call.append(s.elapsed_time(e) * 1e-3 / n)
        B.gemm_shard_check_status(plan, ws)     # raises if an in-kernel wait ran out
        t = statistics.median(per_call)
        d = B_describe(plan, w)
        rows.append({"workload": f"{w.name}_layers{DECODE_LAYERS}", "mode": "ar", "M": w.M, "N": w.N,
                     "K": w.K, "R": w.R, "us": round(t * 1e6, 2),
                     "hbm_gbs": round(w.bytes / t / 1e9, 1),
                     "roofline_frac": round(w.bytes / (pk["hbm_gbs"] * 1e9) / t, 3),
                     "roofline_frac_nominal": round(w.bytes / (NOMINAL_HBM_GBS * 1e9) / t, 3),
                     "bound": "hbm", "kernel": "small_m" if d["schedule"] == 3 else "main",
                     "timing": f"back-to-back calls over {DECODE_LAYERS} weight sets "
                               f"({DECODE_LAYERS * 2 * w.N * w.K / 1e6:.0f} MB, more than L2), no flush"})
        del X_r, Y, calls
    del layers
    torch.cuda.empty_cache()
    return rows


def sweep_floor(dev):
    """The event-to-event time of a one-element kernel after the same L2 flush
    as the sweep's rows: the floor under every row's time (launch and
    completion of a kernel that follows a flush). A row's roofline time plus
    this floor bounds what any kernel can score in this sweep."""
    import torch
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    x = torch.zeros(1, device=dev)
    torch.cuda.synchronize()
    time.sleep(ROW_PAUSE_S)
    times, _ = time_launches(lambda: x.add_(1), steps=20, warmup=3, flush=lambda: flush_buf.fill_(1))
    del flush_buf
    torch.cuda.empty_cache()
    return {"workload": "launch_floor", "us": round(trimmed_mean(times) * 1e3, 2),
            "kernel": "torch one-element add (not this library's)",
            "note": "event to event after the same L2 flush as every row"}


def sweep_pack(plan, ws, dev, pk):
    """The packed gather of per-shard states (HBM-bound copy), timed like the
    GEMM rows: trimmed mean of 20 launches, an L2 flush before each."""
    import torch
    from tensor_gemm_reduction_gb300 import binding as B
    from tensor_gemm_reduction_gb300 import inputs as gi
    w = gi.PACK_SP
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    S = gi.gaussian_states([w.M_r] * w.R, w.T, w.H, seed=w.seed, device=dev)
    P = torch.empty(w.rows_out, w.T * w.H, dtype=torch.bfloat16, device=dev)
    call = B.prepare_pack_gather(plan, S, w.rows_out, P, ws)
    torch.cuda.synchronize()
    time.sleep(ROW_PAUSE_S)
    times, _ = time_launches(call, steps=20, warmup=3, flush=lambda: flush_buf.fill_(1))
    B.gemm_shard_check_status(plan, ws)
    t = trimmed_mean(times) * 1e-3
    row = {"workload": w.name, "mode": "pack", "R": w.R, "M_r": w.M_r, "T": w.T, "H": w.H,
           "rows_out": w.rows_out, "us": round(t * 1e6, 2), "hbm_gbs": round(w.bytes / t / 1e9, 1),
           "roofline_frac": round(w.bytes / (pk["hbm_gbs"] * 1e9) / t, 3),
           "roofline_frac_nominal": round(w.bytes / (NOMINAL_HBM_GBS * 1e9) / t, 3), "bound": "hbm",
           "kernel": "pack"}
    del S, P, flush_buf
    torch.cuda.empty_cache()
    return row


def run_context_mm(args, w):
    """torch.mm (a library GEMM, cuBLAS) on contiguous operands of the same
    shapes: the fused path's context row, not its target. One JSON line per
    workload (--sweep-only names, else --workload), timed like the sweep: a
    median of --steps launches, each after an L2 flush."""
    import torch
    dev = torch.device("cuda:0")
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    names = [s for s in args.sweep_only.split(",") if s] or [w.name]
    for name in names:
        wl = workload_by_name(name)
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        A = torch.randn(wl.M, wl.K, generator=g, device=dev).to(torch.bfloat16)
        W = (torch.randn(wl.N, wl.K, generator=g, device=dev) / math.sqrt(wl.K)).to(torch.bfloat16)
        Y = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device=dev)
        fn = lambda: torch.mm(A, W.t(), out=Y)
        times, _ = time_launches(fn, steps=args.steps, warmup=args.warmup,
                                 flush=lambda: flush_buf.fill_(1))
        if args.profile_window:
            torch.cuda.synchronize()
            torch.cuda.cudart().cudaProfilerStart()
            fn()
            torch.cuda.synchronize()
            torch.cuda.cudart().cudaProfilerStop()
        t = statistics.median(times) * 1e-3
        print(json.dumps({"context": "torch_mm", "workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K,
                          "us": round(t * 1e6, 2), "tflops": round(wl.flops / t / 1e12, 1),
                          "steps": args.steps, "l2": "flushed before every launch"}), flush=True)
        del A, W, Y
        torch.cuda.empty_cache()


def B_describe(plan, w):
    from tensor_gemm_reduction_gb300 import binding as B
    mode = {"ar": B.MODE_AR, "rs": B.MODE_RS, "ag": B.MODE_AG}[w.mode]
    return B.gemm_shard_describe(plan, mode, w.M, w.N, w.K, w.shard_sizes())


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="ag_kda_m32768")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep-only", default="", help="comma-separated workload names")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--ref-rows", type=int, default=4, help="output rows per reference step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--context", choices=("torch_mm",), default=None,
                    help="time torch.mm (cuBLAS) on the concatenated operands instead (context only)")
    ap.add_argument("--option", action="append", default=[], metavar="NAME=VALUE",
                    help="plan option of gsr.h without its GSR_OPT_ prefix (repeatable), e.g. "
                         "schedule=5 or block_n=192; recorded in config.options")
    ap.add_argument("--profile-window", action="store_true",
                    help="with --context: bracket one warm launch with cudaProfilerStart/Stop")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = workload_by_name(args.workload)
    options = parse_options(args.option)

    if args.context is not None:
        run_context_mm(args, w)
        return

    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    from tensor_gemm_reduction_gb300 import binding as B
    from tensor_gemm_reduction_gb300 import build as gbuild

    world, rank, local = init_replicas()
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    gbuild.build()
    pk = peaks()

    plan = B.gemm_shard_plan_create(local, 34816, 8192, 8192, 16)
    for key, value in options.items():
        B.gemm_shard_plan_set_option(plan, getattr(B, key), value)
    ws = B.gemm_shard_workspace_alloc(plan)
    B.gemm_shard_workspace_init(plan, ws)
    run = Runner(w, plan, ws, dev)

    # ---- timed region: K back-to-back steps, inputs resident in HBM
    nvml = NvmlClockSampler(local)
    if nvml.start():
        times, region_ms = replica_region(
            run, args.steps, args.warmup, world, torch.cuda.synchronize,
            lambda step, n: time_launches(step, steps=n, warmup=0, marks=nvml))
        nvml.stop()
        clocks = nvml.summary()
    else:
        with ClockSampler(local) as clk:
            times, region_ms = replica_region(
                run, args.steps, args.warmup, world, torch.cuda.synchronize,
                lambda step, n: time_launches(step, steps=n, warmup=0))
        clocks = clk.summary()
    B.gemm_shard_check_status(plan, ws)
    value, region_s = replica_value(region_ms * 1e-3, w.flops * args.steps, world)
    avg_launch_s = statistics.mean(times) * 1e-3
    achieved = w.flops / avg_launch_s / 1e12
    # The sustained peak is a seconds-long back-to-back loop held at the power
    # limit; it is the matching denominator whenever this loop ran into the
    # same limit (or lasted as long), the burst peak otherwise.
    capped = "sw_power_cap" in clocks.get("reasons", [])
    sustained = capped or region_s > 2.0
    peak = pk["bf16_sustained"] if sustained else pk["bf16_burst"]

    result = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": region_s / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(w, world, options),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(w.name),
                     "peak_kind": ("sustained" if sustained else "burst") + " bf16, " + pk["source"] +
                                  (" (the loop ran at the power limit: sw_power_cap)" if capped else ""),
                     "frac_of_burst": achieved / pk["bf16_burst"],
                     "nominal_peak": NOMINAL_BF16_TFLOPS,
                     "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                     "peak_note": "peak and frac: of measured (cuBLAS bf16 GEMM on this pool's "
                                  "GB300s); frac_of_nominal: of the datasheet dense bf16 peak",
                     "algorithmic_flops_per_launch": w.flops, "avg_launch_us": avg_launch_s * 1e6},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "pages_context": {"gemm_only_us_gb300": 1576.83, "ag_gemm_tp8_us_gb300": 1747.81,
                          "note": "AG-GEMM page, KDA M=32768 row; other hardware setup, not a target"},
    }

    if rank == 0 and not args.no_e2e:
        result["e2e"] = e2e(run, w, args.e2e_steps, world)
    if rank == 0 and not args.no_cpu_baseline:
        host_inp = host_copy(run.inp, w)
        rate, nrows, secs, thr = cpu_oracle_rate(w, host_inp, args.cpu_seconds)
        result["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                  "sample": f"{nrows} whole output rows ({nrows * w.N} outputs) of "
                                            f"{w.name}, {secs:.1f} s"}
    if rank == 0 and not args.no_sweep:
        del run
        torch.cuda.empty_cache()
        names = [s for s in args.sweep_only.split(",") if s]
        result["per_config"] = [sweep_floor(dev)] + sweep(plan, ws, dev, pk, names)
        result["per_config"] += sweep_decode_layers(plan, ws, dev, pk, names)
        if not names or "pack_sp_t4" in names:
            result["per_config"].append(sweep_pack(plan, ws, dev, pk))
    if rank == 0:
        print(json.dumps(result), flush=True)
    finish_replicas(world)


def e2e(run, w, steps, world):
    """Same metric through the public calls with host buffers: every step copies
    all inputs from pinned host memory and reads the whole output back.

    AG uses gemm_ag_flagged: W is copied first and the kernel is launched behind
    it; the activation shards follow on a copy stream, each signalled with
    gemm_shard_signal, so their copies overlap the GEMM on the shards already
    in. The next step's copies wait for the previous kernel. Other modes copy,
    call and read back in order on one stream."""
    import torch
    from tensor_gemm_reduction_gb300 import binding as B
    dev_in = run.inputs()
    dev_out = run.outputs()
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    dev = dev_in[0].device

    if w.mode == "ag":
        # Two device buffer sets alternate between steps, and three streams
        # overlap: the copy stream uploads step N+1's W and shards while the
        # GEMM stream runs step N and the readback stream returns step N-1's Y.
        R = w.R
        A_host, W_host = host_in[:R], host_in[R]
        sets = []
        for b in range(2):
            A_b = dev_in[:R] if b == 0 else [torch.empty_like(a) for a in dev_in[:R]]
            W_b = dev_in[R] if b == 0 else torch.empty_like(dev_in[R])
            Y_b = run.Y if b == 0 else torch.empty_like(run.Y)
            sets.append({"A": A_b, "W": W_b, "Y": Y_b,
                         "ready": torch.zeros(R, dtype=torch.int32, device=dev),
                         "kernel_done": None, "d2h_done": None})
        gemm_s = torch.cuda.Stream(device=dev)
        copy_s = torch.cuda.Stream(device=dev)
        d2h_s = torch.cuda.Stream(device=dev)
        state = {"epoch": 0}

        def step():
            state["epoch"] += 1
            ep = state["epoch"]
            bs = sets[ep % 2]
            with torch.cuda.stream(copy_s):
                if bs["kernel_done"] is not None:
                    copy_s.wait_event(bs["kernel_done"])   # the kernel two steps back is done reading
                bs["W"].copy_(W_host, non_blocking=True)
                w_in = torch.cuda.Event()
                w_in.record(copy_s)
            with torch.cuda.stream(gemm_s):
                gemm_s.wait_event(w_in)
                if bs["d2h_done"] is not None:
                    gemm_s.wait_event(bs["d2h_done"])     # its output buffer has been read back
                B.gemm_ag_flagged(run.plan, bs["A"], bs["W"], bs["Y"], bs["ready"], ep, run.ws)
                done = torch.cuda.Event()
                done.record(gemm_s)
                bs["kernel_done"] = done
            with torch.cuda.stream(copy_s):
                for r in range(R):
                    bs["A"][r].copy_(A_host[r], non_blocking=True)
                    B.gemm_shard_signal(run.plan, bs["ready"].data_ptr() + 4 * r, ep, stream=copy_s)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done)
                host_out[0].copy_(bs["Y"], non_blocking=True)
                out = torch.cuda.Event()
                out.record(d2h_s)
                bs["d2h_done"] = out

        for _ in range(4):
            step()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(copy_s)
        gemm_s.wait_event(t0)
        d2h_s.wait_event(t0)
        for _ in range(steps):
            step()
        gemm_s.wait_event(sets[state["epoch"] % 2]["d2h_done"])
        copy_s.wait_stream(gemm_s)
        t1.record(gemm_s)
        torch.cuda.synchronize()
        B.gemm_shard_check_status(run.plan, run.ws, stream=gemm_s)
        how = ("double-buffered: uploads, gemm_ag_flagged (shards signalled with "
               "gemm_shard_signal) and read-backs of successive steps overlap")
    else:
        def step():
            for d, h in zip(dev_in, host_in):
                d.copy_(h, non_blocking=True)
            run()
            for h, d in zip(host_out, dev_out):
                h.copy_(d, non_blocking=True)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            step()
        t1.record()
        torch.cuda.synchronize()
        how = "copy in, call, copy out on one stream"
    s = t0.elapsed_time(t1) * 1e-3
    return {"value": w.flops * steps / s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": s / steps * 1e3,
            "schedule": how}


if __name__ == "__main__":
    main()
