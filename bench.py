#!/usr/bin/env python3
"""Benchmark of the virtual-rank bf16 allreduce on GB300.

One step = one ``ar_allreduce`` call (C ABI) on the workload, with the
variant under test: the pointer tables already on the device, the kernel(s)
of the variant, the device epoch rotation.  Default workload: R = 8 virtual
ranks of a 512x8192 bf16 tensor each, N(0,1) values, fused LL8 packet
write-mode kernel; the one-shot kernels, the 440x5120 case and the R = 8 and
R = 4 64 MiB cases are measured beside it (``extra``).

Timing: W warm-up steps, then exactly K timed steps bracketed by a barrier
and a device synchronise; CUDA events on the launching stream.  Inputs and
outputs rotate over enough buffer sets that the data touched between two
uses of one set exceeds L2 (no L2 flush needed).  SM clocks and clock-event
reasons are read through NVML during the timed region itself (and by
nvidia-smi around it).  Multi-GPU (torchrun): every rank runs an independent
replica on its own GPU (the path has no exchange step between GPUs); the
timed region is the max over ranks.

``--impl reference`` times the oracle (plain single-threaded C) on the host
cores instead, on a bounded sample of the workload per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs/call and HBM GB/s (% of peak), 8-virtual-rank bf16 allreduce, 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------
# algorithmic bytes per call (R ranks of N bf16 elements)

def alg_bytes(variant: str, R: int, N: int) -> int:
    """Bytes a call must move for the variant's data path.

    fan-out / write mode: every input read once, every output written once
    (4RN, the minimum).  pull: each of the R output ranks reads all R
    inputs (2R^2 N) and writes its output (2RN).  two-phase: 4RN plus the
    reduced shards read back from their owners' outputs in stage 2 (2N; the
    stage-1 stores are already outputs).  fused LL8: 4RN plus each of the
    R-1 foreign shards per rank as 4-byte-per-element packets, written once
    and read once (8(R-1)N)."""
    if variant in ("oneshot_fanout", "oneshot_fanout_bulk"):
        return 4 * R * N
    if variant == "oneshot_pull":
        return 2 * R * R * N + 2 * R * N
    if variant == "twophase":
        return 4 * R * N + (2 * N if R > 1 else 0)
    if variant == "fused_ll8":
        return 4 * R * N + 8 * (R - 1) * N
    if variant in ("fused_ll8_staged", "packet_3op"):
        # plus the reduced shards sent back as packets and read by every rank
        return 4 * R * N + 16 * (R - 1) * N
    raise ValueError(variant)


def launches_per_call(variant: str, R: int) -> int:
    if variant == "packet_3op":
        return 3
    return 2 if (variant == "twophase" and R > 1) else 1


# ----------------------------------------------------------------------------
# distributed helpers (replicas only; the collective is used for timing)

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, world_size=world, rank=rank)
    return world, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_us_per_call(t_max_s: float, calls_per_rank: int, world: int) -> float:
    """All ranks' calls divided into the slowest rank's timed region."""
    return t_max_s * 1e6 / (calls_per_rank * world)


# ----------------------------------------------------------------------------
# peaks, profiles, clocks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "fused_ll8": "k_fused_ll8.cu", "fused_ll8_staged": "k_fused_ll8.cu",
    "packet_3op": "k_fused_ll8.cu",
    "oneshot_fanout": "k_oneshot.cu",
    "oneshot_pull": "k_oneshot.cu", "oneshot_fanout_bulk": "k_oneshot_bulk.cu",
    "twophase": "k_twophase.cu",
    "reduce_scatter": "k_rs_ag.cu", "all_gather": "k_rs_ag.cu",
}


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments, trailing blanks and empty
    lines (string and character literals are kept whole)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (l.rstrip() for l in "".join(out).split("\n"))
    return "\n".join(l for l in lines if l)


def kernel_source_digest(kernel: str) -> str:
    """Digest of the code a kernel is compiled from (its file and the shared
    device header), comments left out: a profile stays valid across edits
    of comments only."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "shot_allreduce_ranks_gb300", "csrc")
    for name in ("ar_internal.cuh", KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel
    and workload, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "%s_%s.txt" % (kernel, workload))
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_digest") != kernel_source_digest(kernel):
            return None
        return int(float(fields["dram_bytes_per_launch"]))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 100):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            self.samples.append((ts, parts))

    def wait_ready(self, timeout=8.0):
        t0 = time.time()
        while self.proc and not self.samples and time.time() - t0 < timeout:
            time.sleep(0.05)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        inside = [p for ts, p in self.samples if t0 <= ts <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i] == "Active"})
        power = [num(p[3]) for p in inside if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max(power) if power else None}


class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (NVIDIA's
    libnvidia-ml, plain ctypes) by a background thread every ~0.2 ms, so that
    even a timed region of a millisecond holds samples.  Read-only queries."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str, period_s: float = 0.0002):
        import ctypes
        self.samples = []
        self.max_mhz = None
        self.thread = None
        self._stop = False
        self.period = period_s
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            dev = ctypes.c_void_p()
            lib.nvmlDeviceGetHandleByUUID.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_void_p)]
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev)) != 0:
                return
            lib.nvmlDeviceGetClockInfo.argtypes = [ctypes.c_void_p, ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_uint)]
            lib.nvmlDeviceGetMaxClockInfo.argtypes = lib.nvmlDeviceGetClockInfo.argtypes
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
            if reasons is None:
                reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
            reasons.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_ulonglong)]
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._lib, self._dev, self._reasons, self._ct = lib, dev, reasons, ctypes
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        except (OSError, AttributeError):
            self.thread = None

    def _run(self):
        ct = self._ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop:
            if (self._lib.nvmlDeviceGetClockInfo(self._dev, 1, ct.byref(clk)) == 0 and
                    self._reasons(self._dev, ct.byref(rs)) == 0):
                self.samples.append((time.time(), float(clk.value), int(rs.value)))
            time.sleep(self.period)

    def stop(self):
        self._stop = True
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        inside = [(mhz, r) for ts, mhz, r in self.samples if t0 <= ts <= t1]
        if not inside:
            return None
        names = sorted({n for _, r in inside for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in inside),
                "sm_mhz_min": min(m for m, _ in inside), "sm_max_mhz": self.max_mhz,
                "reasons": names, "samples": len(inside), "source": "nvml, inside the timed region"}


def host_cpu():
    """(logical cores, CPU model) of the host running this process."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    return os.cpu_count(), model or "unknown"


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[device_index]
        return str(device_index)


# ----------------------------------------------------------------------------
# our arm

def make_sets(R, N, fill, nsets, device, seed0=0):
    import torch
    from shot_allreduce_ranks_gb300 import inputs
    sets = []
    for k in range(nsets):
        xs = inputs.make_inputs(R, N, seed0 + k, fill)
        xin = [x.to(device) for x in xs]
        xout = [torch.empty_like(x) for x in xin]
        sets.append((xs if k == 0 else None, xin, xout))
    return sets


def time_variant(ar, sets, N, variant, steps, warmup, stream, mode="graph", per_graph=50):
    """Time exactly `steps` calls with CUDA events on `stream`.

    mode "graph": the calls are captured into CUDA graphs of `per_graph`
    calls (plus one graph for the remainder) and replayed, the regime of the
    aiter write-mode tables ("CudaGraph: on"); per-call time = region / steps.
    mode "stream": plain back-to-back launches with an event between calls.
    Returns (total_s, per-call durations in s, wall t0, wall t1)."""
    import torch
    ar.set_variant(variant)
    tables = [ar.tables(xin, xout) for _, xin, xout in sets]

    def issue(n, first=0):
        for i in range(first, first + n):
            it, ot = tables[i % len(tables)]
            ar.allreduce_tables(it, ot, N, stream)

    with torch.cuda.stream(stream):
        issue(warmup)
    torch.cuda.synchronize()
    if mode == "graph":
        g_n = max(1, min(per_graph, steps))
        graphs = []
        for n in ([g_n] if steps >= g_n else []) + ([steps % g_n] if steps % g_n else []):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                issue(n)
            graphs.append((g, n))
        full, rest = steps // g_n, steps % g_n
        with torch.cuda.stream(stream):
            for g, _ in graphs:
                g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        w0 = time.time()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(full):
                graphs[0][0].replay()
            if rest:
                graphs[-1][0].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        w1 = time.time()
        barrier()
        total = e0.elapsed_time(e1) * 1e-3
        del graphs
        return total, [total / steps] * steps, w0, w1
    events = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    barrier()
    torch.cuda.synchronize()
    w0 = time.time()
    with torch.cuda.stream(stream):
        events[0].record(stream)
        for i in range(steps):
            it, ot = tables[i % len(tables)]
            ar.allreduce_tables(it, ot, N, stream)
            events[i + 1].record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier()
    per = [events[i].elapsed_time(events[i + 1]) * 1e-3 for i in range(steps)]
    total = events[0].elapsed_time(events[steps]) * 1e-3
    return total, per, w0, w1


def time_flushed(ar, sets, N, variant, steps, stream, flush):
    """Per-call device time with L2 flushed before every call: `flush` (a
    buffer larger than L2) is rewritten on `stream`, then the call runs
    between two events.  Returns the per-call durations in s."""
    import torch
    ar.set_variant(variant)
    tables = [ar.tables(xin, xout) for _, xin, xout in sets]
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(3):
            it, ot = tables[i % len(tables)]
            ar.allreduce_tables(it, ot, N, stream)
        for i, (e0, e1) in enumerate(evs):
            flush.zero_()
            it, ot = tables[i % len(tables)]
            e0.record(stream)
            ar.allreduce_tables(it, ot, N, stream)
            e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) * 1e-3 for e0, e1 in evs]


def spread(durations_s):
    """Median, min, 90th percentile and max of per-call durations, in us."""
    xs = sorted(d * 1e6 for d in durations_s)
    pick = lambda q: xs[min(len(xs) - 1, int(q * (len(xs) - 1) + 0.5))]
    return {"median": round(pick(0.5), 3), "min": round(xs[0], 3), "p90": round(pick(0.9), 3),
            "max": round(xs[-1], 3), "calls": len(xs)}


def time_e2e(ar, R, N, steps, warmup, stream, host_in, host_out):
    import torch
    ar.reserve_host_staging()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            ar.allreduce_host(host_in, host_out, N, stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            ar.allreduce_host(host_in, host_out, N, stream)
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3


def time_link(host_in, host_out, dev_in, dev_out, steps, stream):
    """The host<->device link on its own: per step, the copy engines move
    every input host->device on `stream` while every output goes
    device->host on a second stream (the bytes of one end-to-end step, both
    directions at once).  Returns seconds for `steps` steps."""
    import torch
    side = torch.cuda.Stream(device=stream.device)

    def step():
        side.wait_stream(stream)
        with torch.cuda.stream(stream):
            for d, h in zip(dev_in, host_in):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(side):
            for d, h in zip(dev_out, host_out):
                h.copy_(d, non_blocking=True)
        stream.wait_stream(side)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3


def oracle_time(xs_bits, seconds: float, lib):
    """Time the oracle (single-threaded C) on full calls over these inputs:
    (seconds per call, calls made, rank 0's output)."""
    import oracle
    calls, t0 = 0, time.perf_counter()
    out = None
    while True:
        out = oracle.allreduce_bf16(xs_bits, lib=lib, outputs=out)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds or calls >= 100000:
            break
    return el / calls, calls, out[0]


def device_sets(R, N, nsets, device, seed=0):
    """Buffer sets with N(0,1) bf16 inputs drawn on the device (fast for the
    large extra workloads, whose outputs are not compared here; the GPU tests
    check every workload against the oracle at full size)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = []
    for _ in range(nsets):
        xin = [torch.randn(N, device=device, generator=g).to(torch.bfloat16) for _ in range(R)]
        out.append((None, xin, [torch.empty_like(x) for x in xin]))
    return out


def sets_for(per_set_bytes: int) -> int:
    """Buffer sets so that the data touched between two uses of one set
    exceeds L2 (at least 2)."""
    return min(64, max(2, math.ceil(3 * L2_BYTES / per_set_bytes)))


def time_copy_same_bytes(R, N, steps, stream, device, per_graph=50):
    """Size-matched bandwidth reference: a plain device copy (PyTorch's
    elementwise kernel, not this library's) that reads 2RN bytes and writes
    2RN bytes per call, one buffer of R*N bf16 elements, graph-replayed with
    buffers rotating over more than L2 like the allreduce.  Returns us/call."""
    import torch
    elems = R * N
    nsets = sets_for(4 * elems)
    src = [torch.ones(elems, dtype=torch.bfloat16, device=device) for _ in range(nsets)]
    dst = [torch.empty_like(x) for x in src]
    g_n = max(1, min(per_graph, steps))
    with torch.cuda.stream(stream):
        for i in range(3):
            torch.mul(src[i % nsets], 1, out=dst[i % nsets])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(g_n):
            torch.mul(src[i % nsets], 1, out=dst[i % nsets])
    reps = max(1, steps // g_n)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * g_n)
    del g, src, dst
    torch.cuda.empty_cache()
    return us


def copy_entry(R, N, steps, stream, device, peak, fanout_us=None):
    us = time_copy_same_bytes(R, N, steps, stream, device)
    e = {"us_per_call": round(us, 3),
         "frac_of_measured": round(4 * R * N / us / 1e3 / peak, 4),
         "what": "plain device copy of the same 4RN bytes (torch elementwise kernel), "
                 "graph-replayed, rotating over more than L2"}
    if fanout_us:
        e["fanout_over_copy"] = round(fanout_us / us, 3)
    return e


EXTRA_WORKLOADS = ("r8_440x5120", "r8_512x8192", "r8_64mib", "r4_64mib")
ALL_VARIANTS = ("oneshot_fanout", "oneshot_fanout_bulk", "oneshot_pull", "twophase",
                "fused_ll8", "fused_ll8_staged", "packet_3op")


def run_ours(args):
    import numpy as np
    import torch
    from shot_allreduce_ranks_gb300 import AllReduce, inputs
    from shot_allreduce_ranks_gb300 import build as lib_build

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init("nccl")
    if rank == 0 or not os.path.exists(lib_build.LIB):
        lib_build.build()
    barrier()

    w = inputs.WORKLOADS[args.workload]
    R, N = w.R, w.count
    per_set = 4 * R * N
    nsets = sets_for(per_set)
    sets = make_sets(R, N, w.fill, nsets, dev)
    stream = torch.cuda.Stream(device=dev)
    ar = AllReduce(R, N, device=dev)
    uuid = gpu_id_for(local)
    sampler = ClockSampler(uuid) if not args.no_clocks else None
    if sampler:
        sampler.wait_ready()
    peak, peak_kind = measured_peaks()
    w_load0 = time.time()

    # ---- the other variants on this workload (seconds of the same kind of
    # load right before the timed region)
    extra = {}
    if not args.no_extra:
        for v in ALL_VARIANTS:
            if v == args.variant:
                continue
            n = min(args.steps, 2000)
            t, pv, _, _ = time_variant(ar, sets, N, v, n, 20, stream, args.timing)
            extra[v] = {"us_per_call": round(t * 1e6 / n, 3),
                        "alg_GBps": round(alg_bytes(v, R, N) / statistics.fmean(pv) / 1e9, 1),
                        "frac_min_bytes": round(4 * R * N / statistics.fmean(pv) / 1e9 / peak, 4)}
        other = "stream" if args.timing == "graph" else "graph"
        n = min(args.steps, 2000)
        t, _, _, _ = time_variant(ar, sets, N, args.variant, n, 20, stream, other)
        extra["%s_%s_timing" % (args.variant, other)] = {"us_per_call": round(t * 1e6 / n, 3)}
        # per-call events (an event pair around every launch on the stream):
        # the spread of single calls, warm and with L2 flushed before each
        _, per_stream, _, _ = time_variant(ar, sets, N, args.variant, 200, 20, stream, "stream")
        extra["%s_per_call_stream_us" % args.variant] = spread(per_stream)
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        extra["%s_per_call_l2_flushed_us" % args.variant] = spread(
            time_flushed(ar, sets, N, args.variant, 200, stream, flush))
        del flush
        extra["copy_same_bytes"] = copy_entry(
            R, N, min(args.steps, 2000), stream, dev, peak,
            extra.get("oneshot_fanout", {}).get("us_per_call"))

    # ---- the headline: W warm-up steps, then exactly K timed steps
    nvml = NvmlClocks(uuid) if not args.no_clocks else None
    total, per, w0, w1 = time_variant(ar, sets, N, args.variant, args.steps, args.warmup, stream,
                                      args.timing)
    clocks = nvml.summary(w0, w1) if nvml else None
    if nvml:
        nvml.stop()
    window = sampler.summary(w_load0, w1) if sampler else None
    if clocks is None:
        clocks = window
    elif window:
        clocks["window"] = dict(window, span="nvidia-smi, the %.1f s of calls up to the end of "
                                             "the timed region" % (w1 - w_load0))
    t_max = max_over_ranks(total, dev)
    us_per_call = whole_job_us_per_call(t_max, args.steps, world)
    local_us = total * 1e6 / args.steps
    launch_avg_s = statistics.fmean(per)
    if not args.no_extra:
        extra[args.variant] = {"us_per_call": round(local_us, 3)}

    # ---- the timed variant's own output on input set 0 (checked below)
    xs0, xin0, xout0 = sets[0]
    for o in xout0:
        o.fill_(float("nan"))
    ar.set_variant(args.variant)
    it, ot = ar.tables(xin0, xout0)
    ar.allreduce_tables(it, ot, N, stream)
    torch.cuda.synchronize()
    got = [inputs.bits(o.cpu()) for o in xout0]

    # ---- roofline of the timed kernel
    ab = alg_bytes(args.variant, R, N)
    min_b = 4 * R * N
    achieved = ab / launch_avg_s / 1e9
    traffic = profiled_traffic(args.variant, args.workload)
    roofline = {
        "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
        "frac": round(achieved / peak, 4), "traffic": traffic, "peak_kind": peak_kind,
        "kernel": args.variant, "alg_bytes_per_launch": ab,
        "min_bytes_per_launch": min_b,
        "frac_min_bytes": round(min_b / launch_avg_s / 1e9 / peak, 4),
        "frac_dram": round(traffic / launch_avg_s / 1e9 / peak, 4) if traffic else None,
        "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
        "note": ("achieved/frac count the bytes of the method (4RN plus the LL8 packets, "
                 "each written once and read once; packets stay in L2 and are dropped "
                 "after reading, never written back); frac_min_bytes counts only the "
                 "4RN bytes every allreduce must move to and from HBM; frac_dram uses "
                 "the warm-cache DRAM bytes per launch measured by ncu (traffic)")
        if args.variant in ("fused_ll8", "fused_ll8_staged", "packet_3op") else None}

    # ---- end to end through the host-buffer entry point (pinned host
    # memory), as a user calls it: a handle left on the per-size selector
    # (AR_AUTO), whose host-memory path runs the fan-out on the buffers where
    # they are.
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    host_in = [x.pin_memory() for x in xs0]
    host_out = [torch.empty(N, dtype=torch.bfloat16).pin_memory() for _ in range(R)]
    ar.set_variant("auto")
    t_e2e = time_e2e(ar, R, N, e2e_steps, 3, stream, host_in, host_out)
    t_e2e = max_over_ranks(t_e2e, dev)
    t_link = time_link(host_in, host_out, xin0, xout0, e2e_steps, stream)
    e2e_us = whole_job_us_per_call(t_e2e, e2e_steps, world)
    link_us = t_link * 1e6 / e2e_steps
    e2e = {"value": round(e2e_us, 3), "unit": "us/call",
           "h2d_bytes_per_step": 2 * R * N, "d2h_bytes_per_step": 2 * R * N,
           "steps": e2e_steps,
           "api": "ar_allreduce_host on a default (AR_AUTO) handle: page-locked host buffers "
                  "read and written in place by the oneshot_fanout kernel over NVLink-C2C",
           "link": {"copy_engines_us_per_step": round(link_us, 3),
                    "GBps_each_way": round(2 * R * N / (link_us * 1e-6) / 1e9, 1),
                    "frac": round(link_us / e2e_us, 4),
                    "what": "the same bytes moved by cudaMemcpyAsync alone, host->device and "
                            "device->host concurrently (the link's bound for this step)"}}
    if not args.no_extra:
        ar.set_variant(args.variant)
        t_v = time_e2e(ar, R, N, e2e_steps, 3, stream, host_in, host_out)
        extra["e2e_%s_us_per_call" % args.variant] = round(t_v * 1e6 / e2e_steps, 3)
        pageable_in = [x.clone() for x in xs0]
        pageable_out = [torch.empty(N, dtype=torch.bfloat16) for _ in range(R)]
        t_pg = time_e2e(ar, R, N, min(e2e_steps, 50), 3, stream, pageable_in, pageable_out)
        extra["e2e_pageable_staging_us_per_call"] = round(t_pg * 1e6 / min(e2e_steps, 50), 3)

    # Every call of the run must have completed without a device-side timeout:
    # a packet wait that gave up leaves undefined outputs, so fail loudly.
    status = ar.device_status(stream)
    if status != 0:
        raise RuntimeError("device error word set during the run (status %d)" % status)
    ar.close()
    del sets, host_in, host_out
    torch.cuda.empty_cache()

    # ---- the oracle on the host cores (rank 0, one GPU only), and the check
    # of the timed variant's output against it
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        lib = oracle.load()
        cores, model = host_cpu()
        t_call, calls, want = oracle_time([inputs.bits(x) for x in xs0], args.cpu_seconds, lib)
        bad = sum(int(np.count_nonzero(g != want)) for g in got)
        per_config = {args.workload: {"us_per_call": round(t_call * 1e6, 1),
                                      "GBps_4RN": round(min_b / t_call / 1e9, 3),
                                      "sample": "%d full calls" % calls}}
        if not args.no_extra:
            for name in EXTRA_WORKLOADS:
                if name == args.workload:
                    continue
                wl = inputs.WORKLOADS[name]
                n = min(wl.count, 1 << 21)
                xs = [inputs.bits(x) for x in inputs.make_inputs(wl.R, n, 0, wl.fill)]
                t_s, c_s, _ = oracle_time(xs, args.cpu_seconds / 4, lib)
                t_full = t_s * wl.count / n
                per_config[name] = {
                    "us_per_call": round(t_full * 1e6, 1),
                    "GBps_4RN": round(4 * wl.R * wl.count / t_full / 1e9, 3),
                    "sample": "%d calls on %d of %d elements per rank (R=%d), scaled to a "
                              "full call" % (c_s, n, wl.count, wl.R)}
        cpu = {"value": round(t_call * 1e6, 1), "unit": "us/call", "cores": 1,
               "host_cores": cores, "cpu_model": model, "kind": "oracle",
               "sample": "%d full calls of the workload (R=%d, N=%d), single-threaded C" % (
                   calls, R, N),
               "GBps_4RN": round(min_b / t_call / 1e9, 3),
               "gpu_output_vs_oracle": "bitexact" if bad == 0 else "MISMATCH (%d elements)" % bad,
               "checked": "all %d outputs of one %s call on the timed workload's input set 0"
                          % (R, args.variant),
               "per_config": per_config}
        if bad:
            raise RuntimeError("%s output differs from the oracle in %d elements" % (
                args.variant, bad))

    # ---- the other benchmark workloads: the fused kernel and the fan-out
    if not args.no_extra and world == 1:
        for name in EXTRA_WORKLOADS:
            if name == args.workload:
                continue
            wl = inputs.WORKLOADS[name]
            tsets = device_sets(wl.R, wl.count, sets_for(4 * wl.R * wl.count), dev)
            art = AllReduce(wl.R, wl.count, device=dev)
            for v in ("fused_ll8", "oneshot_fanout"):
                n = min(args.steps, 2000 if wl.count < (1 << 24) else 400)
                t, pv, _, _ = time_variant(art, tsets, wl.count, v, n, 20, stream, args.timing)
                avg = statistics.fmean(pv)
                extra["%s_%s" % (name, v)] = {
                    "us_per_call": round(t * 1e6 / n, 3),
                    "alg_GBps": round(alg_bytes(v, wl.R, wl.count) / avg / 1e9, 1),
                    "frac_min_bytes": round(4 * wl.R * wl.count / avg / 1e9 / peak, 4)}
            if art.device_status(stream) != 0:
                raise RuntimeError("device error word set during the %s extras" % name)
            art.close()
            del tsets
            torch.cuda.empty_cache()
            extra["%s_copy_same_bytes" % name] = copy_entry(
                wl.R, wl.count, min(args.steps, 2000 if wl.count < (1 << 24) else 400), stream,
                dev, peak, extra["%s_oneshot_fanout" % name]["us_per_call"])
        if "%s_fused_ll8" % "r8_64mib" in extra and "r8_64mib_oneshot_fanout" in extra:
            extra["r8_64mib_fused_over_fanout"] = round(
                extra["r8_64mib_fused_ll8"]["us_per_call"] /
                extra["r8_64mib_oneshot_fanout"]["us_per_call"], 3)
    if sampler:
        sampler.stop()

    line = {
        "metric": METRIC, "value": round(us_per_call, 3), "unit": "us/call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_max * 1e3 / args.steps, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "R": R, "count": N,
                   "shape": list(w.shape), "fill": w.fill, "variant": args.variant,
                   "timing": args.timing,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs rotate over %d buffer sets (%.0f MB touched between reuses)"
                         % (nsets, (nsets - 1) * per_set / 1e6)},
        "hbm_GBps": round(achieved, 1),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_call(args.variant, R),
        "clocks": clocks,
        "extra": extra,
        "device_status": "ok",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# reference arm: the oracle on the host cores

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from shot_allreduce_ranks_gb300 import inputs
    oracle.build()
    lib = oracle.load()
    w = inputs.WORKLOADS[args.workload]
    R, N = w.R, w.count
    cores, model = host_cpu()
    # calibrate the per-element cost, then size each step's sample so the
    # whole run stays within about a minute
    probe = min(N, 1 << 16)
    xs = [inputs.bits(x) for x in inputs.make_inputs(R, probe, 0, w.fill)]
    t0 = time.perf_counter()
    oracle.allreduce_bf16(xs, lib=lib)
    per_elem = max((time.perf_counter() - t0) / probe, 1e-10)
    budget = 60.0
    sample = int(budget / ((args.steps + args.warmup) * per_elem))
    sample = max(8, min(N, sample - sample % 8))
    xs = [inputs.bits(x) for x in inputs.make_inputs(R, sample, 0, w.fill)]
    out = None
    for _ in range(args.warmup):
        out = oracle.allreduce_bf16(xs, lib=lib, outputs=out)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        out = oracle.allreduce_bf16(xs, lib=lib, outputs=out)
    el = time.perf_counter() - t0
    us_full_call = el / args.steps * (N / sample) * 1e6
    desc = "%d of %d elements per rank per step (R=%d), single-threaded C, scaled to a full call" % (
        sample, N, R)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us_full_call, 3),
        "unit": "us/call", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 accumulate, bf16 I/O",
        "data": "synthetic",
        "config": {"workload": args.workload, "R": R, "count": N, "shape": list(w.shape),
                   "fill": w.fill, "variant": "oracle"},
        "cpu_baseline": {"value": round(us_full_call, 3), "unit": "us/call", "cores": 1,
                         "host_cores": cores, "cpu_model": model,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(us_full_call, 3), "unit": "us/call",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# sweep mode: every variant over the benchmark message sizes

SWEEP_VARIANTS = ["oneshot_pull", "oneshot_fanout", "oneshot_fanout_bulk", "twophase",
                  "fused_ll8", "fused_ll8_staged", "packet_3op"]


def sweep_counts():
    from shot_allreduce_ranks_gb300 import inputs
    counts = {4096 << k for k in range(14)}
    counts |= {w.count for w in inputs.WORKLOADS.values()}
    return sorted(counts)


# Variants the selector may choose (the staged and three-launch packet forms
# are comparisons, not candidates).
SELECTABLE = ("oneshot_pull", "oneshot_fanout", "oneshot_fanout_bulk", "twophase", "fused_ll8")
MAX_TUNED_COUNT = 1 << 40


def tuning_rows(R, timings):
    """Selector rows (R, max_count, variant) from measured us/call.

    `timings` maps count -> {variant: us}.  The fastest selectable variant at
    each measured count wins; consecutive counts with the same winner merge
    into one row; a row ends at the geometric mean of the last count its
    variant won and the first count the next one won (where the two curves
    cross, to the resolution of the sweep); the last row is open-ended."""
    winners = []
    for c in sorted(timings):
        cand = {v: t for v, t in timings[c].items() if v in SELECTABLE}
        if cand:
            winners.append((c, min(sorted(cand), key=cand.get)))
    rows = []
    for i, (c, v) in enumerate(winners):
        if i + 1 < len(winners) and winners[i + 1][1] == v:
            continue
        if i + 1 < len(winners):
            nxt = winners[i + 1][0]
            bound = max(c, min(math.isqrt(c * nxt), nxt - 1))
        else:
            bound = MAX_TUNED_COUNT
        rows.append((R, bound, v))
    return rows


def write_tuning(path, rows, header):
    """The AR_TUNING_FILE format: one "R max_count variant" row per line."""
    with open(path, "w") as f:
        f.write("# %s\n" % header)
        for R, max_count, v in rows:
            f.write("%d %d %s\n" % (R, max_count, v))


def run_sweep(args):
    """One JSON line per (count, variant): graph-replay us/call and
    algorithmic GB/s, inputs rotating over more than L2."""
    import torch
    from shot_allreduce_ranks_gb300 import AllReduce
    from shot_allreduce_ranks_gb300 import build as lib_build
    lib_build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    dtype = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[args.dtype]
    ebytes = 4 if args.dtype == "fp32" else 2
    R = args.sweep_r
    counts = sweep_counts()
    variants = [v for v in SWEEP_VARIANTS
                if not (R > 8 and v in ("fused_ll8", "fused_ll8_staged",
                                        "packet_3op"))]
    ar = AllReduce(R, max(counts), device=dev, dtype=dtype)
    peak, _ = measured_peaks()
    timings = {}
    for N in counts:
        per = 2 * ebytes * R * N
        nsets = min(16, max(2, math.ceil(3 * L2_BYTES / per)))
        sets = []
        for _ in range(nsets):
            xin = [torch.randn(N, device=dev).to(dtype) for _ in range(R)]
            sets.append((None, xin, [torch.empty_like(x) for x in xin]))
        steps = max(100, min(2000, int(2e5 / (per / 1e6 + 5))))
        ar.set_variant("auto")
        auto_choice = ar.select(N)
        for v in variants:
            t, _, _, _ = time_variant(ar, sets, N, v, steps, 20, stream, "graph")
            us = t * 1e6 / steps
            timings.setdefault(N, {})[v] = us
            alg = alg_bytes(v, R, N) * ebytes // 2
            print(json.dumps({"R": R, "count": N, "dtype": args.dtype, "variant": v,
                              "us_per_call": round(us, 3),
                              "alg_GBps": round(alg / (us * 1e3), 1),
                              "frac_of_measured": round(alg / (us * 1e3) / peak, 4),
                              "auto_selects": auto_choice}), flush=True)
        del sets
        torch.cuda.empty_cache()
    if ar.device_status() != 0:
        raise RuntimeError("device error word set during the sweep")
    ar.close()
    if args.write_tuning:
        rows = tuning_rows(R, timings)
        write_tuning(args.write_tuning, rows,
                     "selector table from bench.py --sweep (R=%d, %s, graph replay); "
                     "load with AR_TUNING_FILE" % (R, args.dtype))
        print(json.dumps({"tuning_file": args.write_tuning,
                          "rows": [list(r) for r in rows]}), flush=True)


def run_collective(args):
    """Reduce-scatter or all-gather of the workload's message, one JSON line:
    graph-replay us/call and algorithmic GB/s.  reduce_scatter: every rank
    holds N elements (R blocks of N/R) and receives its block of the sum;
    all_gather: every rank holds N/R elements and receives all N."""
    import torch
    from shot_allreduce_ranks_gb300 import AllReduce, inputs
    from shot_allreduce_ranks_gb300 import build as lib_build
    lib_build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    dtype = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[args.dtype]
    ebytes = 4 if args.dtype == "fp32" else 2
    w = inputs.WORKLOADS[args.workload]
    R, N = w.R, w.count
    b = N // R
    rs = args.collective == "reduce_scatter"
    n_in, n_out = (R * b, b) if rs else (b, R * b)
    alg = ebytes * R * (n_in + n_out)  # every input read once, every output written once
    nsets = min(16, max(2, math.ceil(3 * L2_BYTES / alg)))
    sets = [([torch.randn(n_in, device=dev).to(dtype) for _ in range(R)],
             [torch.empty(n_out, dtype=dtype, device=dev) for _ in range(R)])
            for _ in range(nsets)]
    ar = AllReduce(R, R * b, device=dev, dtype=dtype)

    def call(i):
        xin, xout = sets[i % nsets]
        if rs:
            ar.reduce_scatter(xin, xout, recvcount=b, stream=stream)
        else:
            ar.all_gather(xin, xout, sendcount=b, stream=stream)

    with torch.cuda.stream(stream):  # also builds every set's pointer tables before capture
        for i in range(max(3, nsets, args.warmup)):
            call(i)
    torch.cuda.synchronize()
    per_graph = 50
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(per_graph):
            call(i)
    reps = max(1, args.steps // per_graph)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * per_graph)
    peak, peak_kind = measured_peaks()
    if ar.device_status() != 0:
        raise RuntimeError("device error word set")
    print(json.dumps({"collective": args.collective, "workload": args.workload, "R": R,
                      "block": b, "dtype": args.dtype, "calls": reps * per_graph,
                      "us_per_call": round(us, 3), "alg_bytes_per_call": alg,
                      "alg_GBps": round(alg / (us * 1e3), 1),
                      "frac_of_measured": round(alg / (us * 1e3) / peak, 4),
                      "peak_kind": peak_kind, "gpu_launches": reps * per_graph}), flush=True)
    ar.close()


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="r8_512x8192")
    p.add_argument("--variant", default="fused_ll8",
                   choices=["oneshot_pull", "oneshot_fanout", "twophase", "fused_ll8",
                            "oneshot_fanout_bulk", "fused_ll8_staged", "packet_3op"])
    p.add_argument("--timing", choices=["graph", "stream"], default="graph",
                   help="graph: calls replayed from CUDA graphs; stream: plain launches")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-extra", action="store_true")
    p.add_argument("--sweep", action="store_true",
                   help="time every variant over the benchmark message sizes (JSON lines)")
    p.add_argument("--sweep-r", type=int, default=8)
    p.add_argument("--write-tuning", default=None, metavar="FILE",
                   help="with --sweep: write the fastest variant per size as an "
                        "AR_TUNING_FILE selector table")
    p.add_argument("--dtype", choices=["bf16", "fp16", "fp32"], default="bf16",
                   help="element type of --sweep and --collective")
    p.add_argument("--collective", choices=["reduce_scatter", "all_gather"], default=None,
                   help="time ar_reduce_scatter / ar_all_gather on the workload (JSON line)")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    a = p.parse_args(argv)
    if a.warmup < 3:
        p.error("--warmup must be >= 3")
    return a


def main(argv=None):
    args = parse_args(argv)
    if args.sweep:
        run_sweep(args)
    elif args.collective:
        run_collective(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
