#!/usr/bin/env python
"""Throughput benchmark of the tiled-attention hot path on GB300.

One step = the whole path once over one batch of synthetic input:
fa_forward (O, LSE) -> fa_backward_dq (delta, dQ) -> fa_backward_dkdv (dK, dV),
bf16 inputs and gradients, fp32 accumulation.  Default workload: B=2 H=16
N=4096 D=128 causal, the forward + split-backward case at D=128, N>=4096.

Metric: attention TFLOP/s with the FLOPs counted algorithmically -- forward
4 B H N^2 D, backward as its 7 GEMMs 14 B H N^2 D, both halved for causal.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline]
                    [--no-workloads] [--sustained-s S]

Besides the headline step, the JSON line carries (at N=1) a ``workloads``
object with every workload shape of the path (each fp32 / bf16 forward, both
masks where both are run, the forward + backward cases), each timed the same
way with its own clock record, and a ``sustained`` object: the headline step
repeated back to back for several seconds, against the sustained tensor peak.

Timing: CUDA events on the launching stream around each kernel of each step;
L2 is flushed (a 512 MB write) before every timed step, outside the events;
a barrier + synchronize brackets the K timed steps; the job time is the max
over ranks.  Multi-GPU (torchrun): every rank runs its own batch of the same
shape (weak scaling, no collective on the data path).
``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload on the host cores (the reference arm of this path).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "bwd_bf16_b2h16n4096d128_causal"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- host-side helpers (CPU-testable)
def step_flops(B, H, N, D, causal, passes=("fwd", "bwd")) -> float:
    per = (4.0 if "fwd" in passes else 0.0) + (14.0 if "bwd" in passes else 0.0)
    f = per * B * H * float(N) * N * D
    return f / 2 if causal else f


def kernel_flops(B, H, N, D, causal):
    c = 0.5 if causal else 1.0
    u = B * H * float(N) * N * D * c
    # the comparator backward is counted in the same 7-GEMM units as the split one (same work, same
    # results), so the two lines compare directly; it performs 5 of those GEMMs
    return {"fwd": 4 * u, "bwd_dq": 6 * u, "bwd_dkdv": 8 * u, "bwd_atomic": 14 * u}


def backward_flops(B, H, N, D, causal):
    """The backward's FLOPs under both conventions: the 7 GEMMs the split backward runs (14 B H N^2 D)
    and the conventional 5-GEMM count (10 B H N^2 D), both halved for causal."""
    c = 0.5 if causal else 1.0
    u = B * H * float(N) * N * D * c
    return {"7gemm": 14 * u, "5gemm": 10 * u}


def backward_summary(ms_dq: float, ms_dkdv: float, B, H, N, D, causal, peak: float) -> dict:
    """The split backward (dQ kernel + dK/dV kernel) as one number under both FLOP conventions."""
    ms = ms_dq + ms_dkdv
    f = backward_flops(B, H, N, D, causal)
    t7 = f["7gemm"] / (ms * 1e-3) / 1e12
    t5 = f["5gemm"] / (ms * 1e-3) / 1e12
    return {"ms": ms, "tflops_7gemm": t7, "frac_7gemm": t7 / peak, "tflops_5gemm": t5, "frac_5gemm": t5 / peak}


def aggregate(local_seconds: float, local_flops: float, world: int, reduce_max=None, reduce_sum=None):
    """Whole-job throughput: all ranks' FLOPs over the slowest rank's time."""
    t = reduce_max(local_seconds) if reduce_max else local_seconds
    f = reduce_sum(local_flops) if reduce_sum else local_flops * world
    return f / t, t


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


CSRC = "attention_tiled_fwd_gb300/csrc/"


def kernel_sources(kernel: str, D: int, dtype: str = "bf16"):
    """The source files whose kernels run for `kernel` at head dimension D (for keying ncu figures)."""
    # fa_api.cu picks the causal work order (the head groups), which sets the DRAM traffic
    common = [CSRC + "sm100_ptx.cuh", CSRC + "fa_internal.h", CSRC + "fa_api.cu"]
    if kernel == "fwd":
        if dtype == "f32":
            return [CSRC + "fwd_f32.cu", CSRC + "fa_internal.h"]
        Dk = 64 if D <= 64 else 128 if D <= 128 else 256
        own = {64: ["fwd_bf16_duo.cu", "sched.cuh"], 128: ["fwd_bf16_pair.cu"]}.get(Dk, [])
        return [CSRC + "fwd_bf16.cu"] + [CSRC + f for f in own] + common
    if kernel == "bwd_dq":
        return [CSRC + ("bwd_dq_k128.cu" if D <= 64 else "bwd_dq.cu")] + common
    if kernel == "bwd_dkdv":
        return [CSRC + ("bwd_dkdv_q128.cu" if D <= 64 else "bwd_dkdv.cu")] + common
    if kernel == "decode_stream":
        return [CSRC + "decode.cu"] + common
    return [CSRC + "bwd_atomic.cu"] + common


def traffic_for(kernel: str, workload: str, D: int = 128, dtype: str = "bf16"):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e:
        return None
    cur = source_hash([os.path.join(ROOT, s) for s in kernel_sources(kernel, D, dtype)])
    return e["bytes_per_launch"] if e.get("source_hash") == cur else None


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*) that the timing rules name.
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                0x80: "hw_power_brake_slowdown"}


def decode_reasons(mask: int):
    """Names of the clock-event reasons set in an NVML reason bit mask."""
    return sorted(name for bit, name in NVML_REASONS.items() if mask & bit)


class NvmlReader:
    """Read-only NVML queries through ctypes: SM clock, its maximum, power draw and the clock-event
    reasons of one GPU, found by PCI bus id (so CUDA and NVML agree on the device).  Nothing is set."""

    def __init__(self, lib, handle, reasons_fn):
        self.lib, self.h, self.reasons_fn = lib, handle, reasons_fn

    @classmethod
    def open(cls, pci_domain: int, pci_bus: int, pci_device: int):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            bus = f"{pci_domain:08x}:{pci_bus:02x}:{pci_device:02x}.0".encode()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                return None
            reasons_fn = None
            for name in ("nvmlDeviceGetCurrentClocksEventReasons", "nvmlDeviceGetCurrentClocksThrottleReasons"):
                try:
                    reasons_fn = getattr(lib, name)
                    break
                except AttributeError:
                    continue
            if reasons_fn is None:
                return None
            r = cls(lib, h, reasons_fn)
            return r if r.read() is not None else None
        except (OSError, AttributeError):
            return None

    def read(self):
        import ctypes
        sm, mx, mw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        NVML_CLOCK_SM = 1
        if (self.lib.nvmlDeviceGetClockInfo(self.h, NVML_CLOCK_SM, ctypes.byref(sm)) != 0 or
                self.lib.nvmlDeviceGetMaxClockInfo(self.h, NVML_CLOCK_SM, ctypes.byref(mx)) != 0 or
                self.reasons_fn(self.h, ctypes.byref(reasons)) != 0):
            return None
        power = mw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw)) == 0 else None
        return {"sm_mhz": float(sm.value), "sm_max_mhz": float(mx.value), "power_w": power,
                "reasons": int(reasons.value)}


class ClockSampler:
    """SM clocks and clock-event reasons sampled while the timed region runs: through NVML every 2 ms
    when it can be opened (reader: an object with read() -> dict as NvmlReader gives), else through
    nvidia-smi every 50 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, reader=None, period_s: float = 0.002):
        self.gpu = gpu_index
        self.reader = reader
        self.period = period_s
        self.proc = None
        self.running = False
        self.lines = []    # nvidia-smi: (time, csv line)
        self.samples = []  # NVML: (time, dict)
        self.t_start = self.t_stop = None

    def start(self):
        if self.reader is None:
            try:
                import torch
                p = torch.cuda.get_device_properties(self.gpu)
                self.reader = NvmlReader.open(p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
            except Exception:
                self.reader = None
        if self.reader is not None:
            self.running = True
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self):
        while self.running:
            r = self.reader.read()
            if r is not None:
                self.samples.append((time.time(), r))
            time.sleep(self.period)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def _inside(self, t):
        return self.t_start is not None and self.t_start <= t <= (self.t_stop or 1e30)

    def stop(self):
        if self.reader is not None and self.running:
            self.running = False
            self.thread.join(timeout=1.0)
            inside = [r for t, r in self.samples if self._inside(t)]
            used = inside if inside else [r for _, r in self.samples[-2:]]
            mhz = [r["sm_mhz"] for r in used]
            mask = 0
            for r in used:
                mask |= r["reasons"]
            power = [r["power_w"] for r in used if r["power_w"] is not None]
            return {"sm_mhz": statistics.median(mhz) if mhz else None,
                    "sm_max_mhz": max(r["sm_max_mhz"] for r in used) if used else None,
                    "reasons": decode_reasons(mask), "samples": len(inside),
                    "power_w_max": max(power) if power else None, "source": "nvml, every 2 ms"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        inside = [r for r in rows if self._inside(r[0])]
        used = inside if inside else rows[-2:]
        mhz = [float(p[1]) for _, p in used if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for _, p in used if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in used for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max((float(p[3]) for _, p in used if p[3].replace(".", "").isdigit()),
                                   default=None), "source": "nvidia-smi, every 50 ms"}


# ----------------------------------------------------------------------------- CPU baseline (the oracle)
def rows_flops(N, D, causal, i0, i1) -> float:
    """Algorithmic FLOPs of query rows [i0, i1) of one head: (4 + 14) x visible keys x D per row."""
    if causal:
        nvis = (i1 * (i1 + 1) - i0 * (i0 + 1)) / 2.0
    else:
        nvis = float(i1 - i0) * N
    return 18.0 * nvis * D


class OracleSample:
    """The float64 oracle's forward + backward over the last r query rows of `heads` heads of the
    workload (one head per host thread), r sized so one run takes about target_s seconds."""

    def __init__(self, w, threads: int):
        import oracle
        from synthetic_inputs import make_qkv
        oracle.build()
        self.oracle = oracle
        self.w = w
        self.threads = threads
        self.heads = [(b, h) for b in range(w.B) for h in range(w.H)][:max(1, threads)]
        self.inp = make_qkv(w.B, w.H, w.N, w.D, w.seed, w.dtype, w.std, with_dO=True)
        self.rows = min(16, w.N)
        self.run()  # calibration on a few rows

    def size_for(self, target_s: float):
        w = self.w
        f_small, t_small = self.last
        per_flop = t_small / max(f_small, 1.0)
        # rows from the end of the head (the heaviest ones when causal): grow until the estimate fits
        lo, hi = 1, w.N
        while lo < hi:
            mid = (lo + hi + 1) // 2
            est = per_flop * rows_flops(w.N, w.D, w.causal[0], w.N - mid, w.N) * len(self.heads)
            if est <= target_s:
                lo = mid
            else:
                hi = mid - 1
        self.rows = max(1, lo)

    def run(self):
        w = self.w
        i0, i1 = w.N - self.rows, w.N
        t0 = time.perf_counter()
        self.oracle.backward_row_range(self.inp["q"], self.inp["k"], self.inp["v"], self.inp["dO"], w.scale,
                                       w.causal[0], self.heads, i0, i1, threads=self.threads)
        dt = time.perf_counter() - t0
        f = rows_flops(w.N, w.D, w.causal[0], i0, i1) * len(self.heads)
        self.last = (f, dt)
        return f, dt

    def describe(self, dt=None):
        w = self.w
        extra = f", {dt:.1f} s" if dt is not None else ""
        return (f"query rows {w.N - self.rows}..{w.N - 1} of {len(self.heads)} of the {w.B * w.H} heads "
                f"(N={w.N}, D={w.D}, causal={w.causal[0]}): float64 forward + backward terms of those rows, "
                f"one head per host thread{extra}")


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    smp = OracleSample(w, cores)
    per_step = max(0.5, min(8.0, 150.0 / (args.steps + args.warmup)))
    smp.size_for(per_step)
    times, flops = [], []
    for it in range(args.warmup + args.steps):
        f, dt = smp.run()
        if it >= args.warmup:
            times.append(dt)
            flops.append(f)
    total = sum(times)
    value = sum(flops) / total / 1e12
    line = {"impl": "reference", "metric": "attention fwd+bwd TFLOP/s (bf16; FLOPs 4 B H N^2 D fwd + 14 B H N^2 D "
                                           "bwd (7 GEMMs), halved causal) and fraction of GB300 dense bf16 peak",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal[0]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "each step: " + smp.describe()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- decode (one GPU, own line)
DECODE_SHAPE = dict(B=4, H=32, n_q=1, N=32768, D=128)  # one new token against a 32K-entry K/V cache


def decode_main(args):
    """Decode throughput: GB/s of algorithmic traffic (K and V read once, q read, O and LSE written)
    against the measured HBM copy bandwidth; L2 flushed before every timed call."""
    import torch
    import attention_tiled_fwd_gb300 as fa
    dev = torch.device("cuda", 0)
    shape = dict(DECODE_SHAPE)
    if args.decode_shape:
        shape.update(zip(("B", "H", "n_q", "N", "D"), (int(x) for x in args.decode_shape.split(","))))
    B, H, nq, N, D = (shape[k] for k in ("B", "H", "n_q", "N", "D"))
    g = torch.Generator().manual_seed(2024)
    q = torch.randn(B, H, nq, D, generator=g).bfloat16().to(dev)
    k = torch.randn(B, H, N, D, generator=g).bfloat16().to(dev)
    v = torch.randn(B, H, N, D, generator=g).bfloat16().to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, nq, device=dev)
    ws = torch.empty(fa.fa_decode_workspace_bytes(B, H, nq, N, D), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.fill_(1.0)
        fa.fa_decode(q, k, v, causal=True, o=o, lse=lse, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    sampler.mark_start()
    for e0, e1 in evs:
        flush.fill_(0.0)
        e0.record(stream)
        fa.fa_decode(q, k, v, causal=True, o=o, lse=lse, workspace=ws, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark_stop()
    clocks = sampler.stop()
    if fa.fa_device_status() != 0:
        raise RuntimeError("device status reports a failure")
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    algo_bytes = 2 * B * H * N * D * 2 + B * H * nq * D * 2 * 2 + B * H * nq * 4
    gbs = algo_bytes / (ms * 1e-3) / 1e9
    peaks, kind = load_peaks()
    peak = float(peaks["hbm_gbs"])
    line = {"metric": "decode attention GB/s (K/V cache read once; bf16)", "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1))",
            "config": {"workload": "decode", **shape, "causal": True,
                       "l2": "flushed before every timed call (512 MB write), outside the timed events"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": traffic_for("decode_stream", decode_key(B, H, nq, N, D), D),
                         "peak_source": f"{kind} hbm_gbs (copy)"},
            "gpu_launches": 2 * args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)


def decode_key(B: int, H: int, n_q: int, N: int, D: int) -> str:
    """The decode shape's key in the committed DRAM-traffic table."""
    return f"decode_b{B}h{H}q{n_q}n{N}d{D}"


# ----------------------------------------------------------------------------- every workload, one GPU
def workload_keys():
    """(key, workload, causal) for every workload shape and mask the path is run in."""
    from synthetic_inputs import WORKLOADS
    out = []
    for w in WORKLOADS.values():
        for causal in w.causal:
            key = w.name if len(w.causal) == 1 else f"{w.name}_{'causal' if causal else 'noncausal'}"
            out.append((key, w, causal))
    return out


def time_workload(fa, torch, dev, w, causal, steps: int, warmup: int, flush, peaks) -> dict:
    """One workload timed like the headline step: the forward (and, where the workload has one, the
    split backward with bf16 gradients) per step, CUDA events around every kernel on the launching
    stream, L2 flushed before every step outside the events, SM clocks sampled during the K steps."""
    from synthetic_inputs import make_qkv
    B, H, N, D = w.B, w.H, w.N, w.D
    bwd = "bwd" in w.passes
    host = make_qkv(B, H, N, D, w.seed, w.dtype, w.std, with_dO=bwd)
    q, k, v = (host[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    kernels = ["fwd"]
    if bwd:
        dO = host["dO"].to(dev)
        dq, dk, dv = (torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev) for _ in range(3))
        delta = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        kernels += ["bwd_dq", "bwd_dkdv"]
    stream = torch.cuda.current_stream()
    scale = w.scale

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        fa.fa_forward(q, k, v, scale=scale, causal=causal, o=o, lse=lse, stream=stream)
        if bwd:
            if evs:
                evs[1].record(stream)
            fa.fa_backward_dq(q, k, v, o, dO, lse, scale=scale, causal=causal, dq=dq, delta=delta, stream=stream)
            if evs:
                evs[2].record(stream)
            fa.fa_backward_dkdv(q, k, v, dO, lse, delta, scale=scale, causal=causal, dk=dk, dv=dv, stream=stream)
        if evs:
            evs[-1].record(stream)

    for _ in range(warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kernels) + 1)] for _ in range(steps)]
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.1)
    torch.cuda.synchronize()
    sampler.mark_start()
    for it in range(steps):
        flush.fill_(float(it))
        step(events[it])
    torch.cuda.synchronize()
    sampler.mark_stop()
    clocks = sampler.stop()
    if fa.fa_device_status() != 0:
        raise RuntimeError(f"device status reports a failure in workload {w.name}")
    ms = {kn: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in events) for i, kn in enumerate(kernels)}
    step_ms = statistics.mean(e[0].elapsed_time(e[-1]) for e in events)
    kf = kernel_flops(B, H, N, D, causal)
    peak = float(peaks["bf16_tflops"])
    entry = {"B": B, "H": H, "N": N, "D": D, "causal": causal, "dtype": w.dtype, "steps": steps,
             "warmup": warmup, "gpu_launches": len(kernels) * steps, "clocks": clocks}
    if w.dtype == "f32":
        # the fp32 FFMA forward: a parity path without a tensor-core roofline; its time is the figure
        entry["kernels"] = {"fwd": {"us": 1e3 * ms["fwd"], "tflops": kf["fwd"] / (ms["fwd"] * 1e-3) / 1e12,
                                    "traffic": traffic_for("fwd", w.name, D, "f32")}}
        entry["step_ms"] = step_ms
        return entry
    key_traffic = w.name if len(w.causal) == 1 else f"{w.name}_{'causal' if causal else 'noncausal'}"
    entry["kernels"] = {kn: {"ms": ms[kn], "tflops": kf[kn] / (ms[kn] * 1e-3) / 1e12,
                             "frac_of_peak": kf[kn] / (ms[kn] * 1e-3) / 1e12 / peak,
                             "traffic": traffic_for(kn, key_traffic, D)} for kn in kernels}
    if bwd:
        entry["backward"] = backward_summary(ms["bwd_dq"], ms["bwd_dkdv"], B, H, N, D, causal, peak)
    f = step_flops(B, H, N, D, causal, w.passes)
    entry["step_ms"] = step_ms
    entry["step_tflops"] = f / (step_ms * 1e-3) / 1e12
    entry["step_frac_of_peak"] = entry["step_tflops"] / peak
    return entry


def time_sustained(fa, torch, dev, w, seconds: float, step_ms_hint: float, peaks) -> dict:
    """The headline step repeated back to back for `seconds`, timed as one region by two CUDA events,
    with clocks and power sampled throughout: the figure to hold against the sustained tensor peak.
    No L2 flush between steps: one step's tensors (Q, K, V, O, dO, dQ, dK, dV) exceed the L2."""
    from synthetic_inputs import make_qkv
    B, H, N, D = w.B, w.H, w.N, w.D
    causal = w.causal[0]
    host = make_qkv(B, H, N, D, w.seed, w.dtype, w.std, with_dO=True)
    q, k, v, dO = (host[n].to(dev) for n in ("q", "k", "v", "dO"))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev) for _ in range(3))
    delta = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        fa.fa_forward(q, k, v, scale=w.scale, causal=causal, o=o, lse=lse, stream=stream)
        fa.fa_backward_dq(q, k, v, o, dO, lse, scale=w.scale, causal=causal, dq=dq, delta=delta, stream=stream)
        fa.fa_backward_dkdv(q, k, v, dO, lse, delta, scale=w.scale, causal=causal, dk=dk, dv=dv, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = int(min(50000, max(10, math.ceil(seconds * 1e3 / max(step_ms_hint, 1e-3)))))
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    sampler.mark_start()
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark_stop()
    clocks = sampler.stop()
    if fa.fa_device_status() != 0:
        raise RuntimeError("device status reports a failure in the sustained run")
    total_s = e0.elapsed_time(e1) / 1e3
    tflops = step_flops(B, H, N, D, causal, ("fwd", "bwd")) * n / total_s / 1e12
    sus = float(peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"])
    return {"workload": w.name, "steps": n, "seconds": total_s, "ms_per_step": 1e3 * total_s / n,
            "tflops": tflops, "peak_sustained": sus, "frac_of_sustained_peak": tflops / sus,
            "frac_of_burst_peak": tflops / float(peaks["bf16_tflops"]), "gpu_launches": 3 * n,
            "l2": "not flushed: one step's tensors (268 MB at this shape) exceed the 129 MB L2",
            "clocks": clocks}


# ----------------------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload timings (every workload shape, each with its own clocks)")
    ap.add_argument("--workload-steps", type=int, default=10, help="timed steps per workload in `workloads`")
    ap.add_argument("--sustained-s", type=float, default=3.0,
                    help="seconds of back-to-back headline steps for `sustained` (0: skip)")
    ap.add_argument("--grad-dtype", choices=("bf16", "f32"), default="bf16")
    ap.add_argument("--decode-shape", default="",
                    help="B,H,n_q,N,D for --workload decode (default: the decode benchmark shape)")
    ap.add_argument("--backward", choices=("split", "atomic"), default="split",
                    help="split: fa_backward_dq + fa_backward_dkdv (the method); atomic: the 5-GEMM comparator "
                         "fa_backward_atomic")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.workload == "decode":
        decode_main(args)
        return

    from synthetic_inputs import WORKLOADS, make_qkv
    w = WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch
    import torch.distributed as dist
    import attention_tiled_fwd_gb300 as fa

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def reduce_max(x):
        if world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def reduce_sum(x):
        if world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        return float(t.item())

    B, H, N, D = w.B, w.H, w.N, w.D
    causal = w.causal[0]
    passes = w.passes
    scale = w.scale
    gdt = torch.bfloat16 if args.grad_dtype == "bf16" else torch.float32
    host = make_qkv(B, H, N, D, w.seed + 1000 * rank, w.dtype, w.std, with_dO="bwd" in passes)
    q, k, v = (host[n].to(dev) for n in ("q", "k", "v"))
    dO = host["dO"].to(dev) if "bwd" in passes else None
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    if "bwd" in passes:
        dq = torch.empty((B, H, N, D), dtype=gdt, device=dev)
        dk = torch.empty_like(dq)
        dv = torch.empty_like(dq)
        delta = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq_acc = torch.empty((B, H, N, D), dtype=torch.float32, device=dev) if args.backward == "atomic" else None
    stream = torch.cuda.current_stream()
    bwd_kernels = ["bwd_dq", "bwd_dkdv"] if args.backward == "split" else ["bwd_atomic"]
    kernels = ["fwd"] + (bwd_kernels if "bwd" in passes else [])

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        fa.fa_forward(q, k, v, scale=scale, causal=causal, o=o, lse=lse, stream=stream)
        if "bwd" in passes and args.backward == "atomic":
            if evs:
                evs[1].record(stream)
            fa.fa_backward_atomic(q, k, v, o, dO, lse, scale=scale, causal=causal, dq_accum=dq_acc, dq=dq, dk=dk,
                                  dv=dv, delta=delta, stream=stream)
        elif "bwd" in passes:
            if evs:
                evs[1].record(stream)
            fa.fa_backward_dq(q, k, v, o, dO, lse, scale=scale, causal=causal, dq=dq, delta=delta, stream=stream)
            if evs:
                evs[2].record(stream)
            fa.fa_backward_dkdv(q, k, v, dO, lse, delta, scale=scale, causal=causal, dk=dk, dv=dv, stream=stream)
        if evs:
            evs[-1].record(stream)

    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # > 129 MB L2
    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if fa.fa_device_status() != 0:
        raise RuntimeError("device status reports a failure during warm-up")

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    nev = len(kernels) + 1
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    barrier()
    sampler.mark_start()
    for s in range(args.steps):
        flush.fill_(float(s))
        step(events[s])
    barrier()
    sampler.mark_stop()
    clocks = sampler.stop()
    if fa.fa_device_status() != 0:
        raise RuntimeError("device status reports a failure in the timed region")

    per_kernel = {kname: [] for kname in kernels}
    step_ms = []
    for evs in events:
        for i, kname in enumerate(kernels):
            per_kernel[kname].append(evs[i].elapsed_time(evs[i + 1]))
        step_ms.append(evs[0].elapsed_time(evs[-1]))
    local_s = sum(step_ms) / 1e3
    flops = step_flops(B, H, N, D, causal, passes)
    value, t_max = aggregate(local_s, flops * args.steps, world, reduce_max, reduce_sum)
    kf = kernel_flops(B, H, N, D, causal)
    mean_ms = {kname: statistics.mean(v_) for kname, v_ in per_kernel.items()}
    kernel_tflops = {kname: kf[kname] / (mean_ms[kname] * 1e-3) / 1e12 for kname in kernels}
    dom = max(kernels, key=lambda kn: mean_ms[kn])
    peaks, peak_kind = load_peaks()
    peak = float(peaks["bf16_tflops"])
    roofline = {"bound": "tensor", "kernel": dom, "achieved": kernel_tflops[dom], "peak": peak,
                "unit": "TFLOP/s", "frac": kernel_tflops[dom] / peak, "traffic": traffic_for(dom, w.name, D),
                "peak_source": f"{peak_kind} bf16_tflops (burst, cuBLAS bf16 GEMM)",
                "peak_sustained": float(peaks.get("bf16_tflops_sustained", 0)) or None}

    backward = (backward_summary(mean_ms["bwd_dq"], mean_ms["bwd_dkdv"], B, H, N, D, causal, peak)
                if "bwd_dq" in mean_ms else None)

    # ---- every workload shape, then the headline step held for several seconds (one GPU only)
    workloads = sustained = None
    if world == 1 and not args.no_workloads:
        workloads = {}
        for key, ww, cz in workload_keys():
            workloads[key] = time_workload(fa, torch, dev, ww, cz, max(3, args.workload_steps), 3, flush, peaks)
            torch.cuda.empty_cache()
    if world == 1 and args.sustained_s > 0 and "bwd" in passes and args.backward == "split":
        sustained = time_sustained(fa, torch, dev, w, args.sustained_s, 1e3 * t_max / args.steps, peaks)
        torch.cuda.empty_cache()

    # ---- end to end through the public API: pinned host inputs in, results back out.  Every step copies
    # its inputs in and its gradients out; the copies of neighbouring steps overlap the step's kernels (H2D
    # of step s+1 and D2H of step s-1 on their own streams, two buffer sets), as a training loop would.
    e2e = None
    if not args.no_e2e:
        pin = {n: t.pin_memory() for n, t in host.items()}
        out_names = ["o"] + (["dq", "dk", "dv"] if "bwd" in passes else [])
        outs = [{n: torch.empty((B, H, N, D), dtype=(o.dtype if n == "o" else gdt)).pin_memory()
                 for n in out_names} for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in outs[0].values())
        # two device buffer sets: inputs, outputs and intermediates of one step each
        bufs = []
        for _ in range(2):
            bset = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
            bset["o"] = torch.empty_like(o)
            bset["lse"] = torch.empty_like(lse)
            if "bwd" in passes:
                for n in ("dq", "dk", "dv"):
                    bset[n] = torch.empty((B, H, N, D), dtype=gdt, device=dev)
                bset["delta"] = torch.empty((B, H, N), dtype=torch.float32, device=dev)
                if args.backward == "atomic":
                    bset["acc"] = torch.empty((B, H, N, D), dtype=torch.float32, device=dev)
            bufs.append(bset)

        def run_step(bs, st):
            fa.fa_forward(bs["q"], bs["k"], bs["v"], scale=scale, causal=causal, o=bs["o"], lse=bs["lse"], stream=st)
            if "bwd" in passes and args.backward == "atomic":
                fa.fa_backward_atomic(bs["q"], bs["k"], bs["v"], bs["o"], bs["dO"], bs["lse"], scale=scale,
                                      causal=causal, dq_accum=bs["acc"], dq=bs["dq"], dk=bs["dk"], dv=bs["dv"],
                                      delta=bs["delta"], stream=st)
            elif "bwd" in passes:
                fa.fa_backward_dq(bs["q"], bs["k"], bs["v"], bs["o"], bs["dO"], bs["lse"], scale=scale,
                                  causal=causal, dq=bs["dq"], delta=bs["delta"], stream=st)
                fa.fa_backward_dkdv(bs["q"], bs["k"], bs["v"], bs["dO"], bs["lse"], bs["delta"], scale=scale,
                                    causal=causal, dk=bs["dk"], dv=bs["dv"], stream=st)

        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        n_e2e = max(3, min(args.steps, 50))
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for it in range(n_e2e):
            bi = it % 2
            bs = bufs[bi]
            with torch.cuda.stream(s_in):
                if it >= 2:
                    s_in.wait_event(comp_done[bi])  # step it-2 has finished reading this buffer set
                for n, t in pin.items():
                    bs[n].copy_(t, non_blocking=True)
                in_done[bi].record(s_in)
            stream.wait_event(in_done[bi])
            if it >= 2:
                stream.wait_event(out_done[bi])  # step it-2's results have been copied out
            run_step(bs, stream)
            comp_done[bi].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[bi])
                for n in out_names:
                    outs[bi][n].copy_(bs[n], non_blocking=True)
                out_done[bi].record(s_out)
        stream.wait_event(out_done[(n_e2e - 1) % 2])
        stream.wait_event(out_done[(n_e2e - 2) % 2])
        e1.record(stream)
        barrier()
        e2e_s = e0.elapsed_time(e1) / 1e3
        e2e_val, _ = aggregate(e2e_s, flops * n_e2e, world, reduce_max, reduce_sum)
        e2e = {"value": e2e_val / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": n_e2e,
               "overlap": "H2D of step s+1 and D2H of step s-1 on their own streams while step s computes"}

    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        smp = OracleSample(w, cores)
        smp.size_for(15.0)
        f, dt = smp.run()
        cpu_baseline = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                        "sample": smp.describe(dt)}

    if rank == 0:
        line = {
            "metric": "attention fwd+bwd TFLOP/s (bf16; FLOPs 4 B H N^2 D fwd + 14 B H N^2 D bwd (7 GEMMs), "
                      "halved causal) and fraction of GB300 dense bf16 peak",
            "value": value / 1e12, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1), per-rank seed)",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "D": D, "causal": causal, "passes": list(passes),
                       "grad_dtype": args.grad_dtype, "backward": args.backward,
                       "global_batch": B * world, "seq_len": N,
                       "parallelism": f"replicas x{world} (independent batches)",
                       "l2": "flushed before every timed step (512 MB write), outside the timed events"},
            "kernels": {kn: {"ms": mean_ms[kn], "tflops": kernel_tflops[kn],
                             "frac_of_peak": kernel_tflops[kn] / peak} for kn in kernels},
            "backward": backward,
            "roofline": roofline,
            "cpu_baseline": cpu_baseline,
            "e2e": e2e,
            # fa_backward_atomic launches three kernels (delta, the key-tile pass, dQ conversion)
            "gpu_launches": (len(kernels) + (2 if args.backward == "atomic" and "bwd" in passes else 0)) * args.steps,
            "clocks": clocks,
            "workloads": workloads,
            "sustained": sustained,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
