#!/usr/bin/env python3
"""Benchmark of the forward SSD scan (libssd) on GB300.

Prints one JSON line.  Metric: SSD scan forward tokens*heads per second on
one GPU (B*L*H / time), with the achieved fraction of the HBM roofline of the
dominant kernel.  A step is one full forward scan (all steps of the method)
over one batch of synthetic input that is already resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Under torchrun (N > 1) every rank runs its own copy of the workload on its own
GPU (the scan shards over batch rows and heads with no exchange, so this is
weak scaling); the step time is the maximum over ranks.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_04_gb300.inputs import WORKLOADS, Workload, make_inputs  # noqa: E402

METRIC = "SSD scan fwd tokens·heads/s at 1 GB300; % of HBM/tensor roofline"
UNIT = "tokens·heads/s"
DEFAULT_WORKLOAD = "mamba2_2p7b_layer"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------ accounting
def algorithmic_bytes(w: Workload, final_state: bool = True) -> int:
    """Bytes a scan must move at least once: read x, dt_raw, B, C, the three
    per-head parameter vectors and the initial state (when given); write y
    and the final state.  Chunk states and scratch are not counted."""
    es = 2 if w.dtype == "bf16" else 4
    BL = w.batch * w.seqlen
    x = BL * w.nheads * w.headdim * es
    dt = BL * w.nheads * 4
    bc = 2 * BL * w.ngroups * w.dstate * es
    par = 3 * w.nheads * 4
    state = w.batch * w.nheads * w.headdim * w.dstate * 4
    return x + dt + bc + par + (state if w.init_state else 0) + x + (state if final_state else 0)


def algorithmic_flops(w: Workload) -> int:
    """Tensor FLOPs of the chunked method at its stated chunk length Q:
    causal C B^T per (chunk, group), causal masked M x, chunk state and C P
    per (chunk, head), state passing per (chunk, head)."""
    Q, N, P = w.chunk, w.dstate, w.headdim
    nc = -(-w.seqlen // Q)
    tri = Q * (Q + 1) // 2
    per_cg = 2 * tri * N
    per_ch = 2 * tri * P + 2 * Q * N * P + 2 * Q * N * P + 2 * N * P
    return w.batch * nc * (w.ngroups * per_cg + w.nheads * per_ch)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "ssd_chunk_fused_kernel": ("ssd_chunk.cu", "ptx.cuh", "tmap.h"),
    "ssd_decode_kernel": ("ssd_decode.cu",),
    "ssd_seq_kernel": ("ssd_seq.cu", "warp_rows.cuh", "f32x2.cuh"),
    "ssd_seq_rows_kernel": ("ssd_seq.cu", "warp_rows.cuh", "f32x2.cuh"),
    "ssd_trap_seq_kernel": ("ssd_trap.cu", "warp_rows.cuh"),
    "ssd_trap_decode_kernel": ("ssd_trap.cu", "warp_rows.cuh"),
    "ssd_conv1d_silu_kernel": ("ssd_neighbors.cu",),
    "ssd_gated_rmsnorm_kernel": ("ssd_neighbors.cu",),
    "ssd_bwd_kernel": ("ssd_bwd.cu", "warp_rows.cuh"),
    "ssd_scan_bwd": ("ssd_bwd.cu", "ssd_bwd_chunk.cu", "ssd_bwd_tc.cu", "warp_rows.cuh", "f32x2.cuh", "ptx.cuh", "tmap.h"),
    "ssd_complex_seq_kernel": ("ssd_complex.cu", "warp_rows.cuh", "f32x2.cuh"),
    "ssd_complex_decode_kernel": ("ssd_complex.cu", "warp_rows.cuh", "f32x2.cuh"),
    "ssd_complex_tc_kernel": ("ssd_complex_tc.cu", "ptx.cuh", "tmap.h"),
}

# fp32 FFMA peak of one GB300: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz
# (the maximum SM clock), for kernels bound by plain fp32 arithmetic
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def seq_kernel_name(w: Workload) -> str:
    """The sequential path's kernel for these sizes: the row layout where N % 4
    == 0, N <= 512 and P fits 16 warps of 8 / NV rows, else the slice layout."""
    nv = 1 if w.dstate <= 128 else (2 if w.dstate <= 256 else 4)
    rows = w.dstate % 4 == 0 and 4 <= w.dstate <= 512 and w.headdim <= 16 * (8 // nv)
    return "ssd_seq_rows_kernel" if rows else "ssd_seq_kernel"


def bwd_chunk_flops(w: Workload) -> int:
    """fp32 flops of the chunk-form backward (chunks of 64 steps) per call:
    per (b, h, chunk) the local states 2 N P Q, and the gradients C B^T (Q^2 N),
    dy x^T (Q^2 P), dx (Q^2 P + Q N P), dB (Q^2 N + Q P N), dC (Q^2 N + Q P N)
    multiply-adds, 2 flops each."""
    Q, N, P = 64, w.dstate, w.headdim
    nc = (w.seqlen + Q - 1) // Q
    fma = 5 * N * P * Q + 3 * Q * Q * N + 2 * Q * Q * P
    return 2 * fma * w.batch * w.nheads * nc


def complex_flops(w: Workload) -> int:
    """fp32 flops of the complex scan per call: per state float and step, the
    complex update (2 multiply-adds and 1 multiply per float of a complex
    pair) and the readout (1 multiply-add), FMA counted as 2."""
    return 7 * w.dstate * w.headdim * w.seqlen * w.batch * w.nheads


def source_digest(kernel: str = "ssd_chunk_fused_kernel") -> str:
    """Digest of a kernel's sources, to tell whether stored ncu counters
    still describe the kernel that runs."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_04_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel", "ssd_chunk_fused_kernel") != kernel:
        return None
    if e.get("source_digest") != source_digest(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------ clocks
# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes; no
    Python package needed).  Nothing here changes a setting of the GPU."""

    def __init__(self, torch_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        bus = None
        try:
            pr = torch.cuda.get_device_properties(torch_index)
            bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        except (AttributeError, RuntimeError):
            bus = None
        ok = bus is not None and self.lib.nvmlDeviceGetHandleByPciBusId_v2(
            bus.encode(), ctypes.byref(self.h)) == 0
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(torch_index, ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def max_sm(self):
        v = self.ct.c_uint()
        return float(v.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.ct.byref(v)) == 0 else None

    def sample(self):
        mhz, rs = self.ct.c_uint(), self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(mhz)) != 0:   # NVML_CLOCK_SM
            return None
        self.reasons_fn(self.h, self.ct.byref(rs))
        return float(mhz.value), int(rs.value)

    def power_w(self):
        mw = self.ct.c_uint()
        return mw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.h, self.ct.byref(mw)) == 0 else None

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while the
    timed region runs.  Through NVML every 0.2 ms when the driver's library
    loads (so that a timed region of a few milliseconds still gets samples),
    else through an nvidia-smi loop every 50 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.samples = []       # (sm MHz, power W, reason bits) from NVML
        self.thread = None
        self.nvml = None
        self.stop = threading.Event()
        self.source = None

    def __enter__(self):
        try:
            self.nvml = _Nvml(self.index)
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return self
        except (OSError, AttributeError):
            self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _poll(self):
        while True:
            v = self.nvml.sample()
            if v is not None:
                self.samples.append(v)
            if self.stop.is_set():
                break
            time.sleep(0.0002)
        self.power = self.nvml.power_w()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self):
        if self.nvml is not None:
            mx = self.nvml.max_sm()
            self.nvml.close()
            reasons = set()
            for _, bits in self.samples:
                for bit, name in _NVML_REASONS.items():
                    if bits & bit:
                        reasons.add(name)
            sm = [v[0] for v in self.samples]
            return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                    "reasons": sorted(reasons), "samples": len(sm),
                    "power_w_end": getattr(self, "power", None),
                    "source": "nvml: SM clock and clock-event reasons polled through the timed region"}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0, "source": self.source}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, every 50 ms"}


# ------------------------------------------------------------ config and L2
L2_BYTES = 129 * 2**20          # GB300 L2
FLUSH_BYTES = 256 * 2**20       # a write this large leaves none of a step's inputs in L2


def flushes_l2(step_bytes: int) -> bool:
    """Whether timed steps that move `step_bytes` (their algorithmic bytes) are
    separated by an L2 flush: when those bytes do not exceed twice the L2, the
    next step would otherwise find much of its input still there."""
    return step_bytes <= 2 * L2_BYTES


def workload_config(w: Workload, seed: int, flush: bool) -> dict:
    """The `config` object of a bench line: the workload, identical for the
    libssd arm and the reference arm (the run's own choices, such as the
    kernel path, go elsewhere in the line)."""
    c = {"workload": w.name}
    if w.op != "ssd":
        c["op"] = w.op
    c.update({"batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
              "dstate": w.dstate, "ngroups": w.ngroups, "chunk": w.chunk, "dtype": w.dtype,
              "init_state": w.init_state, "final_state": True,
              "l2": ("flushed between timed steps (a 256 MB write outside the step's events)"
                     if flush else "inputs larger than L2 (no flush)"),
              "seed": seed})
    return c


def timed_region(ssd, step, steps, stream, dev, dist, local, flush):
    """K steps between a barrier and a synchronize on both sides, each step
    bracketed by CUDA events on the launching stream, with the clocks sampled
    throughout.  With `flush`, a 256 MB write between steps (outside their
    events) evicts the workload from L2, and the region's time is the sum of
    the steps' own times.  Returns (max-over-ranks total ms, per-step ms,
    clock summary, library launches)."""
    scrub = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    launches0 = ssd.launch_count()
    with ClockSampler(local) as clk:
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(steps):
            if flush:
                scrub.fill_(float(i))
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
    launches = ssd.launch_count() - launches0
    per = [a.elapsed_time(b) for a, b in evs]
    total = sum(per) if flush else t_start.elapsed_time(t_end)
    return max_over_ranks(dist, total, dev), per, clk.summary(), launches


# ------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle
def oracle_sample(w: Workload, inp: dict, nb: int, hp: int, ls: int) -> dict:
    """fp64 inputs for a sample of the workload: the first `nb` batch rows, the
    first `hp` heads (all heads, or heads of group 0 only when fewer) and the
    first `ls` steps."""
    if hp >= w.nheads:
        hs, gs = slice(None), slice(None)
    else:
        hp = min(hp, w.nheads // w.ngroups)
        hs, gs = slice(0, hp), slice(0, 1)
    cut = {"x": (slice(0, nb), slice(0, ls), hs), "dt_raw": (slice(0, nb), slice(0, ls), hs),
           "B": (slice(0, nb), slice(0, ls), gs), "C": (slice(0, nb), slice(0, ls), gs),
           "init_state": (slice(0, nb), hs), "dt_bias": (hs,), "A_log": (hs,), "D": (hs,)}
    return {k: (None if v is None else v[cut[k]].double().numpy()) for k, v in inp.items()}


def size_oracle_sample(w: Workload, inp: dict, target_s: float):
    """(nb, hp, ls) for an oracle run of about `target_s` seconds, from the
    time of one calibration chain; the whole workload when that fits."""
    import oracle
    cores = oracle.max_threads()
    lc = min(w.seqlen, 512)
    f64 = oracle_sample(w, inp, 1, 1, lc)
    t0 = time.perf_counter()
    oracle.ssd_fwd(**f64)
    per_step = max((time.perf_counter() - t0) / lc, 1e-9)   # one chain, one thread
    chains = w.batch * w.nheads
    full = -(-chains // cores) * w.seqlen * per_step
    if full <= target_s:
        return w.batch, w.nheads, w.seqlen
    ls = w.seqlen
    fit = int(target_s / (ls * per_step)) * cores          # chains that fit at full length
    if fit < 1:
        return 1, 1, max(16, min(w.seqlen, int(target_s / per_step)))
    if fit >= w.nheads:
        return min(w.batch, fit // w.nheads), w.nheads, ls
    return 1, min(fit, w.nheads // w.ngroups), ls


def cpu_oracle_sample(w: Workload, inp: dict, shape, min_seconds: float = 0.0):
    """Times the fp64 oracle on the sample `shape` = (nb, hp, ls), repeated
    until `min_seconds` have passed.  Returns (tokens*heads per second, cores,
    description)."""
    import oracle
    nb, hp, ls = shape
    f64 = oracle_sample(w, inp, nb, hp, ls)
    hp = f64["x"].shape[2]
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.ssd_fwd(**f64)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    th = nb * ls * hp
    return (th * reps / dt, oracle.max_threads(),
            f"{nb} of {w.batch} batch rows x {hp} of {w.nheads} heads x {ls} of {w.seqlen} steps "
            f"({th} token*heads), {reps} run(s) in {dt:.2f} s")


# ------------------------------------------------------------ GPU arm
def run_gpu(args, w: Workload):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    from selective_state_space_04_gb300 import build
    build.build()
    from selective_state_space_04_gb300 import ssd

    inp = make_inputs(w, seed=args.seed + rank)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    fin = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    path = ssd.select_path((w.batch, w.seqlen, w.nheads, w.headdim), w.ngroups, w.dstate, w.chunk,
                           w.dtype, args.path)
    if path < 0:
        raise SystemExit(f"workload {w.name} not supported: status {-path}")

    def step():
        ssd.ssd_scan_fwd(d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"],
                         d["init_state"], chunk=w.chunk, path=args.path, y=y, final_state=fin,
                         stream=stream, schedule=args.schedule)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if ssd.device_error() != 0:
        raise SystemExit("device error during warm-up")

    # timed region: K steps, per-step CUDA events on the launching stream; a
    # workload that L2 could hold gets an L2 flush between steps, outside the
    # step's events, and its time is the sum of the steps' own times
    flush = flushes_l2(algorithmic_bytes(w))
    total_ms, per_launch_ms, clocks, launches = timed_region(ssd, step, args.steps, stream, dev, dist,
                                                             local, flush)
    if ssd.device_error() != 0:
        raise SystemExit("device error during the timed region")
    warm = None
    if flush:
        # the same steps back to back with no flush (the workload stays in L2)
        ws, we = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ws.record(stream)
        for _ in range(args.steps):
            step()
        we.record(stream)
        torch.cuda.synchronize(dev)
        wms = ws.elapsed_time(we) / args.steps
        warm = {"value": w.token_heads / (wms / 1e3), "ms_per_step": wms,
                "note": "L2-warm: the same steps back to back, no flush"}
    ms_per_step = total_ms / args.steps
    th = w.token_heads
    value = world * th * args.steps / (total_ms / 1e3)

    # end-to-end through the host-buffer entry point: pinned inputs in, y and
    # final state out, every step
    pin = {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}
    yh = torch.empty_like(pin["x"]).pin_memory()
    fh = torch.empty(tuple(fin.shape), dtype=torch.float32).pin_memory()

    def step_host():
        ssd.ssd_scan_fwd_host(pin["x"], pin["dt_raw"], pin["dt_bias"], pin["A_log"], pin["B"],
                              pin["C"], pin["D"], pin["init_state"], chunk=w.chunk, path=args.path,
                              y=yh, final_state=fh, stream=stream, schedule=args.schedule)

    e2e_steps = max(1, min(args.steps, 20))
    step_host()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        step_host()
    e2e_s = max_over_ranks(dist, time.perf_counter() - t0, dev)
    h2d = sum(v.numel() * v.element_size() for v in pin.values() if v is not None)
    d2h = yh.numel() * yh.element_size() + fh.numel() * fh.element_size()
    e2e_value = world * th * e2e_steps / e2e_s

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    alg_bytes = algorithmic_bytes(w, final_state=True)
    # the decode step has no tensor work: its arithmetic is a few fp32 operations
    # per state entry, far below what the state's bytes take to stream
    alg_flops = 0 if path == ssd.PATH_DECODE else algorithmic_flops(w)
    avg_launch_s = statistics.mean(per_launch_ms) / 1e3
    hbm_peak = float(peaks["hbm_gbs"])
    achieved_gbs = alg_bytes / avg_launch_s / 1e9
    t_hbm = alg_bytes / (hbm_peak * 1e9)
    t_tensor = alg_flops / (float(peaks["bf16_tflops"]) * 1e12)
    kernel = {ssd.PATH_CHUNKED: "ssd_chunk_fused_kernel", ssd.PATH_DECODE: "ssd_decode_kernel"}.get(
        path, seq_kernel_name(w))
    traffic = stored_traffic(w.name, kernel)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": workload_config(w, args.seed, flush),
        "run": {"path": {ssd.PATH_CHUNKED: "chunked", ssd.PATH_DECODE: "decode"}.get(path, "sequential"),
                "schedule": ssd.chunk_schedule((w.batch, w.seqlen, w.nheads, w.headdim), w.ngroups,
                                               w.dstate, w.chunk, w.dtype, schedule=args.schedule),
                "launches_per_step": int(launches) // max(1, args.steps)},
        "roofline": {
            "bound": "hbm" if t_hbm >= t_tensor else "tensor",
            "kernel": kernel,
            "achieved": achieved_gbs,
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": achieved_gbs / hbm_peak,
            "peak_source": peak_src,
            "traffic": traffic,
            "algorithmic_bytes_per_launch": alg_bytes,
            "algorithmic_tensor_flops_per_launch": alg_flops,
            "avg_launch_ms": avg_launch_s * 1e3,
            "roofline_ms": max(t_hbm, t_tensor) * 1e3,
            "frac_of_nominal_8TBs": alg_bytes / avg_launch_s / 8.0e12,
        },
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "ssd_scan_fwd_host (pinned host buffers)"},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if warm is not None:
        line["warm_l2"] = warm
    if not args.no_cpu_baseline and world == 1:
        shape = size_oracle_sample(w, inp, 10.0)
        v, cores, sample = cpu_oracle_sample(w, inp, shape, min_seconds=10.0)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ reference arm
def run_reference(args, w: Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    inp = make_inputs(w, seed=args.seed)
    # each step is one oracle run on a sample sized so that the whole run
    # (warm-up and timed steps) takes about two minutes of host time
    per_step_s = min(10.0, max(0.02, 120.0 / (args.steps + args.warmup)))
    shape = size_oracle_sample(w, inp, per_step_s)
    for _ in range(args.warmup):
        cpu_oracle_sample(w, inp, shape)
    times, th_total, sample, cores = 0.0, 0, "", 0
    for _ in range(args.steps):
        v, cores, sample = cpu_oracle_sample(w, inp, shape)
        th = shape[0] * min(shape[1], w.nheads) * shape[2]
        if shape[1] < w.nheads:
            th = shape[0] * min(shape[1], w.nheads // w.ngroups) * shape[2]
        times += th / v
        th_total += th
    value = th_total / times
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": times / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w, args.seed, flushes_l2(algorithmic_bytes(w))),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "per step: " + sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ trapezoidal scan
TRAP_KEYS = ("v", "k", "q", "dt", "a", "trap", "D", "h0", "k0", "v0")


def trap_algorithmic_bytes(w: Workload) -> int:
    """Bytes the trapezoidal scan must move at least once: read v, k, q, dt, a,
    trap, D and the carried states (when given); write y and the states."""
    es = 2 if w.dtype == "bf16" else 4
    BL, BH = w.batch * w.seqlen, w.batch * w.nheads
    vy = 2 * BL * w.nheads * w.headdim * es
    kq = 2 * BL * w.ngroups * w.dstate * es
    coef = 3 * BL * w.nheads * 4
    states = BH * (w.headdim * w.dstate * 4 + (w.dstate + w.headdim) * es)
    return vy + kq + coef + w.nheads * 4 + (states if w.init_state else 0) + states


def trap_oracle_rate(w: Workload, inp: dict, nb: int, min_seconds: float = 0.0):
    """token*heads/s of the fp64 trapezoidal oracle on the first nb batch rows
    (all heads, all steps), repeated until min_seconds have passed."""
    from oracle.trap import trap_fwd
    sl = {n: (None if inp[n] is None else (inp[n] if n == "D" else inp[n][:nb])) for n in TRAP_KEYS}
    reps, t0 = 0, time.perf_counter()
    while True:
        trap_fwd(**sl)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    th = nb * w.seqlen * w.nheads
    return th * reps / dt, (f"{nb} of {w.batch} batch rows x {w.nheads} heads x {w.seqlen} steps "
                            f"({th} token*heads), {reps} run(s) in {dt:.2f} s")


def trap_sample_rows(w: Workload, inp: dict, target_s: float) -> int:
    rate, _ = trap_oracle_rate(w, inp, 1)
    return max(1, min(w.batch, int(target_s * rate / (w.seqlen * w.nheads))))

def run_gpu_trap(args, w: Workload):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    from selective_state_space_04_gb300 import build
    build.build()
    from selective_state_space_04_gb300 import ssd
    from selective_state_space_04_gb300.inputs import make_trap_inputs

    inp = make_trap_inputs(w, seed=args.seed + rank)
    d = {n: (None if inp[n] is None else inp[n].to(dev)) for n in TRAP_KEYS}
    y = torch.empty_like(d["v"])
    hf = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=dev)
    kf = torch.empty((w.batch, w.nheads, w.dstate), dtype=d["v"].dtype, device=dev)
    vf = torch.empty((w.batch, w.nheads, w.headdim), dtype=d["v"].dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    tpath = args.path if args.path in ("chunked", "sequential") else "auto"

    def step():
        ssd.ssd_trap_scan_fwd(*(d[n] for n in TRAP_KEYS), y=y, h_final=hf, k_final=kf, v_final=vf,
                              stream=stream, path=tpath, schedule=args.schedule)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    flush = flushes_l2(trap_algorithmic_bytes(w))
    total_ms, per_launch_ms, clocks, launches = timed_region(ssd, step, args.steps, stream, dev, dist,
                                                             local, flush)
    # the chunked kernel in its trapezoidal mode takes one more launch (the carried k,
    # v): 2 launches per step, 4 on the split schedule; the sequential kernel takes 1
    per_step = launches // max(1, args.steps)
    chunked = per_step >= 2
    th = w.token_heads
    value = world * th * args.steps / (total_ms / 1e3)

    # end to end: every step copies its inputs from pinned host memory, runs the
    # scan through the public call and copies y and the states back
    pin = {n: (None if inp[n] is None else inp[n].contiguous().pin_memory()) for n in TRAP_KEYS}
    outs = [(y, torch.empty(tuple(y.shape), dtype=y.dtype).pin_memory()),
            (hf, torch.empty(tuple(hf.shape), dtype=hf.dtype).pin_memory()),
            (kf, torch.empty(tuple(kf.shape), dtype=kf.dtype).pin_memory()),
            (vf, torch.empty(tuple(vf.shape), dtype=vf.dtype).pin_memory())]

    def step_e2e():
        for n in TRAP_KEYS:
            if pin[n] is not None:
                d[n].copy_(pin[n], non_blocking=True)
        step()
        for dv, hv in outs:
            hv.copy_(dv, non_blocking=True)
        torch.cuda.synchronize(dev)

    e2e_steps = max(1, min(args.steps, 20))
    step_e2e()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        step_e2e()
    e2e_s = max_over_ranks(dist, time.perf_counter() - t0, dev)
    h2d = sum(t.numel() * t.element_size() for t in pin.values() if t is not None)
    d2h = sum(hv.numel() * hv.element_size() for _, hv in outs)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    alg_bytes = trap_algorithmic_bytes(w)
    avg_launch_s = statistics.mean(per_launch_ms) / 1e3
    hbm_peak = float(peaks["hbm_gbs"])
    achieved = alg_bytes / avg_launch_s / 1e9
    kernel = ("ssd_chunk_fused_kernel" if chunked
              else ("ssd_trap_decode_kernel" if w.seqlen == 1 else "ssd_trap_seq_kernel"))
    line = {
        "metric": "trapezoidal (Mamba-3 SISO) scan fwd tokens·heads/s at 1 GB300; % of HBM roofline",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": workload_config(w, args.seed, flush),
        "run": {"path": "chunked" if chunked else "sequential",
                "schedule": ("split" if per_step == 4 else "ranges or pieces") if chunked else "none",
                "launches_per_step": per_step},
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": peak_src,
                     "traffic": stored_traffic(w.name, kernel), "algorithmic_bytes_per_launch": alg_bytes,
                     "timed": "each step: the scan kernel plus, on the chunked path, the small launch that "
                              "writes the carried k and v",
                     "algorithmic_tensor_flops_per_launch": 0, "avg_launch_ms": avg_launch_s * 1e3,
                     "roofline_ms": alg_bytes / (hbm_peak * 1e9) * 1e3},
        "e2e": {"value": world * th * e2e_steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "ssd_trap_scan_fwd with pinned host copies in and out"},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        nb = trap_sample_rows(w, inp, 10.0)
        v, sample = trap_oracle_rate(w, inp, nb, min_seconds=10.0)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)


def run_reference_trap(args, w: Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from selective_state_space_04_gb300.inputs import make_trap_inputs
    inp = make_trap_inputs(w, seed=args.seed)
    nb = trap_sample_rows(w, inp, min(10.0, max(0.02, 120.0 / (args.steps + args.warmup))))
    for _ in range(args.warmup):
        trap_oracle_rate(w, inp, nb)
    secs, th_total, sample = 0.0, 0, ""
    for _ in range(args.steps):
        v, sample = trap_oracle_rate(w, inp, nb)
        th = nb * w.seqlen * w.nheads
        secs += th / v
        th_total += th
    value = th_total / secs
    line = {
        "impl": "reference",
        "metric": "trapezoidal (Mamba-3 SISO) scan fwd tokens·heads/s at 1 GB300; % of HBM roofline",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.seed, flushes_l2(trap_algorithmic_bytes(w))),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": "per step: " + sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ steps around the scan
CONV_TAPS = 4


def complex_takes_tc(w: Workload, path: str = "auto") -> bool:
    """Whether the complex scan runs its chunk form on the tensor cores (the
    library's rule: bf16, P = 64, N = 128, at least two steps, unless the
    sequential kernel is asked for)."""
    return path != "sequential" and w.dtype == "bf16" and w.headdim == 64 and w.dstate == 128 and w.seqlen >= 2


def neighbor_setup(w: Workload, dev, seed: int, path: str = "auto"):
    """(host inputs, device inputs, device outputs, step function, algorithmic
    bytes, kernel name, oracle function of the first nb batch rows) of the
    conv1d + SiLU, gated RMSNorm, backward or complex-scan workload ``w``."""
    from selective_state_space_04_gb300 import ssd
    from selective_state_space_04_gb300.inputs import make_conv_inputs, make_gnorm_inputs
    import oracle.neighbors as on
    es = 2 if w.dtype == "bf16" else 4
    BL, HP, GN = w.batch * w.seqlen, w.nheads * w.headdim, w.ngroups * w.dstate
    if w.op == "conv":
        inp = make_conv_inputs(w, K=CONV_TAPS, seed=seed)
        d = {n: (None if t is None else t.to(dev)) for n, t in inp.items()}
        Cc = HP + 2 * GN
        outs = {"x": torch.empty((w.batch, w.seqlen, w.nheads, w.headdim), dtype=d["xbc"].dtype, device=dev),
                "B": torch.empty((w.batch, w.seqlen, w.ngroups, w.dstate), dtype=d["xbc"].dtype, device=dev),
                "C": torch.empty((w.batch, w.seqlen, w.ngroups, w.dstate), dtype=d["xbc"].dtype, device=dev),
                "conv_state_out": torch.empty((w.batch, CONV_TAPS - 1, Cc), dtype=d["xbc"].dtype, device=dev)}

        def step(stream):
            ssd.conv1d_silu_fwd(d["xbc"], d["weight"], d["bias"], d["conv_state"], nheads=w.nheads,
                                headdim=w.headdim, ngroups=w.ngroups, dstate=w.dstate, stream=stream, **outs)

        state = w.batch * (CONV_TAPS - 1) * Cc * es
        nbytes = 2 * BL * Cc * es + Cc * (CONV_TAPS + 1) * 4 + (state if w.init_state else 0) + state

        def ref(nb):
            on.conv1d_silu(inp["xbc"][:nb], inp["weight"], inp["bias"],
                           None if inp["conv_state"] is None else inp["conv_state"][:nb],
                           w.nheads, w.headdim, w.ngroups, w.dstate)
        return inp, d, outs, step, nbytes, "ssd_conv1d_silu_kernel", ref
    if w.op == "conv_scan":
        # the conv1d + SiLU and the scan in one call (the x channels' conv inside the
        # chunked scan kernel); dt and the head parameters drawn as for the scan
        inp = make_conv_inputs(w, K=CONV_TAPS, seed=seed)
        si = make_inputs(w.with_(init_state=False), seed + 1)
        for n in ("dt_raw", "dt_bias", "A_log", "D"):
            inp[n] = si[n]
        d = {n: (None if t is None else t.to(dev)) for n, t in inp.items()}
        Cc = HP + 2 * GN
        outs = {"y": torch.empty((w.batch, w.seqlen, w.nheads, w.headdim), dtype=d["xbc"].dtype, device=dev),
                "final_state": torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32,
                                           device=dev),
                "conv_state_out": torch.empty((w.batch, CONV_TAPS - 1, Cc), dtype=d["xbc"].dtype, device=dev)}

        def step(stream):
            ssd.conv_scan_fwd(d["xbc"], d["weight"], d["bias"], d["conv_state"], d["dt_raw"], d["dt_bias"],
                              d["A_log"], d["D"], nheads=w.nheads, headdim=w.headdim, ngroups=w.ngroups,
                              dstate=w.dstate, chunk=w.chunk, stream=stream, **outs)
        cstate = w.batch * (CONV_TAPS - 1) * Cc * es
        sstate = w.batch * w.nheads * w.headdim * w.dstate * 4
        nbytes = (BL * Cc * es + Cc * (CONV_TAPS + 1) * 4 + (cstate if w.init_state else 0) + cstate   # conv
                  + BL * w.nheads * 4 + 3 * w.nheads * 4 + BL * HP * es + sstate)                     # scan

        def ref(nb):
            sub = lambda t: None if t is None else t[:nb]   # noqa: E731
            rx, rB, rC, _ = on.conv1d_silu(sub(inp["xbc"]), inp["weight"], inp["bias"], sub(inp["conv_state"]),
                                           w.nheads, w.headdim, w.ngroups, w.dstate)
            import oracle
            oracle.ssd_fwd(rx, sub(inp["dt_raw"]), inp["dt_bias"], inp["A_log"], rB, rC, inp["D"])

        def two_calls(stream):   # the same work as ssd_conv1d_silu_fwd, then ssd_scan_fwd
            x, Bm, Cm, _ = ssd.conv1d_silu_fwd(d["xbc"], d["weight"], d["bias"], d["conv_state"], nheads=w.nheads,
                                               headdim=w.headdim, ngroups=w.ngroups, dstate=w.dstate,
                                               conv_state_out=outs["conv_state_out"], stream=stream)
            ssd.ssd_scan_fwd(x, d["dt_raw"], d["dt_bias"], d["A_log"], Bm, Cm, d["D"], chunk=w.chunk,
                             y=outs["y"], final_state=outs["final_state"], stream=stream)
        step.two_calls = two_calls
        return inp, d, outs, step, nbytes, "ssd_chunk_fused_kernel", ref
    if w.op == "complex":
        from selective_state_space_04_gb300.inputs import make_complex_inputs
        import oracle.complex_scan as ocx
        inp = make_complex_inputs(w, seed=seed)
        d = {n: (None if t is None else t.to(dev)) for n, t in inp.items()}
        outs = {"y": torch.empty_like(d["x"]),
                "final_state": torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32,
                                           device=dev)}

        cpath = path if path in ("chunked", "sequential") else "auto"

        def step(stream):
            ssd.complex_scan_fwd(d["x"], d["dt_raw"], d["dt_bias"], d["A_polar"], d["B"], d["C"], d["D"],
                                 d["init_state"], path=cpath, y=outs["y"], final_state=outs["final_state"],
                                 stream=stream)
        state = w.batch * w.nheads * w.headdim * w.dstate * 4
        nbytes = (2 * BL * HP * es + BL * w.nheads * 4 + 2 * BL * GN * es + 4 * w.nheads * 4
                  + (state if w.init_state else 0) + state)

        def ref(nb):
            ocx.complex_fwd(inp["x"][:nb], inp["dt_raw"][:nb], inp["dt_bias"], inp["A_polar"], inp["B"][:nb],
                            inp["C"][:nb], inp["D"], None if inp["init_state"] is None else inp["init_state"][:nb])
        kernel = ("ssd_complex_decode_kernel" if w.seqlen == 1 else
                  "ssd_complex_tc_kernel" if complex_takes_tc(w, cpath) else "ssd_complex_seq_kernel")
        return inp, d, outs, step, nbytes, kernel, ref
    if w.op == "bwd":
        inp = make_inputs(w, seed=seed)
        rng = np.random.Generator(np.random.PCG64(seed + 1))
        inp["dy"] = torch.from_numpy(rng.standard_normal((w.batch, w.seqlen, w.nheads, w.headdim),
                                                          dtype=np.float32)).to(inp["x"].dtype)
        inp["d_final"] = torch.from_numpy(0.1 * rng.standard_normal((w.batch, w.nheads, w.headdim, w.dstate),
                                                                    dtype=np.float32))
        d = {n: (None if t is None else t.to(dev)) for n, t in inp.items()}
        outs = {}

        def step(stream):
            outs.update(ssd.ssd_scan_bwd(d["x"], d["dt_raw"], d["dt_bias"], d["A_log"], d["B"], d["C"], d["D"],
                                         d["init_state"], d["dy"], d["d_final"], stream=stream))
        f32 = 4
        BH = w.batch * w.nheads
        state = BH * w.headdim * w.dstate * f32
        nbytes = (2 * BL * HP * es + BL * w.nheads * f32 + 2 * BL * GN * es + 3 * w.nheads * f32
                  + (state if w.init_state else 0) + state                        # inputs, dy, d_final
                  + BL * HP * f32 + BL * w.nheads * f32 + 2 * BL * GN * f32 + 3 * w.nheads * f32 + state)  # grads

        def ref(nb):   # nb batch rows, the first 4 heads (the oracle keeps every state)
            import oracle.backward as ob
            hp = min(4, w.nheads // w.ngroups)
            sl = inp
            ob.ssd_bwd(sl["x"][:nb, :, :hp], sl["dt_raw"][:nb, :, :hp], sl["dt_bias"][:hp], sl["A_log"][:hp],
                       sl["B"][:nb, :, :1], sl["C"][:nb, :, :1], sl["D"][:hp],
                       None if sl["init_state"] is None else sl["init_state"][:nb, :hp], sl["dy"][:nb, :, :hp],
                       sl["d_final"][:nb, :hp])
        ref.heads = min(4, w.nheads // w.ngroups)
        return inp, d, outs, step, nbytes, "ssd_scan_bwd", ref
    inp = make_gnorm_inputs(w, seed=seed)
    d = {n: t.to(dev) for n, t in inp.items()}
    outs = {"out": torch.empty_like(d["y"])}

    def step(stream):
        ssd.gated_rmsnorm_fwd(d["y"], d["z"], d["weight"], 1e-6, out=outs["out"], stream=stream)

    def ref(nb):
        on.gated_rmsnorm(inp["y"][:nb], inp["z"][:nb], inp["weight"])
    return inp, d, outs, step, 3 * BL * HP * es + HP * 4, "ssd_gated_rmsnorm_kernel", ref


NEIGHBOR_NAMES = {"conv_scan": "causal conv1d + SiLU and SSD scan fwd (fused)", "conv": "causal conv1d + SiLU fwd", "gnorm": "gated RMSNorm fwd", "bwd": "SSD scan backward",
                  "complex": "complex-valued (ET) scan fwd"}


def neighbor_oracle_rate(w: Workload, ref, target_s: float, min_seconds: float = 0.0):
    """(token*heads/s, description) of the fp64 oracle on enough batch rows
    (whole sequences) for about target_s seconds per run."""
    t0 = time.perf_counter()
    ref(1)
    per_row = max(time.perf_counter() - t0, 1e-6)
    nb = max(1, min(w.batch, int(target_s / per_row)))
    reps, t0 = 0, time.perf_counter()
    while True:
        ref(nb)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    heads = getattr(ref, "heads", w.nheads)
    th = nb * w.seqlen * heads
    return th * reps / dt, (f"{nb} of {w.batch} batch rows x {w.seqlen} steps x {heads} of {w.nheads} heads "
                            f"({th} token*heads), {reps} run(s) in {dt:.2f} s")

def run_gpu_neighbor(args, w: Workload):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    from selective_state_space_04_gb300 import build
    build.build()
    from selective_state_space_04_gb300 import ssd
    inp, d, outs, step, alg_bytes, kernel, ref = neighbor_setup(w, dev, args.seed + rank, args.path)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        step(stream)
    torch.cuda.synchronize(dev)
    flush = flushes_l2(alg_bytes)
    total_ms, per_launch_ms, clocks, launches = timed_region(ssd, lambda: step(stream), args.steps, stream,
                                                             dev, dist, local, flush)
    th = w.token_heads
    value = world * th * args.steps / (total_ms / 1e3)
    # end to end: pinned host copies of the inputs in and of the outputs back, every step
    pin = {n: (None if t is None else t.contiguous().pin_memory()) for n, t in inp.items()}
    back = {n: torch.empty(tuple(t.shape), dtype=t.dtype).pin_memory() for n, t in outs.items()}

    def step_e2e():
        for n, t in pin.items():
            if t is not None:
                d[n].copy_(t, non_blocking=True)
        step(stream)
        for n, t in outs.items():
            back[n].copy_(t, non_blocking=True)
        torch.cuda.synchronize(dev)

    e2e_steps = max(1, min(args.steps, 20))
    step_e2e()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        step_e2e()
    e2e_s = max_over_ranks(dist, time.perf_counter() - t0, dev)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    avg_launch_s = statistics.mean(per_launch_ms) / 1e3
    hbm_peak = float(peaks["hbm_gbs"])
    achieved = alg_bytes / avg_launch_s / 1e9
    roof = {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "peak_source": peak_src,
            "traffic": stored_traffic(w.name, kernel), "algorithmic_bytes_per_launch": alg_bytes,
            "algorithmic_tensor_flops_per_launch": 0, "avg_launch_ms": avg_launch_s * 1e3,
            "roofline_ms": alg_bytes / (hbm_peak * 1e9) * 1e3}
    if w.op == "bwd" and w.headdim <= 64 and w.dstate <= 128:
        # the chunk-form backward, whole call timed.  Its contractions run on the
        # tensor cores for bf16 with P = 64, N = 128 (the chunk states and the
        # gradient pass), else as fp32 FFMA: the roofline is that pipe.
        flops = bwd_chunk_flops(w)
        tf = flops / avg_launch_s / 1e12
        if w.dtype == "bf16" and w.headdim == 64 and w.dstate == 128:
            tc_peak = float(peaks["bf16_tflops"])
            roof = {"bound": "tensor", "kernel": "ssd_scan_bwd (whole call: ssd_bwd_tc_chain_kernel, "
                                                  "ssd_bwd_tc_grad_kernel, ssd_bwd_finish4_kernel)",
                    "achieved": tf, "peak": tc_peak, "unit": "TFLOP/s", "frac": tf / tc_peak,
                    "peak_source": peak_src + " (bf16 dense, burst)",
                    "traffic": stored_traffic(w.name, kernel), "contraction_flops_per_launch": flops,
                    "fp32_pipe_frac": tf / FP32_PEAK_TFLOPS,
                    "algorithmic_bytes_per_launch": alg_bytes, "hbm_frac": achieved / hbm_peak,
                    "avg_launch_ms": avg_launch_s * 1e3, "roofline_ms": flops / (tc_peak * 1e12) * 1e3,
                    "note": "latency-bound: neither the tensor pipe nor HBM is busy (see its profile)"}
        else:
            roof = {"bound": "alu", "kernel": "ssd_scan_bwd (whole call: ssd_bwd_local_kernel, ssd_bwd_pass_kernel, "
                                              "ssd_bwd_grad_kernel, ssd_bwd_finish4_kernel)",
                    "achieved": tf, "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s", "frac": tf / FP32_PEAK_TFLOPS,
                    "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz",
                    "traffic": stored_traffic(w.name, kernel), "fp32_flops_per_launch": flops,
                    "algorithmic_bytes_per_launch": alg_bytes, "hbm_frac": achieved / hbm_peak,
                    "avg_launch_ms": avg_launch_s * 1e3, "roofline_ms": flops / (FP32_PEAK_TFLOPS * 1e12) * 1e3}
    if w.op == "complex" and w.seqlen > 1 and not complex_takes_tc(w, args.path):
        # the state stays in registers over the sequence: fp32 arithmetic bounds it
        flops = complex_flops(w)
        tf = flops / avg_launch_s / 1e12
        roof = {"bound": "alu", "kernel": kernel, "achieved": tf, "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s",
                "frac": tf / FP32_PEAK_TFLOPS, "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz",
                "traffic": stored_traffic(w.name, kernel), "fp32_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": alg_bytes, "hbm_frac": achieved / hbm_peak,
                "avg_launch_ms": avg_launch_s * 1e3, "roofline_ms": flops / (FP32_PEAK_TFLOPS * 1e12) * 1e3}
    name = NEIGHBOR_NAMES[w.op]
    line = {
        "metric": f"{name} tokens·heads/s at 1 GB300; % of HBM roofline",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": workload_config(w, args.seed, flush),
        "roofline": roof,
        "e2e": {"value": world * th * e2e_steps / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in pin.values() if t is not None),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in back.values()),
                "steps": e2e_steps, "api": "the public call with pinned host copies in and out"},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if hasattr(step, "two_calls"):
        # the same work as two library calls (conv, then scan), timed the same way
        for _ in range(3):
            step.two_calls(stream)
        torch.cuda.synchronize(dev)
        t_ms, _, _, _ = timed_region(ssd, lambda: step.two_calls(stream), args.steps, stream, dev, None, local,
                                     flush)
        line["two_call_chain"] = {"ms_per_step": t_ms / args.steps,
                                  "value": th * args.steps / (t_ms / 1e3),
                                  "calls": "ssd_conv1d_silu_fwd, then ssd_scan_fwd (x, B, C through device memory)"}
    if not args.no_cpu_baseline and world == 1:
        v, sample = neighbor_oracle_rate(w, ref, 10.0, min_seconds=10.0)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)


def run_reference_neighbor(args, w: Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    _, _, _, _, nbytes, _, ref = neighbor_setup(w, torch.device("cpu"), args.seed)
    per_step = min(10.0, max(0.02, 120.0 / (args.steps + args.warmup)))
    for _ in range(args.warmup):
        neighbor_oracle_rate(w, ref, per_step)
    secs, th_total, sample = 0.0, 0, ""
    for _ in range(args.steps):
        v, sample = neighbor_oracle_rate(w, ref, per_step)
        th = int(sample.split("(")[1].split(" ")[0])
        secs += th / v
        th_total += th
    value = th_total / secs
    name = NEIGHBOR_NAMES[w.op]
    line = {
        "impl": "reference", "metric": f"{name} tokens·heads/s at 1 GB300; % of HBM roofline",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.seed, flushes_l2(nbytes)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": "per step: " + sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="libssd", choices=["libssd", "reference"])
    ap.add_argument("--path", default="auto", choices=["auto", "chunked", "sequential", "decode"])
    ap.add_argument("--schedule", default="auto", choices=["auto", "ranges", "pieces", "split"],
                    help="the chunked path's schedule (the forward scan workloads)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    w = WORKLOADS[args.workload]
    if w.op == "trap":
        (run_reference_trap if args.impl == "reference" else run_gpu_trap)(args, w)
    elif w.op in ("conv", "conv_scan", "gnorm", "bwd", "complex"):
        (run_reference_neighbor if args.impl == "reference" else run_gpu_neighbor)(args, w)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
