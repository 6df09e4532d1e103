#!/usr/bin/env python
"""Benchmark of the canvas sampler step on GB300.

One step = one pass of the whole per-step hot path over one batch of synthetic canvases:
logits GEMM, softmax statistics, exp(y - m) split + Gumbel-max, self-conditioning GEMM, the
reduction of s, the sampled tokens and confidences, and the lock / re-noise / stop update.
The default workload is one B=1 canvas of 256 positions over a 262,144-token vocabulary at
d = 2816 (the shapes of the DiffusionGemma pages; synthetic data).

    python bench.py [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line. Under torchrun every rank runs its own canvas on its own GPU (weak
scaling, no data-path collective); the timed region is bracketed by barriers and the slowest
rank's time is reported.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from canvas_sampler_gb300 import workloads as W  # noqa: E402

METRIC = "canvas sampler steps/s & TFLOP/s (B=1, 256×262144 vocab) vs roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_FILES = {
    "vocab_pass": os.path.join(ROOT, "profiles", "vocab_pass_tc_step_v262144_d2816.md"),
    "selfcond": os.path.join(ROOT, "profiles", "selfcond_tc_step_v262144_d2816.md"),
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.BENCH_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--kernel-impl", default="auto", choices=["auto", "tensor", "simt", "fused"])
    ap.add_argument("--vocab", type=int, default=None, help="override V (profiling runs)")
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling runs)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--sustained-seconds", type=float, default=3.0,
                    help="length of the power-capped sustained pass (0: none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--loop", action="store_true",
                    help="time the whole denoising loop (ds_denoise_loop) of the workload, as a "
                         "CUDA graph and as plain launches, instead of one step")
    ap.add_argument("--cpu-positions", type=int, default=256,
                    help="canvas positions in the oracle's timed sample (256: one full step)")
    return ap.parse_args()


# ------------------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(seed: int, rank: int) -> int:
    """Each rank samples its own canvas: the sampler seed is offset by the rank."""
    return int(seed) + int(rank)


def reduce_max(value: float, dist, device) -> float:
    """The slowest rank's value (the job's time); a no-op for a single process."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock / throttle reasons, each stamped with the host time at which
    it arrived, so that the samples that fall inside a timed region can be told apart."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []  # (host time, csv line)
        self.first = threading.Event()

    def start(self, wait_s: float = 3.0):
        """Start sampling; returns once the first sample has arrived (or after wait_s)."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "-i", str(self.gpu),
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            self.first.wait(wait_s)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))
            self.first.set()

    @staticmethod
    def summarise(lines):
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": max(mx),
               "reasons": sorted(reasons), "samples": len(sm)}
        if pw:
            out["power_w"] = statistics.median(pw)
        return out

    def stop(self, window=None):
        """Summary of the samples; with window = (t0, t1) (host times), of those that arrived
        inside it (the window's own summary under "region", all samples otherwise)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        if window is None:
            return self.summarise(self.lines)
        t0, t1 = window
        inside = [x for x in self.lines if t0 <= x[0] <= t1]
        out = self.summarise(inside) or self.summarise(self.lines)
        if out is not None:
            out["interval_ms"] = self.interval_ms
            out["in_region"] = bool(inside)
        return out


class NvmlClockSampler:
    """SM clock, power and clock-event reasons polled through the driver's NVML library
    (libnvidia-ml, read-only queries) every millisecond on a thread, so that a timed region of a
    few milliseconds still has samples of its own; the same summary as ClockSampler."""
    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index: int, interval_ms: float = 1.0):
        import ctypes
        self.gpu, self.interval_ms = gpu_index, interval_ms
        self.samples = []  # (host time, sm MHz, max MHz, power W, reasons bitmask)
        self._stop = threading.Event()
        self.ok = False
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(self.h)):
                return
            self.lib, self.ct = lib, ctypes
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_uint(1), ctypes.byref(mx))
            self.max_mhz = float(mx.value)
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _poll(self):
        ct, lib = self.ct, self.lib
        clk, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            lib.nvmlDeviceGetClockInfo(self.h, ct.c_uint(1), ct.byref(clk))  # NVML_CLOCK_SM
            lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
            self.reason_fn(self.h, ct.byref(rs))
            self.samples.append((time.time(), float(clk.value), self.max_mhz,
                                 pw.value / 1000.0, int(rs.value)))
            time.sleep(self.interval_ms / 1e3)

    def start(self):
        if not self.ok:
            return
        self.t = threading.Thread(target=self._poll, daemon=True)
        self.t.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 2.0:
            time.sleep(0.001)

    def stop(self, window=None):
        if not self.ok:
            return None
        self._stop.set()
        self.t.join(timeout=2)
        sel = self.samples
        if window is not None:
            inside = [x for x in self.samples if window[0] <= x[0] <= window[1]]
            sel = inside or self.samples
        if not sel:
            return None
        reasons = sorted({n for x in sel for bit, n in self.REASONS.items() if x[4] & bit})
        out = {"sm_mhz": statistics.median(x[1] for x in sel),
               "sm_min_mhz": min(x[1] for x in sel), "sm_max_mhz": self.max_mhz,
               "reasons": reasons, "samples": len(sel),
               "power_w": statistics.median(x[3] for x in sel), "source": "nvml",
               "interval_ms": self.interval_ms}
        if window is not None:
            out["in_region"] = bool([x for x in self.samples if window[0] <= x[0] <= window[1]])
        return out


def clock_sampler(gpu_index: int):
    """NVML polling when the driver's library loads, else nvidia-smi sampling."""
    s = NvmlClockSampler(gpu_index)
    return s if s.ok else ClockSampler(gpu_index)


# the files each tensor-core kernel is compiled from (its own file first)
KERNEL_SOURCES = {
    k: [os.path.join(ROOT, "canvas_sampler_gb300", "csrc", f) for f in files]
    for k, files in (
        ("vocab_pass", ("ds_tc_fused.cu", "ds_tc_common.cuh", "ds_internal.h", "ds_common.cuh")),
        ("selfcond", ("ds_tc_selfcond.cu", "ds_sample.cuh", "ds_tc_common.cuh", "ds_internal.h",
                      "ds_common.cuh")))}


def kernel_source_hash(kernel: str = "vocab_pass") -> str:
    """sha256 over a tensor-core kernel's sources (the files it is compiled from)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(f, "rb").read())
    return h.hexdigest()


def measured_traffic(kernel: str):
    """DRAM bytes per launch of a kernel from its committed ncu summary, if the kernel's
    sources have not changed since the capture (else None)."""
    if kernel not in PROFILE_FILES:
        return None
    try:
        text = open(PROFILE_FILES[kernel]).read()
    except OSError:
        return None
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    if not (m_b and m_h):
        return None
    return float(m_b.group(1)) if kernel_source_hash(kernel) == m_h.group(1) else None


def region_peak_key(region_s: float, peaks: dict, clocks: dict | None = None) -> str:
    """The bf16 peak a timed region is held to: the burst figure for a region shorter than a
    second that ran at full clocks (its own clock samples, where there are any, at >= 97% of the
    maximum SM clock with no power cap), else the sustained one (the power controller has
    lowered the clocks, as it does within a fraction of a second of back-to-back steps)."""
    burst = region_s < 1.0
    if burst and clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        burst = (clocks["sm_mhz"] >= 0.97 * clocks["sm_max_mhz"] and
                 "sw_power_cap" not in clocks.get("reasons", []))
    key = "bf16_tflops" if burst else "bf16_tflops_sustained"
    return key if key in peaks else "bf16_tflops"


def algorithmic_flops(w: W.Workload) -> float:
    return 4.0 * w.B * w.L * w.V * w.d


# ------------------------------------------------------------------------------ oracle timing

def oracle_sample_seconds(w, inp, E64, positions, reps=1):
    import oracle
    H64 = oracle.bf16_bits_to_f64(inp["H"]) if w.dtype == "bf16" else inp["H"].astype(np.float64)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.sampler_step(H64, E64, inp["T"], inp["tau"], inp["canvas"], inp["lock"], inp["step"],
                            inp["done"], inp["seed"], top_k=w.top_k, max_steps=w.max_steps,
                            positions=positions)
    return (time.perf_counter() - t0) / reps


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def workload_of(args) -> W.Workload:
    w = W.WORKLOADS[args.workload]
    if args.vocab or args.batch:
        w = W.scaled(w, V=args.vocab or w.V, B=args.batch or w.B)
    return w


def run_reference(args):
    """The reference arm: the fp64 oracle (the pages ship no code), timed as it stands on the
    host's cores over whole steps of the workload (every canvas position, full vocabulary), one
    oracle step per bench step, so that the printed value is what a whole step costs."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = workload_of(args)
    inp = W.make_inputs(w)
    import oracle
    E64 = oracle.bf16_bits_to_f64(inp["E"]) if w.dtype == "bf16" else inp["E"].astype(np.float64)
    pos = np.arange(w.L)
    for _ in range(args.warmup):
        oracle_sample_seconds(w, inp, E64, pos)
    t = [oracle_sample_seconds(w, inp, E64, pos) for _ in range(args.steps)]
    sec_per_step = float(np.mean(t))
    value = 1.0 / sec_per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec_per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "V": w.V, "d": w.d,
                   "impl": "oracle", "parallelism": "single",
                   "l2": "host memory (no GPU)", "state_reset": "every step from the same state"},
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"each step: one whole fp64 oracle step over all {w.L} canvas "
                                   f"positions x {w.B} sequence(s), full vocabulary"},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "tflops": algorithmic_flops(w) / sec_per_step / 1e12,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ our arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    from canvas_sampler_gb300.sampler import CanvasState, Sampler, StepOutputs

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload_of(args)
    inp = W.make_inputs(w)
    seed = rank_seed(inp["seed"], rank)

    def upload(a):
        if w.dtype == "fp32":
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    E = upload(inp["E"])
    H = upload(inp["H"]) if inp["H"] is not None else None
    if H is None:  # stand-in workloads: time the step on the first stand-in hidden state
        raise SystemExit("bench times fixed-H workloads; stand-in loops are covered by the tests")
    T = torch.from_numpy(inp["T"]).to(dev)
    tau = torch.from_numpy(inp["tau"]).to(dev)
    sampler = Sampler(w.V, w.d, canvas_len=w.L, max_batch=w.B, dtype=w.dtype, top_k=w.top_k,
                      max_steps=w.max_steps, impl=args.kernel_impl)
    B, L = w.B, w.L
    # state in one byte buffer so that one copy resets it before every step (every sequence
    # stays active, so every step does the full work)
    nb = B * L * 4 + B * 4 + B * L + B
    pristine = torch.zeros(nb, dtype=torch.uint8, device=dev)
    buf = torch.zeros(nb, dtype=torch.uint8, device=dev)

    def views(t):
        o = 0
        cv = t[o:o + B * L * 4].view(torch.int32).view(B, L); o += B * L * 4
        st = t[o:o + B * 4].view(torch.int32); o += B * 4
        lk = t[o:o + B * L].view(B, L); o += B * L
        dn = t[o:o + B]
        return CanvasState(cv, lk, st, dn)

    p = views(pristine)
    p.canvas.copy_(torch.from_numpy(inp["canvas"]))
    state = views(buf)
    out = StepOutputs.empty(B, L, w.d, device=dev)
    stream = torch.cuda.current_stream()

    def one_step():
        buf.copy_(pristine)
        sampler.step(H, E, T, tau, state, seed, out=out, stream=stream)

    for _ in range(max(3, args.warmup)):
        one_step()
    torch.cuda.synchronize()
    assert sampler.device_status() == 0
    if world > 1:
        dist.barrier()
    clocks = clock_sampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else
                           int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    clocks.start()  # returns at its first sample: the timed region starts right after
    launches0 = sampler.launch_count
    # coarse phase events inside the timed region (ends of the logits, up-to-self-conditioning,
    # self-conditioning and final phases): enough for both GEMMs' live durations, with fewer
    # events between the step's kernels
    sampler.set_phase_timing(True, coarse=True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_region0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        one_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_region1 = time.time()
    if world > 1:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    phases, nsteps = sampler.phase_times()
    sampler.set_phase_timing(False)
    launches = sampler.launch_count - launches0
    # samples that arrived while the timed steps ran (the region's own clock record; a region
    # shorter than the sampling interval has none, and then every sample is summarised)
    clk = clocks.stop(window=(t_region0, t_region1))
    # every phase, on a short untimed pass after the timed region (informational breakdown)
    sampler.set_phase_timing(True)
    for _ in range(min(args.steps, 20)):
        one_step()
    breakdown, nbd = sampler.phase_times()
    sampler.set_phase_timing(False)
    ms = reduce_max(ms, dist if world > 1 else None, dev)
    status = sampler.device_status()

    # end to end through the public API: pinned host buffers in, results back, every step
    hs = CanvasState(torch.from_numpy(inp["canvas"].copy()).pin_memory(),
                     torch.zeros(B, L, dtype=torch.uint8).pin_memory(),
                     torch.zeros(B, dtype=torch.int32).pin_memory(),
                     torch.zeros(B, dtype=torch.uint8).pin_memory())
    hout = StepOutputs.empty(B, L, w.d, pin=True)
    Hh = H.cpu().pin_memory()
    Th, tauh = T.cpu().pin_memory(), tau.cpu().pin_memory()
    h2d = Hh.numel() * Hh.element_size() + 2 * B * 4 + hs.canvas.numel() * 4 + B * L + B * 4 + B
    d2h = sum(t.numel() * t.element_size() for t in vars(hout).values()) + B * L * 4 + B * L + B * 4 + B
    for _ in range(2):
        sampler.step_host(Hh, E, Th, tauh, hs, seed, hout, stream=stream)
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        hs.lock.zero_(); hs.done.zero_(); hs.step.zero_()
        sampler.step_host(Hh, E, Th, tauh, hs, seed, hout, stream=stream)
    e2e_s = time.perf_counter() - t0
    e2e_s = reduce_max(e2e_s, dist if world > 1 else None, dev)

    step_s = ms / 1e3 / args.steps
    value = world * args.steps / (ms / 1e3)
    flops = algorithmic_flops(w)
    peaks, peak_src = load_peaks()
    # dominant kernel: the fused vocabulary pass (logits and self-conditioning GEMMs, 4 B L V d
    # algorithmic FLOP per launch; the phase named "logits" spans it, the convert and selfcond
    # phases are empty), or on the unfused path the self-conditioning GEMM (2 B L V d). The bf16
    # hi/lo doubling of the self-conditioning tensor work is not algorithmic.
    fused = sampler.impl == "fused"
    dom = max(phases, key=phases.get) if nsteps else "selfcond"
    dom_ms = phases.get(dom, 0.0) / max(1, nsteps)
    if fused and dom == "logits":
        dom, dom_flops = "vocab_pass", 4.0 * w.B * w.L * w.V * w.d
    else:
        dom_flops = {"logits": 2.0 * w.B * w.L * w.V * w.d,
                     "selfcond": 2.0 * w.B * w.L * w.V * w.d}.get(dom)
    # the timed region lasts well under a second at full clocks (the power controller has not
    # yet lowered them): its kernels are measured against the burst bf16 peak; only a region
    # of a second or more, or the sustained pass below, is held to the sustained peak
    region_s = ms / 1e3
    peak_key = region_peak_key(region_s, peaks, clk)
    peak_tf = float(peaks.get(peak_key, FALLBACK_PEAKS[peak_key]))
    roof = None
    if dom_flops and dom_ms > 0:
        ach = dom_flops / (dom_ms / 1e3) / 1e12
        traffic = measured_traffic(dom)
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak_tf,
                "unit": "TFLOP/s", "frac": ach / peak_tf, "traffic": traffic,
                "peak_source": f"{peak_key} ({peak_src})"}
        if dom == "selfcond":
            # the bf16 hi + lo split doubles the GEMM's tensor work: the fraction of the peak the
            # tensor cores actually run at (the algorithmic frac is capped at 1/2)
            roof["frac_cap"] = 0.5
            roof["tensor_work_frac"] = 2.0 * ach / peak_tf
        # the tensor-core step without top-k launches 4 kernels when the row merge and the race
        # run inside the self-conditioning launch (logits, self-conditioning, finalize, lock),
        # 6 when they have launches of their own
        if dom == "selfcond" and sampler.impl == "tensor" and launches == 4 * args.steps:
            roof["note"] = ("the launch also runs the step's Gumbel-max race on warps of its own; "
                            "only the GEMM's 2 B L V d FLOP are counted")
    # the vocabulary pass (both GEMMs with the epilogues fused into them: the logits and
    # self-conditioning phases, or the fused kernel) against the tensor roofline of its
    # 4 B L V d algorithmic FLOP; the bf16 hi/lo split makes its tensor work 6 B L V d, so no
    # schedule exceeds 2/3 of it
    vp_ms = (phases.get("logits", 0.0) + phases.get("selfcond", 0.0)) / max(1, nsteps)
    vp = None
    if vp_ms > 0:
        vp_ach = 4.0 * w.B * w.L * w.V * w.d / (vp_ms / 1e3) / 1e12
        vp = {"bound": "tensor", "ms": vp_ms, "achieved": vp_ach, "peak": peak_tf,
              "unit": "TFLOP/s", "frac": vp_ach / peak_tf, "frac_cap": 2.0 / 3.0}
    # sustained (last, so that the passes above run on a GPU that has not been throttled):
    # seconds of back-to-back steps, long enough for the power controller to settle (the timed
    # region above is a fraction of a second at full clocks)
    sustained = None
    if args.sustained_seconds > 0:
        n_sus = max(1, int(args.sustained_seconds * 1e3 / max(ms / args.steps, 1e-3)))
        sclk = clock_sampler(clocks.gpu)
        sclk.start()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        for _ in range(n_sus):
            one_step()
        s1.record(stream)
        torch.cuda.synchronize()
        sus_ms = reduce_max(s0.elapsed_time(s1), dist if world > 1 else None, dev)
        sclk_sum = sclk.stop()
        sus_step_ms = sus_ms / n_sus
        sus_peak = float(peaks.get("bf16_tflops_sustained",
                                   FALLBACK_PEAKS["bf16_tflops_sustained"]))
        sus_tf = flops / (sus_step_ms / 1e3) / 1e12
        sustained = {"value": world * n_sus / (sus_ms / 1e3), "unit": "steps/s", "steps": n_sus,
                     "ms_per_step": sus_step_ms, "clocks": sclk_sum,
                     "step_roofline": {"achieved": sus_tf, "peak": sus_peak, "unit": "TFLOP/s",
                                       "frac": sus_tf / sus_peak,
                                       "peak_source": f"bf16_tflops_sustained ({peak_src})"}}
        if sclk_sum and sclk_sum.get("sm_mhz"):
            # step time x median SM clock: a clock-independent cost of the step (ms x MHz),
            # comparable with the timed region's at its own clock
            sustained["ms_x_mhz"] = sus_step_ms * sclk_sum["sm_mhz"]
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "V": w.V, "d": w.d,
                   "impl": sampler.impl, "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "inputs larger than L2 (E is %.2f GB); no flush" % (w.V * w.d * 2 / 1e9),
                   "state_reset": "one device copy of the 2 KB canvas state before each step"},
        "tflops": world * flops / step_s / 1e12,
        "step_roofline": {"bound": "tensor", "achieved": flops / step_s / 1e12, "peak": peak_tf,
                          "unit": "TFLOP/s", "frac": flops / step_s / 1e12 / peak_tf,
                          "note": "4 B L V d algorithmic FLOP per step over the whole step, "
                                  f"against {peak_key}"},
        "roofline": roof,
        "vocab_pass_roofline": vp,
        "phase_ms_per_step": {k: v / max(1, nsteps) for k, v in phases.items()},
        "phase_breakdown_ms_per_step": {k: v / max(1, nbd) for k, v in breakdown.items()},
        "gpu_launches": launches,
        "e2e": {"value": world * args.e2e_steps / e2e_s, "unit": "steps/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "clocks": clk,
        "timed_region_s": region_s,
        "ms_x_mhz": (step_s * 1e3 * clk["sm_mhz"]) if clk and clk.get("sm_mhz") else None,
        "sustained": sustained,
        "device_status": status,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        E64 = oracle.bf16_bits_to_f64(inp["E"]) if w.dtype == "bf16" else inp["E"].astype(np.float64)
        n = max(1, min(w.L, args.cpu_positions))
        pos = np.arange(n)
        sec = oracle_sample_seconds(w, inp, E64, pos)
        sec_step = sec * (w.L / n) * w.B
        line["cpu_baseline"] = {
            "value": 1.0 / sec_step, "unit": "steps/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": (f"fp64 oracle over {n} of {w.L} canvas positions (full vocabulary), "
                       f"{sec:.1f} s" + (": one whole step" if w.L / n * w.B == 1 else
                                         f", scaled by {w.L / n * w.B:g} to one step"))}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_loop(args):
    """The workload's whole denoising loop through ds_denoise_loop (fixed H, or the stand-in
    hidden states for stand-in workloads): device time per loop and per iteration, as one CUDA
    graph with a device-side stop condition and as plain launches. One JSON line."""
    import torch

    from canvas_sampler_gb300.sampler import CanvasState, Sampler, StepOutputs

    dev = torch.device("cuda", 0)
    w = workload_of(args)
    inp = W.make_inputs(w)

    def upload(a):
        if w.dtype == "fp32":
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    E = upload(inp["E"])
    T = torch.from_numpy(inp["T"]).to(dev)
    tau = torch.from_numpy(inp["tau"]).to(dev)
    standin = w.h_mode == "standin"
    H = None if standin else upload(inp["H"])
    Wt = upload(inp["W"]) if standin else None
    sampler = Sampler(w.V, w.d, canvas_len=w.L, max_batch=w.B, dtype=w.dtype, top_k=w.top_k,
                      max_steps=w.max_steps, impl=args.kernel_impl)
    B, L = w.B, w.L
    state = CanvasState.from_numpy(inp["canvas"], inp["lock"], inp["step"], inp["done"],
                                   device=dev)
    init = CanvasState.from_numpy(inp["canvas"], inp["lock"], inp["step"], inp["done"],
                                  device=dev)
    out = StepOutputs.empty(B, L, w.d, device=dev)
    H_buf = torch.zeros(B, L, w.d, dtype=torch.bfloat16, device=dev) if standin else None

    def one_loop(use_graph):
        for k in ("canvas", "lock", "step", "done"):
            getattr(state, k).copy_(getattr(init, k))
        out.s.zero_()  # the stand-in starts from s_prev = 0
        sampler.loop(E, T, tau, state, inp["seed"], out, H=H, W=Wt, H_buf=H_buf,
                     max_iters=w.max_steps, use_graph=use_graph)

    res = {}
    for use_graph in (True, False):
        for _ in range(max(1, args.warmup)):
            one_loop(use_graph)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = clock_sampler(0 if "CUDA_VISIBLE_DEVICES" not in os.environ else
                               int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0]))
        clocks.start()
        t0 = time.time()
        ev0.record()
        for _ in range(args.steps):
            one_loop(use_graph)
        ev1.record()
        torch.cuda.synchronize()
        t1 = time.time()
        clk = clocks.stop(window=(t0, t1))
        ms = ev0.elapsed_time(ev1) / args.steps
        iters = int(state.step.max().item())  # the loop runs until its last sequence is done
        res["graph" if use_graph else "plain"] = {
            "ms_per_loop": ms, "iterations": iters, "ms_per_iteration": ms / max(1, iters),
            "steps_per_s": iters / (ms / 1e3), "timed_region_s": t1 - t0, "clocks": clk}
    assert sampler.device_status() == 0
    line = {"mode": "loop", "workload": w.name, "B": B, "L": L, "V": w.V, "d": w.d,
            "top_k": w.top_k, "h_mode": w.h_mode, "max_steps": w.max_steps,
            "loops": args.steps, "warmup": args.warmup, "impl": sampler.impl,
            "note": "device time of one whole loop (state reset by device copies inside the "
                    "timed region), CUDA events on the launching stream", **res}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.loop:
        return run_loop(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
