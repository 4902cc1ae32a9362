#!/usr/bin/env python3
"""Throughput of the single-GPU MoE layer (router top-k -> Dispatch -> Linear-1 +
SwiGLU -> Linear-2 -> Combine) on synthetic seeded inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload large] [--also fine,skew,smallT]
    python bench.py --impl reference ...     # the CPU oracle, timed the same way

One step = one moe_forward over the whole batch of T tokens, inputs and weights
resident in HBM; L2 is flushed (256 MiB write) before every step, outside the
timed events.  The headline is the large layer (T=4096, H=7168, I=2048, E=256,
top-8); the fine-grained, skewed and 128-token workloads are timed in the same
process the same way and reported under "workloads".  "e2e" is the same metric through
moe_forward_host: K back-to-back calls on page-locked host x and y, their copies pipelined
beside the neighbouring steps' kernels, timed as one span up to the last y in host memory.
Rank 0 prints one JSON line.  With torchrun (N > 1) every rank
runs an independent replica on its own GPU (the layer is not sharded) and the
time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer TFLOP/s and tokens/s on 1 GB300; % of bf16 tensor/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


# idle time before each workload's warm-up and before its e2e steps: a latency-bound workload
# timed right after heavy work (input generation, a weight-streaming workload) ran at a
# power-limited SM clock, and the weight-streaming layer's steps slow as a run goes on
IDLE_BEFORE_S = 0.5


def load_traffic(kernel: str, workload: str, schedule: int):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu record, only while
    the kernel's sources are unchanged since the capture (else None), and a note saying how the
    figure was taken (a record may be a smaller case scaled to the full launch)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            recs = json.load(f)[kernel]
        if isinstance(recs, dict):
            recs = [recs]
        for rec in recs:
            if rec["workload"] != workload or rec["schedule"] != schedule:
                continue
            h = hashlib.sha256()
            for src in rec["sources"]:
                with open(os.path.join(ROOT, src), "rb") as f:
                    h.update(f.read())
            if h.hexdigest() != rec["source_sha256"]:
                return None, "sources changed since the capture"
            return float(rec["dram_bytes_per_launch"]), rec.get("note", "ncu capture of this workload")
        return None, "no capture of this workload"
    except Exception:
        return None, "no traffic record"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples with host timestamps."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"--loop-ms={period_ms}", "-i", str(index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        win = [s for t, s in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if len(win) < 3:   # short timed region: widen to the loaded period around it
            win = [s for t, s in self.samples if t0 - 2.0 <= t <= t1 + 0.5]
            note = "timed region shorter than the sampling period: samples from warm-up + timed steps"
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        mhz, mx, reasons = [], [], set()
        for s in win:
            try:
                mhz.append(float(s[0]))
                mx.append(float(s[1]))
            except ValueError:
                continue
            for n, v in zip(names, s[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(win), "note": note}


class NvmlSampler:
    """SM clock, power and clock-event reasons read through NVML (ctypes, read-only calls) every
    `period_ms` on a thread, with host timestamps; a timed region of a few tens of ms still gets
    samples.  Falls back to ClockSampler (nvidia-smi) when NVML cannot be loaded."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_ms: float = 5.0):
        import ctypes
        self.samples = []
        self.ok = False
        self.stop_flag = False
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
                return
        except Exception:
            return
        self.lib, self.h, self.period = lib, h, period_ms / 1e3
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
        self.ok = True
        self.th = threading.Thread(target=self._run, daemon=True)
        self.th.start()

    def _run(self):
        import ctypes
        mhz, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_r = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_flag:
            t = time.perf_counter()
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:   # NVML_CLOCK_SM
                p = float(pw.value) / 1e3 if self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw)) == 0 else None
                r = int(rs.value) if get_r(self.h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((t, float(mhz.value), p, r))
            time.sleep(self.period)

    def stop(self):
        self.stop_flag = True
        if self.ok:
            self.th.join(timeout=1.0)

    def summary(self, t0: float, t1: float):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "note": "no NVML sample inside the timed region"}
        reasons = sorted({n for s in win for bit, n in self.REASONS.items() if s[3] & bit})
        pw = [s[2] for s in win if s[2] is not None]
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(win), "power_w_max": max(pw) if pw else None,
                "note": f"NVML every {self.period * 1e3:.0f} ms inside the timed region"}


def clock_sampler(index: int):
    s = NvmlSampler(index)
    return s if s.ok else ClockSampler(index)


# ----------------------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, group_ready: bool) -> float:
    """Maximum of `value` over all ranks (identity without a process group)."""
    if not group_ready:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(group_ready: bool):
    if group_ready:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- oracle timing
def weight_source(wl, d=None):
    """Expert slices for the oracle: host copies of the device tensors the seeded generator drew
    (when the GPU holds them: a copy per expert, no host-side regeneration), else the host
    implementation of the same generator (bit-identical values)."""
    if d is not None:
        return lambda which, e: d[which][e].contiguous().view(__import__("torch").int16).cpu().numpy().view("uint16")
    return lambda which, e: synth.expert_slice_host(wl, which, e)


def oracle_sample(wl, n_tok: int, seed: int, weights_of):
    """The CPU oracle on n_tok sampled tokens (routing of the sample + their k experts each).
    Returns (seconds of the oracle's own arithmetic, useful FLOPs, threads, tokens, experts);
    fetching the expert weights is not timed."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    tok = np.sort(rng.choice(wl.T, size=min(n_tok, wl.T), replace=False)).astype(np.int64)
    h = synth.host_inputs(wl, weights=False)
    x = np.ascontiguousarray(h["x"][tok])
    bias = h["bias"] if wl.zipf_s else None
    tm = {}
    r = oracle.forward(x, h["Wr"], bias, lambda e: weights_of("W1", e), lambda e: weights_of("W2", e), wl.k,
                       timing=tm)
    experts = len({int(e) for e in r["ids"].ravel()})
    flops = len(tok) * (2.0 * wl.H * wl.E + wl.k * 6.0 * wl.H * wl.I)
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return tm["compute_s"], flops, threads, len(tok), experts


def calibrate_tokens(wl, budget_s: float, weights_of):
    n0 = max(2, min(os.cpu_count() or 1, 16))
    dt, _, _, n, _ = oracle_sample(wl, n0, 0, weights_of)
    return max(2, min(int(budget_s / max(dt / n, 1e-9)), wl.T))


def cpu_baseline(wl, budget_s: float, weights_of):
    import oracle
    oracle.build()
    n = calibrate_tokens(wl, budget_s, weights_of)
    dt, flops, threads, n, ne = oracle_sample(wl, n, 2, weights_of)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {wl.T} tokens (router + their {wl.k} experts each, {ne} experts touched), "
                      f"{dt:.1f} s of oracle arithmetic; expert weights copied per expert from the seeded "
                      f"generator's tensors, untimed",
            "tokens_per_s": n / dt}


def run_reference(args, wl):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    d = None
    try:
        import torch
        if torch.cuda.is_available():        # the seeded generator draws the weights on the device:
            torch.cuda.set_device(0)         # the oracle only reads host copies of them
            d = synth.device_inputs(wl)
    except Exception:
        d = None
    weights_of = weight_source(wl, d)
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = calibrate_tokens(wl, min(budget, 8.0), weights_of)
    for _ in range(args.warmup):
        oracle_sample(wl, n, 3, weights_of)
    times, flops_tot, toks = 0.0, 0.0, 0
    threads = 1
    for i in range(args.steps):
        dt, fl, threads, nn, _ = oracle_sample(wl, n, 10 + i, weights_of)
        times += dt
        flops_tot += fl
        toks += nn
    value = flops_tot / times / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * times / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32-accumulate bf16",
            "data": "synthetic (seeded generator)",
            "config": config_of(wl, args), "note": "the CPU oracle on the host cores; no GPU work is timed",
            "tokens_per_s": toks / times,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step {n} of {wl.T} tokens (router + their experts); the oracle's "
                                       f"arithmetic timed, expert weights fetched untimed"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def config_of(wl, args, single=None):
    """The workload, the schedule options and the L2 policy of the GPU arm's timed steps: the
    same dict for both arms (the reference arm runs on the host and says so in "note").  single:
    the launch form of this entry (default: the --single-launch option)."""
    if single is None:
        single = getattr(args, "single_launch", False)
    sched = {0: "wave-serial", 1: "interleaved", 2: "phased (L1 launch, L2 launch)",
             3: "auto (wave-serial, one wave of all experts)"}[args.schedule]
    split = "streaming" if args.gemm_split == "auto" else args.gemm_split
    cfg = {"workload": f"{wl.name}: {wl.description}", "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
           "top_k": wl.k, "zipf_s": wl.zipf_s, "schedule": sched, "gemm_split": split,
           "wave_experts": args.wave_experts, "lead_waves": args.lead_waves,
           "launch": "single (MOE_FLAG_SINGLE_LAUNCH)" if single else "multi",
           "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write)",
           "parallelism": f"replicas x{args.gpus} (no sharding)"}
    if getattr(args, "exact_logits", False):
        cfg["router"] = "all logits canonical (MOE_FLAG_EXACT_LOGITS)"
    return cfg


# ----------------------------------------------------------------------------- GPU arm
def _events(n):
    import torch
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]


def measure(wl, d, args, dev, local, peaks, peak_src, group, ws, sampler, with_e2e=True, extra_flags=0):
    """One workload: W warm-up steps, K timed steps (CUDA events on the launching stream, L2
    flushed before each step outside the events), the host-buffer e2e steps, and the per-stage
    split from a second plan.  Returns the fields of its JSON entry."""
    import torch
    import mixture_experts_layer_top_gb300 as moe

    bias = synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None
    flags = {"auto": 0, "streaming": moe.MOE_FLAG_GEMM_STREAMING, "compute": moe.MOE_FLAG_GEMM_COMPUTE}[args.gemm_split]
    flags |= extra_flags
    if getattr(args, "exact_logits", False):
        flags |= moe.MOE_FLAG_EXACT_LOGITS
    single = bool(flags & moe.MOE_FLAG_SINGLE_LAUNCH)
    cfg = dict(schedule=args.schedule, wave_experts=args.wave_experts, lead_waves=args.lead_waves)
    layer = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, flags=flags, **cfg), local, router_bias=bias)
    logits = torch.empty((wl.T, wl.E), dtype=torch.float32, device=dev)
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    fwd = lambda: layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=logits, y=y)   # noqa: E731

    torch.cuda.synchronize()
    time.sleep(IDLE_BEFORE_S)                   # the power state the input generation left settles
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        fwd()
    layer.check()
    counts = layer.routing(wl.T)["counts"].cpu()
    touched = int((counts > 0).sum())
    launches = layer.launch_count()

    torch.cuda.synchronize()
    barrier(group)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ev = _events(args.steps)
    for i in range(args.steps):                # no host synchronisation inside the timed steps
        flush.zero_()
        ev[i][0].record()
        fwd()
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(group)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    layer.check()
    clocks = sampler.summary(t0, t1) if sampler else None
    ms_per_step = reduce_max(sum(a.elapsed_time(b) for a, b in ev), group) / args.steps

    # ---- e2e: back-to-back host-buffer C-ABI calls, every copy inside the timed region.
    # MOE_FLAG_HOST_PIPELINE: x_host is written once, on the host, before the steps; each step's
    # upload runs beside the previous step's GEMM and its y copy beside the next step, so the
    # region is one span from the first step's start to the last y landing in host memory
    # (moe_host_wait).  L2: the steps stream the expert weights, several times L2 on every
    # workload but the tiny one; that one is flushed between steps, the flushes' own time
    # (events around each) taken out of the span.
    e2e = None
    if with_e2e:
        layer_h = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, flags=flags | moe.MOE_FLAG_HOST_PIPELINE,
                                             **cfg), local, router_bias=bias)
        x_host = d["x"].cpu().pin_memory()
        y_host = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
        weight_bytes = 3 * wl.E * wl.H * wl.I * 2
        l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
        flush_steps = weight_bytes < 4 * l2_bytes   # weights not well beyond L2: flush between steps
        torch.cuda.synchronize()
        time.sleep(IDLE_BEFORE_S)               # the same idle start as the device-buffer steps
        for _ in range(2):
            layer_h.forward_host(x_host, d["Wr"], d["W1"], d["W2"], logits, y_host)
        layer_h.host_wait()
        flush.zero_()
        torch.cuda.synchronize()
        fev = _events(args.steps)
        span = _events(1)[0]
        span[0].record()
        for i in range(args.steps):
            if flush_steps and i:
                fev[i][0].record()
                flush.zero_()
                fev[i][1].record()
            layer_h.forward_host(x_host, d["Wr"], d["W1"], d["W2"], logits, y_host)
        layer_h.host_wait()
        span[1].record()
        torch.cuda.synchronize()
        layer_h.check()
        layer_h.close()
        if not torch.equal(y_host.view(torch.int16), y.cpu().view(torch.int16)):
            raise RuntimeError("host-buffer forward disagrees with the device-buffer forward")
        flush_ms = sum(fev[i][0].elapsed_time(fev[i][1]) for i in range(1, args.steps)) if flush_steps else 0.0
        e_ms = reduce_max(span[0].elapsed_time(span[1]) - flush_ms, group) / args.steps
        e2e = {"value": ws * wl.useful_flops() / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": wl.T * wl.H * 2, "d2h_bytes_per_step": wl.T * wl.H * 2,
               "ms_per_step": e_ms, "tokens_per_s": ws * wl.T / (e_ms * 1e-3),
               "host_pipeline": True,
               "timing": "one span over the back-to-back steps, first step's start to the last y in host memory",
               "overlap": ("each forward's upload and routing run beside the previous forward's last kernels, "
                           "its output copy beside the next forward; the first upload and the last copy are exposed"),
               "l2": (f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write), flush time taken out"
                      if flush_steps else
                      f"not flushed: the {weight_bytes / 2**30:.2f} GiB of expert weights exceed L2 "
                      f"({l2_bytes >> 20} MiB)")}
    layer.close()
    # ---- per-stage breakdown on a second plan whose library records events between stages
    # (those events serialise the stream, so the timed steps above run without them)
    layer_t = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, flags=flags | moe.MOE_FLAG_STAGE_TIMING,
                                         **cfg), local, router_bias=bias)
    stages = []
    for i in range(3 + min(args.steps, 20)):
        flush.zero_()
        layer_t.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=logits, y=y)
        if i >= 3:
            stages.append(layer_t.stage_times())
    layer_t.check()
    layer_t.close()
    del flush

    flops = wl.useful_flops()
    R = wl.T * wl.k
    w_bytes = 6.0 * wl.H * wl.I * touched
    layer_bytes = 2.0 * wl.T * wl.H * 2 + 2.0 * wl.H * wl.E + 4.0 * wl.T * wl.E + w_bytes
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = layer_bytes / (peaks["hbm_gbs"] * 1e9)
    t_step = ms_per_step * 1e-3
    stage_avg = {k: statistics.mean(s[k] for s in stages) for k in stages[0]}
    if single:
        # one kernel: the library's stage events bracket the counts memset and the whole layer
        stage_avg = {"memset_counts": stage_avg["router_topk"], "fused_layer": stage_avg["grouped_gemm"]}
        kernel, g_ms = "fused_layer_kernel", stage_avg["fused_layer"]
    else:
        # dominant kernel: the persistent grouped GEMM (Linear-1 + SwiGLU, Linear-2 + scale)
        kernel, g_ms = "grouped_gemm_kernel", stage_avg["grouped_gemm"]
    g_flops = 6.0 * wl.H * wl.I * R
    g_bytes = w_bytes                               # compulsory: each touched expert's weights once
    tensor_bound = g_flops / (peaks["bf16_tflops"] * 1e12) >= g_bytes / (peaks["hbm_gbs"] * 1e9)
    if tensor_bound:
        ach = g_flops / (g_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"]}
    else:
        ach = g_bytes / (g_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"]}
    traffic, traffic_note = load_traffic(kernel, wl.name, args.schedule)
    roof.update({"traffic": traffic, "traffic_unit": "bytes per launch (ncu dram read+write)",
                 "traffic_note": traffic_note,
                 "kernel": kernel, "ms_per_launch": g_ms,
                 "launches_per_step": 2 if (args.schedule == 2 and not single) else 1,
                 "peak_source": f"{peak_src} ({'bf16_tflops burst' if tensor_bound else 'hbm_gbs'})",
                 "algorithmic": (f"{g_flops:.4g} FLOP (6*H*I per routed row x {R} rows)" if tensor_bound
                                 else f"{g_bytes:.4g} B (6*H*I bytes per touched expert x {touched})")})
    nominal_tc, nominal_hbm = 2250.0, 7900.0
    return {
        "value": ws * flops / t_step / 1e12, "unit": "TFLOP/s", "ms_per_step": ms_per_step,
        "tokens_per_s": ws * wl.T / t_step,
        "config": config_of(wl, args, single),
        "layer_roofline": {"bound": "tensor" if t_tc >= t_hbm else "hbm", "frac": max(t_tc, t_hbm) / t_step,
                           "frac_of_nominal": max(flops / (nominal_tc * 1e12),
                                                  layer_bytes / (nominal_hbm * 1e9)) / t_step,
                           "t_tensor_us": t_tc * 1e6, "t_hbm_us": t_hbm * 1e6,
                           "compulsory_bytes": layer_bytes, "useful_flops": flops, "experts_touched": touched,
                           "peaks": "measured (MEASURED_PEAKS); frac_of_nominal against 2.25 PF/s bf16, 7.9 TB/s"},
        "roofline": roof,
        "stages_ms": stage_avg,
        "gpu_launches": launches * args.steps,
        "e2e": e2e,
        "clocks": clocks,
    }


def _shared_inputs(wl, have: dict, dev):
    """Device inputs of wl, reusing another workload's weight tensors when the shapes and seed
    match (the generator gives the same values for the same tensor id, index and seed)."""
    import torch
    key = (wl.H, wl.I, wl.E, wl.seed)
    if key in have:
        d = dict(have[key])
        d["x"] = synth.normal_bf16_torch(wl.T * wl.H, 1.0, synth.TID_X, wl.seed, device=dev).view(wl.T, wl.H)
        d["bias"] = torch.from_numpy(synth.zipf_bias(wl.E, wl.zipf_s)).to(dev)
        return d
    d = synth.device_inputs(wl, device=dev)
    if 6 * wl.H * wl.I * wl.E >= 1 << 30:
        have.clear()                             # keep one weight set of 1 GB or more resident at a time
    have[key] = d
    return d


def run_ours(args, wl):
    import torch
    import mixture_experts_layer_top_gb300 as moe

    ws, rank, local = dist_env()
    group = False
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        group = True
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.build()
    peaks, peak_src = load_peaks()
    sampler = None if args.no_clocks else clock_sampler(local)

    have = {}
    main_flags = moe.MOE_FLAG_SINGLE_LAUNCH if args.single_launch else 0
    main = measure(wl, _shared_inputs(wl, have, dev), args, dev, local, peaks, peak_src, group, ws, sampler,
                   with_e2e=not args.no_e2e, extra_flags=main_flags)
    # the other workloads: those with under 1 GB of expert weights first (latency-bound: timed
    # before a weight-streaming run leaves the GPU at its power limit, which lowered the SM clock
    # to ~1.56 GHz for the tiny layer's steps), then those sharing the resident weights' shape, so
    # that each weight set is drawn once (22.5 GB for the large shape)
    jobs = [(n, False) for n in args.also.split(",") if n and n != "none" and n != wl.name]
    jobs += [(n, True) for n in args.also_single.split(",") if n and n != "none"]
    shape = lambda n: (synth.WORKLOADS[n].H, synth.WORKLOADS[n].I, synth.WORKLOADS[n].E)   # noqa: E731
    small = lambda n: 6 * synth.WORKLOADS[n].H * synth.WORKLOADS[n].I * synth.WORKLOADS[n].E < 1 << 30   # noqa: E731
    jobs.sort(key=lambda j: (not small(j[0]), shape(j[0]) != (wl.H, wl.I, wl.E), shape(j[0])))
    extra = {}
    for name, single in jobs:
        w2 = synth.WORKLOADS[name]
        key = f"{name} (single launch)" if single else name
        extra[key] = measure(w2, _shared_inputs(w2, have, dev), args, dev, local, peaks, peak_src, group, ws, sampler,
                             with_e2e=(not args.no_e2e) and not single,
                             extra_flags=moe.MOE_FLAG_SINGLE_LAUNCH if single else main_flags)
        launches = extra[key].pop("gpu_launches")
        if single:
            extra[key]["launches_per_step"] = launches // args.steps
    have.clear()
    torch.cuda.empty_cache()
    if sampler:
        sampler.stop()

    if rank != 0:
        if group:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        try:
            cpu = cpu_baseline(wl, args.cpu_budget, weight_source(wl, _shared_inputs(wl, {}, dev)))
        except Exception as ex:  # reported, not fatal
            cpu = {"value": None, "error": str(ex)[:200]}

    line = {
        "metric": METRIC, "value": main["value"], "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded generator)",
        "config": main["config"],
        "tokens_per_s": main["tokens_per_s"],
        "layer_roofline": main["layer_roofline"],
        "roofline": main["roofline"],
        "stages_ms": main["stages_ms"],
        "gpu_launches": main["gpu_launches"],
        "e2e": main["e2e"],
        "cpu_baseline": cpu,
        "clocks": main["clocks"],
        "peaks": {**peaks, "source": peak_src},
        "workloads": extra,
    }
    print(json.dumps(line))
    if group:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- schedule sweep
SWEEP_SCHEDULES = [("auto", 3, 0, 1), ("wave-serial, waves fill the SMs", 0, 0, 1), ("wave-serial, 32 experts", 0, 32, 1),
                   ("interleaved lead 1", 1, 0, 1), ("interleaved lead 2", 1, 0, 2), ("interleaved lead 3", 1, 0, 3),
                   ("interleaved 32 experts lead 1", 1, 32, 1), ("phased", 2, 0, 1)]


def sweep_points():
    for s in (0.0, 0.6, 1.2, 2.0):
        for T in (512, 2048, 8192, 16384):
            yield synth.Workload(f"fine-shape T={T} zipf={s}", T, 2048, 768, 128, 8, zipf_s=s)
    for s in (0.0, 1.2):
        for T in (128, 1024, 4096):
            yield synth.Workload(f"large-shape T={T} zipf={s}", T, 7168, 2048, 256, 8, zipf_s=s)


def run_schedule_sweep(args):
    """Every tile schedule on every sweep point, in alternating rounds (same process, same
    inputs), with the L2 flushed before each step: one JSON line per (point, schedule) with the
    median step and grouped-GEMM times (CUDA events; the stage events of the library)."""
    import torch
    import mixture_experts_layer_top_gb300 as moe
    moe.build()
    torch.cuda.set_device(0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    have = {}
    for wl in sweep_points():
        d = _shared_inputs(wl, have, torch.device("cuda", 0))
        bias = synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None
        layers = {name: moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, schedule=sc, wave_experts=we,
                                                   lead_waves=lead, flags=moe.MOE_FLAG_STAGE_TIMING), 0,
                                     router_bias=bias)
                  for name, sc, we, lead in SWEEP_SCHEDULES}
        lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
        y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
        res = {n: ([], []) for n in layers}
        for layer in layers.values():
            for _ in range(3):
                layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=lg, y=y)
            layer.check()
        counts = layers["auto"].routing(wl.T)["counts"].cpu()
        for _ in range(3):
            for name, layer in layers.items():
                for _ in range(10):
                    flush.zero_()
                    a, b = _events(1)[0]
                    a.record()
                    layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=lg, y=y)
                    b.record()
                    b.synchronize()
                    res[name][0].append(a.elapsed_time(b))
                    res[name][1].append(layer.stage_times()["grouped_gemm"])
        for name, layer in layers.items():
            layer.check()
            layer.close()
            print(json.dumps({"point": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "zipf_s": wl.zipf_s,
                              "experts_touched": int((counts > 0).sum()), "max_rows": int(counts.max()),
                              "schedule": name, "step_ms": statistics.median(res[name][0]),
                              "gemm_ms": statistics.median(res[name][1])}), flush=True)
    return 0


# ----------------------------------------------------------------------------- grouped-GEMM wait trace
def run_gemm_trace(args, wl):
    """The grouped GEMM's per-role wait times on wl with the chosen schedule (MOE_FLAG_TRACE,
    moe_trace_read): per CTA the nanoseconds each role spent blocked - producer on a free stage,
    producer on Linear-1 readiness, MMA issuer on a free accumulator, MMA issuer on operands,
    epilogue on an accumulator - summed over the CTAs and divided by their summed lifetimes;
    median over `--steps` forwards after `--warmup`, L2 flushed before each, beside the GEMM
    launch time of a second plan (its stage events).  One JSON line."""
    import numpy as np
    import torch
    import mixture_experts_layer_top_gb300 as moe
    moe.build()
    torch.cuda.set_device(0)
    d = synth.device_inputs(wl, device="cuda")
    bias = synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    cfg = dict(schedule=args.schedule, wave_experts=args.wave_experts, lead_waves=args.lead_waves)
    traced = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, flags=moe.MOE_FLAG_TRACE, **cfg), 0,
                          router_bias=bias)
    timed = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, flags=moe.MOE_FLAG_STAGE_TIMING, **cfg), 0,
                         router_bias=bias)
    lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    fracs, gemm = [], []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        traced.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=lg, y=y)
        tr = moe.moe_trace_read(traced.plan)[:-1].astype(np.float64)   # the last row: single-launch stamps
        live = tr[:, 5] > 0
        flush.zero_()
        timed.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=lg, y=y)
        g = timed.stage_times()["grouped_gemm"]
        if i >= args.warmup:
            fracs.append(tr[live, :5].sum(axis=0) / tr[live, 5].sum())
            gemm.append(g)
    traced.check()
    timed.check()
    traced.close()
    timed.close()
    med = np.median(np.array(fracs), axis=0)
    names = ("producer_free_stage", "producer_l1_readiness", "mma_free_accumulator", "mma_operands",
             "epilogue_accumulator")
    print(json.dumps({"workload": f"{wl.name}: {wl.description}", "schedule": config_of(wl, args)["schedule"],
                      "forwards": args.steps, "gemm_ms": round(statistics.median(gemm), 4),
                      "wait_fraction_of_cta_lifetime": {n: round(float(v), 3) for n, v in zip(names, med)},
                      "note": "a wait is clocked from its first failed barrier probe: waits that end inside "
                              "that probe are not counted"}), flush=True)
    return 0


# ----------------------------------------------------------------------------- single-launch phases
PHASE_NAMES = ("router_logits", "topk", "dispatch", "gather", "grouped_gemm", "combine")


def run_phase_trace(args, wl):
    """The single-launch layer (MOE_FLAG_SINGLE_LAUNCH with MOE_FLAG_TRACE) on wl: the time of
    each phase inside the launch from the kernel's own %globaltimer stamps at the phase boundaries
    (CTA 0; the last row of moe_trace_read), beside the multi-launch path's stage times (CUDA
    events between the stages); `--steps` forwards of each after `--warmup`, alternating, L2
    flushed before each; medians.  One JSON line."""
    import numpy as np
    import torch
    import mixture_experts_layer_top_gb300 as moe
    moe.build()
    torch.cuda.set_device(0)
    d = synth.device_inputs(wl, device="cuda")
    bias = synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    single = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k,
                                        flags=moe.MOE_FLAG_SINGLE_LAUNCH | moe.MOE_FLAG_TRACE), 0, router_bias=bias)
    multi = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, flags=moe.MOE_FLAG_STAGE_TIMING), 0,
                         router_bias=bias)
    lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    phases, stages = [], []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        single.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=lg, y=y)
        stamps = moe.moe_trace_read(single.plan)[-1][:len(PHASE_NAMES) + 1].astype(np.int64)
        flush.zero_()
        multi.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=lg, y=y)
        st = multi.stage_times()
        if i >= args.warmup:
            phases.append(np.diff(stamps) / 1e3)
            stages.append(st)
    single.check()
    multi.check()
    single.close()
    multi.close()
    ph = np.median(np.array(phases), axis=0)
    print(json.dumps({"workload": f"{wl.name}: {wl.description}", "forwards": args.steps,
                      "single_launch_phases_us": {n: round(float(v), 2) for n, v in zip(PHASE_NAMES, ph)},
                      "single_launch_total_us": round(float(ph.sum()), 2),
                      "multi_launch_stages_us": {n: round(1e3 * statistics.median(s[n] for s in stages), 2)
                                                 for n in stages[0]},
                      "note": "phases: %globaltimer stamps of CTA 0 inside the one launch; stages: CUDA events "
                              "between the multi-launch path's kernels (they serialise its launches)"}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)   # >= 0.2 s timed, several 50 ms clock samples
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default="large",
                    help="the workload of the headline line (default: the large layer)")
    ap.add_argument("--also-single", default="tiny,smallT",
                    help="comma-separated workloads also timed with the whole layer in one launch "
                         "(MOE_FLAG_SINGLE_LAUNCH), reported under 'workloads' as '<name> (single launch)'")
    ap.add_argument("--also", default="fine,skew,smallT,tiny",
                    help="comma-separated workloads also timed in the same run, reported under 'workloads' "
                         "('none': only the headline workload)")
    ap.add_argument("--shape", default="",
                    help="T,H,I,E,k[,zipf_s]: a custom workload (same laws and seed) instead of --workload, "
                         "e.g. a cut-down case for a profiler capture")
    ap.add_argument("--schedule", type=int, choices=(0, 1, 2, 3), default=3,
                    help="0 wave-serial, 1 interleaved, 2 phased, 3 auto (the library's choice)")
    ap.add_argument("--wave-experts", type=int, default=0, help="experts per wave (0: fill the SMs)")
    ap.add_argument("--lead-waves", type=int, default=1, help="interleave lead D (interleaved schedule)")
    ap.add_argument("--gemm-split", choices=("auto", "streaming", "compute"), default="auto",
                    help="shared-memory split of the grouped GEMM (auto: the library default, streaming)")
    ap.add_argument("--single-launch", action="store_true",
                    help="run the headline (and --also) workloads with the whole layer in one launch")
    ap.add_argument("--schedule-sweep", action="store_true",
                    help="time every tile schedule over a sweep of routing skew and token counts (JSON lines)")
    ap.add_argument("--exact-logits", action="store_true",
                    help="every router logit in the canonical order on the CUDA cores (MOE_FLAG_EXACT_LOGITS)")
    ap.add_argument("--gemm-trace", action="store_true",
                    help="per-role wait times of the grouped GEMM on --workload with --schedule (one JSON line)")
    ap.add_argument("--phase-trace", action="store_true",
                    help="time the phases inside the single-launch layer on --workload (one JSON line)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=16.0, help="seconds of oracle work for cpu_baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    wl = synth.WORKLOADS[args.workload]
    if args.shape:
        v = args.shape.split(",")
        T, H, I, E, k = (int(a) for a in v[:5])
        z = float(v[5]) if len(v) > 5 else 0.0
        wl = synth.Workload(f"custom-{T}x{H}x{I}x{E}x{k}" + (f"-z{z}" if z else ""), T, H, I, E, k, zipf_s=z,
                            description=f"custom T={T} H={H} I={I} E={E} top-{k}" + (f" Zipf({z})" if z else ""))
    if args.schedule_sweep:
        return run_schedule_sweep(args)
    if args.phase_trace:
        return run_phase_trace(args, wl)
    if args.gemm_trace:
        return run_gemm_trace(args, wl)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
