#!/usr/bin/env python3
"""Throughput of the single-GPU MoE layer (router top-k -> Dispatch -> Linear-1 +
SwiGLU -> Linear-2 -> Combine) on synthetic seeded inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload fine] [--schedule 3]
    python bench.py --impl reference ...     # the CPU oracle, timed the same way

One step = one moe_forward over the whole batch of T tokens, inputs and weights
resident in HBM; L2 is flushed (256 MiB write) before every step, outside the
timed events.  Rank 0 prints one JSON line.  With torchrun (N > 1) every rank
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


def load_traffic(kernel: str, workload: str, schedule: int):
    """DRAM bytes per launch of `kernel` from the committed ncu record, only while the
    kernel's sources are unchanged since the capture (else None)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        if rec["workload"] != workload or rec["schedule"] != schedule:
            return None
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        return float(rec["dram_bytes_per_launch"]) if h.hexdigest() == rec["source_sha256"] else None
    except Exception:
        return None


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
_WCACHE = {}


def _expert(wl, which, e):
    key = (wl.name, which, e)
    if key not in _WCACHE:
        _WCACHE[key] = synth.expert_slice_host(wl, which, e)
    return _WCACHE[key]


def oracle_sample(wl, n_tok: int, seed: int = 1):
    """Time the CPU oracle on n_tok sampled tokens (routing of the sample + their k experts).
    Returns (seconds, useful FLOPs, threads).  Weight generation is not timed."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    tok = np.sort(rng.choice(wl.T, size=min(n_tok, wl.T), replace=False)).astype(np.int64)
    h = synth.host_inputs(wl, weights=False)
    x = np.ascontiguousarray(h["x"][tok])
    bias = h["bias"] if wl.zipf_s else None
    logits = oracle.router_logits(x, h["Wr"], bias)
    ids, _ = oracle.topk(logits, wl.k)
    experts = sorted({int(e) for e in ids.ravel()})
    W1 = {e: _expert(wl, "W1", e) for e in experts}
    W2 = {e: _expert(wl, "W2", e) for e in experts}
    t0 = time.perf_counter()
    oracle.forward(x, h["Wr"], bias, W1.get, W2.get, wl.k)
    dt = time.perf_counter() - t0
    flops = len(tok) * (2.0 * wl.H * wl.E + wl.k * 6.0 * wl.H * wl.I)
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return dt, flops, threads, len(tok), len(experts)


def calibrate_tokens(wl, budget_s: float):
    dt, _, threads, n, _ = oracle_sample(wl, max(2, min(os.cpu_count() or 1, 16)))
    per_tok = dt / n
    n_target = int(budget_s / max(per_tok, 1e-9))
    expert_bytes = 6.0 * wl.H * wl.I                        # W1[e] + W2[e], bf16
    if wl.E * expert_bytes > 24e9:                          # keep the sample's host weights under ~24 GB
        n_target = min(n_target, max(2, int(24e9 / (wl.k * expert_bytes))))
    return max(2, min(n_target, wl.T))


def cpu_baseline(wl, budget_s: float):
    import oracle
    oracle.build()
    n = calibrate_tokens(wl, budget_s)
    dt, flops, threads, n, ne = oracle_sample(wl, n, seed=2)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} of {wl.T} tokens (router + their {wl.k} experts each, {ne} experts touched), "
                      f"{dt:.1f} s; inputs regenerated on the host, generation untimed",
            "tokens_per_s": n / dt}


def run_reference(args, wl):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = calibrate_tokens(wl, min(budget, 8.0))
    for _ in range(args.warmup):
        oracle_sample(wl, n, seed=3)
    times, flops_tot, toks = 0.0, 0.0, 0
    threads = 1
    for i in range(args.steps):
        dt, fl, threads, nn, _ = oracle_sample(wl, n, seed=10 + i)
        times += dt
        flops_tot += fl
        toks += nn
    value = flops_tot / times / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * times / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32-accumulate bf16",
            "data": "synthetic (seeded generator)",
            "config": config_of(wl, args, l2="host CPU run"),
            "tokens_per_s": toks / times,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step {n} of {wl.T} tokens (router + their experts)"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def config_of(wl, args, l2):
    sched = {0: "wave-serial", 1: "interleaved", 2: "phased (L1 launch, L2 launch)",
             3: "auto (wave-serial, one wave of all experts)"}[args.schedule]
    split = "streaming" if args.gemm_split == "auto" else args.gemm_split
    return {"workload": f"{wl.name}: {wl.description}", "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
            "top_k": wl.k, "zipf_s": wl.zipf_s, "schedule": sched, "gemm_split": split,
            "wave_experts": args.wave_experts, "lead_waves": args.lead_waves, "l2": l2,
            "parallelism": f"replicas x{args.gpus} (no sharding)"}


# ----------------------------------------------------------------------------- GPU arm
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

    bias = synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None
    d = synth.device_inputs(wl, device=dev)
    flags = {"auto": 0, "streaming": moe.MOE_FLAG_GEMM_STREAMING, "compute": moe.MOE_FLAG_GEMM_COMPUTE}[args.gemm_split]
    layer = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, schedule=args.schedule, flags=flags,
                                       wave_experts=args.wave_experts, lead_waves=args.lead_waves),
                         local, router_bias=bias)
    logits = torch.empty((wl.T, wl.E), dtype=torch.float32, device=dev)
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    sampler = ClockSampler(local) if not args.no_clocks else None
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=logits, y=y)
    layer.check()
    r = layer.routing(wl.T)
    counts = r["counts"].cpu()
    touched = int((counts > 0).sum())
    launches = layer.launch_count()

    torch.cuda.synchronize()
    barrier(group)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):                # no host synchronisation inside the timed steps
        flush.zero_()
        ev[i][0].record()
        layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=logits, y=y)
        ev[i][1].record()
    torch.cuda.synchronize()
    barrier(group)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    layer.check()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = reduce_max(sum(step_ms), group)
    ms_per_step = total_ms / args.steps

    # ---- e2e: the host-buffer C-ABI call, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        x_host = d["x"].cpu().pin_memory()
        y_host = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
        for _ in range(2):
            flush.zero_()
            layer.forward_host(x_host, d["Wr"], d["W1"], d["W2"], logits, y_host)
        torch.cuda.synchronize()
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            eev[i][0].record()
            layer.forward_host(x_host, d["Wr"], d["W1"], d["W2"], logits, y_host)
            eev[i][1].record()
        torch.cuda.synchronize()
        layer.check()
        if not torch.equal(y_host.view(torch.int16), y.cpu().view(torch.int16)):
            raise RuntimeError("host-buffer forward disagrees with the device-buffer forward")
        e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in eev), group) / args.steps
        e2e = {"value": ws * wl.useful_flops() / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": wl.T * wl.H * 2, "d2h_bytes_per_step": wl.T * wl.H * 2,
               "ms_per_step": e_ms, "tokens_per_s": ws * wl.T / (e_ms * 1e-3)}
    # ---- per-stage breakdown on a second plan whose library records events between stages
    # (those events serialise the stream, so the headline steps above run without them)
    layer_t = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, schedule=args.schedule,
                                         flags=flags | moe.MOE_FLAG_STAGE_TIMING, wave_experts=args.wave_experts,
                                         lead_waves=args.lead_waves), local, router_bias=bias)
    stages = []
    for i in range(3 + min(args.steps, 20)):
        flush.zero_()
        layer_t.forward(d["x"], d["Wr"], d["W1"], d["W2"], logits=logits, y=y)
        if i >= 3:
            stages.append(layer_t.stage_times())
    layer_t.check()
    layer_t.close()
    if sampler:
        sampler.stop()
    clocks = sampler.summary(t0, t1) if sampler else None

    if rank != 0:
        return 0

    flops = wl.useful_flops()
    R = wl.T * wl.k
    w_bytes = 6.0 * wl.H * wl.I * touched
    layer_bytes = 2.0 * wl.T * wl.H * 2 + 2.0 * wl.H * wl.E + 4.0 * wl.T * wl.E + w_bytes
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = layer_bytes / (peaks["hbm_gbs"] * 1e9)
    t_step = ms_per_step * 1e-3
    stage_avg = {k: statistics.mean(s[k] for s in stages) for k in stages[0]}

    # dominant kernel: the persistent grouped GEMM (Linear-1 + SwiGLU, Linear-2 + scale)
    g_ms = stage_avg["grouped_gemm"]
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
    traffic = load_traffic("grouped_gemm_kernel", wl.name, args.schedule)
    roof.update({"traffic": traffic, "traffic_unit": "bytes per launch (ncu dram read+write)",
                 "kernel": "grouped_gemm_kernel", "ms_per_launch": g_ms,
                 "launches_per_step": 2 if args.schedule == 2 else 1,
                 "peak_source": f"{peak_src} ({'bf16_tflops burst' if tensor_bound else 'hbm_gbs'})",
                 "algorithmic": (f"{g_flops:.4g} FLOP (6*H*I per routed row x {R} rows)" if tensor_bound
                                 else f"{g_bytes:.4g} B (6*H*I bytes per touched expert x {touched})")})

    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        try:
            cpu = cpu_baseline(wl, args.cpu_budget)
        except Exception as ex:  # reported, not fatal
            cpu = {"value": None, "error": str(ex)[:200]}

    line = {
        "metric": METRIC, "value": ws * flops / t_step / 1e12, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded generator)",
        "config": config_of(wl, args, l2=f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write)"),
        "tokens_per_s": ws * wl.T / t_step,
        "layer_roofline": {"bound": "tensor" if t_tc >= t_hbm else "hbm", "frac": max(t_tc, t_hbm) / t_step,
                           "t_tensor_us": t_tc * 1e6, "t_hbm_us": t_hbm * 1e6,
                           "compulsory_bytes": layer_bytes, "useful_flops": flops,
                           "experts_touched": touched},
        "roofline": roof,
        "stages_ms": stage_avg,
        "gpu_launches": launches * args.steps,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "peaks": {**peaks, "source": peak_src},
    }
    print(json.dumps(line))
    if group:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)   # >= 0.2 s timed, several 50 ms clock samples
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default="fine")
    ap.add_argument("--schedule", type=int, choices=(0, 1, 2, 3), default=3,
                    help="0 wave-serial, 1 interleaved, 2 phased, 3 auto (the library's choice)")
    ap.add_argument("--wave-experts", type=int, default=0, help="experts per wave (0: fill the SMs)")
    ap.add_argument("--lead-waves", type=int, default=1, help="interleave lead D (interleaved schedule)")
    ap.add_argument("--gemm-split", choices=("auto", "streaming", "compute"), default="auto",
                    help="shared-memory split of the grouped GEMM (auto: the library default, streaming)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
