"""Host logic of bench.py: the max-over-ranks reduction of the replica path
(world size 2 over gloo on the CPU) and the clock-sample summary."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    v = bench.reduce_max(10.0 + 5.0 * rank, True)
    bench.barrier(True)
    q.put((rank, v))
    dist.destroy_process_group()


def test_reduce_max_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
    assert out == {0: 15.0, 1: 15.0}


def test_reduce_max_single_process_is_identity():
    assert bench.reduce_max(3.5, False) == 3.5


def test_clock_summary_flags_throttling():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.proc = None
    cs.samples = [(1.0 + 0.1 * i, ["1900", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active",
                                   "Active" if i == 2 else "Not Active"]) for i in range(10)]
    s = cs.summary(1.0, 2.0)
    assert s["sm_mhz"] == 1900 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]


def test_workload_flops():
    wl = bench.synth.WORKLOADS["fine"]
    assert wl.useful_flops() == pytest.approx(6 * 2048 * 768 * 8192 * 8 + 2 * 2048 * 128 * 8192)


def _reference_arm(rank: int):
    import subprocess
    env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                           "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_rank0_prints_one_line_other_ranks_exit_quietly():
    """The reference arm (the oracle timed on the host cores): under a launcher only rank 0
    works and prints one JSON line with the contract's keys; any other rank exits 0 silently."""
    import json
    r1 = _reference_arm(1)
    assert r1.returncode == 0 and r1.stdout.strip() == "", r1.stderr[-2000:]
    r0 = _reference_arm(0)
    assert r0.returncode == 0, r0.stderr[-2000:]
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("tiny")
