"""Single-GPU mixture-of-experts layer for GB300 (sm_103a) - Python binding.

The layer (router top-k -> Dispatch -> Linear-1 + SwiGLU -> Linear-2 ->
Combine) runs entirely in ``libmoe_gb300.so``; this module only marshals
arguments through the C ABI declared in ``include/moe_gb300.h``.  The
functions below carry the C names; ``MoELayer`` is a convenience wrapper over
torch tensors (torch supplies device memory and streams only).

There is no CPU fallback: importing works without a GPU, but every call needs
the built library and a CUDA device, and raises otherwise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_OOM = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6

MOE_SCHED_WAVE_SERIAL = 0
MOE_SCHED_INTERLEAVED = 1
MOE_SCHED_PHASED = 2
MOE_SCHED_AUTO = 3

MOE_FLAG_ACT_BILINEAR = 1 << 0
MOE_FLAG_STAGE_TIMING = 1 << 1
MOE_FLAG_TRACE = 1 << 2
MOE_FLAG_GEMM_STREAMING = 1 << 3
MOE_FLAG_GEMM_COMPUTE = 1 << 4
MOE_FLAG_EXACT_LOGITS = 1 << 5
MOE_FLAG_SINGLE_LAUNCH = 1 << 6
MOE_FLAG_HOST_PIPELINE = 1 << 7
TRACE_FIELDS = ("prod_wait_empty_ns", "prod_wait_ready_ns", "mma_wait_tempty_ns", "mma_wait_full_ns",
                "epi_wait_tfull_ns", "cta_ns", "tiles_l1", "tiles_l2")
MOE_FLAG_TEST_STALL = 1 << 8
MOE_FLAG_TEST_BAD_ID = 1 << 9

MOE_NUM_STAGES = 5
STAGE_NAMES = ("router_topk", "dispatch", "gather", "grouped_gemm", "combine")

EXPORTED = ("moe_plan", "moe_workspace_bytes", "moe_forward", "moe_forward_host", "moe_host_wait", "moe_get_status",
            "moe_debug_routing",
            "moe_debug_intermediates", "moe_stage_times", "moe_last_launch_count", "moe_plan_destroy",
            "moe_status_string", "moe_schedule_host", "moe_dispatch_static", "moe_trace_read", "moe_trace_tiles",
            "moe_router_bound", "moe_debug_schedule")


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {moe_status_string(status)} ({status})")


class moe_config_t(ctypes.Structure):
    _fields_ = [("T_max", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("schedule", ctypes.c_int32),
                ("wave_experts", ctypes.c_int32), ("lead_waves", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("timeout_ns", ctypes.c_int64),
                ("router_bias", ctypes.c_void_p)]


_lib = None


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def load() -> ctypes.CDLL:
    """Load libmoe_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with mixture_experts_layer_top_gb300.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    P = ctypes.POINTER
    L.moe_plan.argtypes = [P(moe_config_t), ctypes.c_int, P(vp)]
    L.moe_workspace_bytes.argtypes = [P(moe_config_t), P(ctypes.c_size_t)]
    L.moe_forward.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
    L.moe_forward_host.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
    L.moe_get_status.argtypes = [vp, vp]
    L.moe_host_wait.argtypes = [vp, vp]
    L.moe_debug_routing.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp]
    L.moe_debug_intermediates.argtypes = [vp, i32, vp, vp, vp]
    L.moe_stage_times.argtypes = [vp, P(ctypes.c_float)]
    L.moe_last_launch_count.argtypes = [vp, P(i32)]
    L.moe_router_bound.argtypes = [vp, i32, P(ctypes.c_float)]
    L.moe_debug_schedule.argtypes = [vp, vp, ctypes.c_int64, P(ctypes.c_int64), vp]
    L.moe_plan_destroy.argtypes = [vp]
    L.moe_status_string.argtypes = [ctypes.c_int]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_schedule_host.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, vp, i64, P(i64)]
    L.moe_dispatch_static.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
    L.moe_trace_read.argtypes = [vp, vp, ctypes.c_size_t, P(ctypes.c_size_t)]
    L.moe_trace_tiles.argtypes = [vp, vp, ctypes.c_size_t, P(ctypes.c_size_t)]
    for f in EXPORTED:
        if f != "moe_status_string":
            getattr(L, f).restype = ctypes.c_int
    _lib = L
    return L


# --------------------------------------------------------------------------- C-named calls
def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_workspace_bytes(cfg: moe_config_t) -> int:
    n = ctypes.c_size_t(0)
    st = load().moe_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n))
    if st != MOE_OK:
        raise MoEError(st, "moe_workspace_bytes")
    return n.value


def moe_plan(cfg: moe_config_t, device: int = 0) -> int:
    h = ctypes.c_void_p(0)
    st = load().moe_plan(ctypes.byref(cfg), int(device), ctypes.byref(h))
    if st != MOE_OK:
        raise MoEError(st, "moe_plan")
    return h.value


def moe_forward(plan: int, T: int, x: int, router_logits: int, W_router: Optional[int], W1_gate_up: int,
                W2: int, y: int, stream: int) -> int:
    return load().moe_forward(plan, int(T), x, router_logits, W_router, W1_gate_up, W2, y, stream)


def moe_forward_host(plan: int, T: int, x_host: int, router_logits: int, W_router: Optional[int],
                     W1_gate_up: int, W2: int, y_host: int, stream: int) -> int:
    return load().moe_forward_host(plan, int(T), x_host, router_logits, W_router, W1_gate_up, W2, y_host,
                                   stream)


def moe_get_status(plan: int, stream: int) -> int:
    return load().moe_get_status(plan, stream)


def moe_host_wait(plan: int, stream: int) -> int:
    return load().moe_host_wait(plan, stream)


def moe_debug_routing(plan: int, T: int, ids, w, counts, offsets, row_pair, row_of, stream: int) -> int:
    return load().moe_debug_routing(plan, int(T), ids, w, counts, offsets, row_pair, row_of, stream)


def moe_debug_intermediates(plan: int, T: int, h, P, stream: int) -> int:
    return load().moe_debug_intermediates(plan, int(T), h, P, stream)


def moe_stage_times(plan: int):
    arr = (ctypes.c_float * MOE_NUM_STAGES)()
    st = load().moe_stage_times(plan, arr)
    if st != MOE_OK:
        raise MoEError(st, "moe_stage_times")
    return list(arr)


def moe_router_bound(plan: int, T: int) -> float:
    c = ctypes.c_float(0.0)
    st = load().moe_router_bound(plan, T, ctypes.byref(c))
    if st != MOE_OK:
        raise MoEError(st, "moe_router_bound")
    return c.value


def moe_last_launch_count(plan: int) -> int:
    n = ctypes.c_int32(0)
    st = load().moe_last_launch_count(plan, ctypes.byref(n))
    if st != MOE_OK:
        raise MoEError(st, "moe_last_launch_count")
    return n.value


def moe_trace_read(plan: int) -> np.ndarray:
    """Per-CTA wait-time counters of the last forward's grouped GEMM: [CTAs + 1, 8] uint64
    (fields in TRACE_FIELDS; the last row: the phase stamps of a single-launch forward).
    Needs MOE_FLAG_TRACE."""
    n = ctypes.c_size_t(0)
    L = load()
    st = L.moe_trace_read(plan, None, 0, ctypes.byref(n))
    if st != MOE_OK:
        raise MoEError(st, "moe_trace_read")
    out = np.zeros(n.value, dtype=np.uint64)
    st = L.moe_trace_read(plan, out.ctypes.data, n.value, ctypes.byref(n))
    if st != MOE_OK:
        raise MoEError(st, "moe_trace_read")
    return out.reshape(-1, len(TRACE_FIELDS))


TILE_TRACE_FIELDS = ("sm_id", "start_ns", "acc_ready_ns", "end_ns")


def moe_trace_tiles(plan: int) -> np.ndarray:
    """Per-tile trace of the last forward's grouped GEMM: [tiles, 2 (CTA rank), 4] uint64 (fields
    in TILE_TRACE_FIELDS), tiles in the order of moe_debug_schedule.  Needs MOE_FLAG_TRACE."""
    n = ctypes.c_size_t(0)
    L = load()
    st = L.moe_trace_tiles(plan, None, 0, ctypes.byref(n))
    if st != MOE_OK:
        raise MoEError(st, "moe_trace_tiles")
    out = np.zeros(n.value, dtype=np.uint64)
    if n.value:
        st = L.moe_trace_tiles(plan, out.ctypes.data, n.value, ctypes.byref(n))
        if st != MOE_OK:
            raise MoEError(st, "moe_trace_tiles")
    return out.reshape(-1, 2, len(TILE_TRACE_FIELDS))


def moe_plan_destroy(plan: int) -> int:
    return load().moe_plan_destroy(plan)


def moe_dispatch_static(T: int, E: int, k: int, ids, w, offsets, row_pair, row_of, row_w, stream: int) -> int:
    """Dispatch sort that allocates nothing (scratch in a fixed array inside the library);
    for callers that cannot call cudaMalloc.  Device pointers; see include/moe_gb300.h."""
    return load().moe_dispatch_static(int(T), int(E), int(k), ids, w, offsets, row_pair, row_of, row_w, stream)


def moe_schedule_host(counts, H: int, I: int, num_sms: int, schedule: int, wave_experts: int = 0,
                      lead_waves: int = 1):
    """Tile order the device scheduler builds for these per-expert row counts.
    Returns (tiles [n, 4] int32 {phase | n_block << 1, expert, m_block, m_tile}, n_linear1)."""
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    n = (ctypes.c_int64 * 2)()
    L = load()
    st = L.moe_schedule_host(counts.ctypes.data, len(counts), H, I, num_sms, schedule, wave_experts,
                             lead_waves, None, 0, n)
    if st != MOE_OK:
        raise MoEError(st, "moe_schedule_host")
    tiles = np.full((n[1], 4), -1, dtype=np.int32)
    st = L.moe_schedule_host(counts.ctypes.data, len(counts), H, I, num_sms, schedule, wave_experts,
                             lead_waves, tiles.ctypes.data, n[1], n)
    if st != MOE_OK:
        raise MoEError(st, "moe_schedule_host")
    return tiles, int(n[0])


# --------------------------------------------------------------------------- torch wrapper
@dataclass
class MoEConfig:
    T_max: int
    H: int
    I: int
    E: int
    top_k: int
    schedule: int = MOE_SCHED_AUTO
    wave_experts: int = 0
    lead_waves: int = 1
    flags: int = 0
    timeout_ns: int = 0

    def c(self, bias_ptr=None) -> moe_config_t:
        return moe_config_t(self.T_max, self.H, self.I, self.E, self.top_k, self.schedule,
                            self.wave_experts, self.lead_waves, self.flags, self.timeout_ns, bias_ptr)


def _ptr(t):
    return None if t is None else t.data_ptr()


class MoELayer:
    """One plan (workspace for T_max tokens) on one device.

    ``forward(x, W_router, W1, W2, logits=None, y=None)``: x bf16 [T,H], W_router bf16 [H,E]
    (or None when ``logits`` [T,E] fp32 is given as input), W1 bf16 [E,H,2I], W2 bf16 [E,I,H].
    Returns (y bf16 [T,H], logits fp32 [T,E])."""

    def __init__(self, cfg: MoEConfig, device: int = 0, router_bias=None):
        import torch
        self.cfg = cfg
        self.device = device
        self._bias_host = None
        bias_ptr = None
        if router_bias is not None:
            b = np.ascontiguousarray(np.asarray(router_bias, dtype=np.float32))
            assert b.shape == (cfg.E,)
            self._bias_host = b
            bias_ptr = b.ctypes.data
        with torch.cuda.device(device):
            self.plan = moe_plan(cfg.c(bias_ptr), device)

    def close(self):
        if getattr(self, "plan", None):
            moe_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _stream():
        import torch
        return torch.cuda.current_stream().cuda_stream

    def forward(self, x, W_router, W1, W2, logits=None, y=None, check: bool = False):
        import torch
        T = x.shape[0]
        dev = x.device
        if y is None:
            y = torch.empty((T, self.cfg.H), dtype=torch.bfloat16, device=dev)
        if logits is None:
            if W_router is None:
                raise ValueError("need W_router or logits")
            logits = torch.empty((T, self.cfg.E), dtype=torch.float32, device=dev)
        st = moe_forward(self.plan, T, _ptr(x), _ptr(logits), _ptr(W_router), _ptr(W1), _ptr(W2), _ptr(y),
                         self._stream())
        if st != MOE_OK:
            raise MoEError(st, "moe_forward")
        if check:
            self.check()
        return y, logits

    def forward_host(self, x_host, W_router, W1, W2, logits, y_host, check: bool = False):
        """x_host / y_host: CPU bf16 tensors (page-locked for asynchronous copies)."""
        T = x_host.shape[0]
        st = moe_forward_host(self.plan, T, _ptr(x_host), _ptr(logits), _ptr(W_router), _ptr(W1), _ptr(W2),
                              _ptr(y_host), self._stream())
        if st != MOE_OK:
            raise MoEError(st, "moe_forward_host")
        if check:
            self.check()
        return y_host, logits

    def host_wait(self):
        """Make the current stream wait for the output copies of the pipelined host forwards
        (MOE_FLAG_HOST_PIPELINE) enqueued so far."""
        st = moe_host_wait(self.plan, self._stream())
        if st != MOE_OK:
            raise MoEError(st, "moe_host_wait")

    def check(self):
        st = moe_get_status(self.plan, self._stream())
        if st != MOE_OK:
            raise MoEError(st, "device status")

    def routing(self, T: int) -> dict:
        import torch
        k, E = self.cfg.top_k, self.cfg.E
        d = dict(ids=torch.empty((T, k), dtype=torch.int32, device="cuda"),
                 w=torch.empty((T, k), dtype=torch.float32, device="cuda"),
                 counts=torch.empty(E, dtype=torch.int32, device="cuda"),
                 offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
                 row_pair=torch.empty(T * k, dtype=torch.int32, device="cuda"),
                 row_of=torch.empty(T * k, dtype=torch.int32, device="cuda"))
        st = moe_debug_routing(self.plan, T, *[_ptr(d[n]) for n in
                                               ("ids", "w", "counts", "offsets", "row_pair", "row_of")],
                               self._stream())
        if st != MOE_OK:
            raise MoEError(st, "moe_debug_routing")
        return d

    def intermediates(self, T: int, want_h: bool = True, want_P: bool = True):
        import torch
        R = T * self.cfg.top_k
        h = torch.empty((R, self.cfg.I), dtype=torch.bfloat16, device="cuda") if want_h else None
        P = torch.empty((R, self.cfg.H), dtype=torch.float32, device="cuda") if want_P else None
        st = moe_debug_intermediates(self.plan, T, _ptr(h), _ptr(P), self._stream())
        if st != MOE_OK:
            raise MoEError(st, "moe_debug_intermediates")
        return h, P

    def stage_times(self):
        return dict(zip(STAGE_NAMES, moe_stage_times(self.plan)))

    def launch_count(self) -> int:
        return moe_last_launch_count(self.plan)

    def schedule(self):
        """(tiles [n, 4] int32, n_linear1, workers) the last forward's Dispatch built on the device."""
        L = load()
        n = (ctypes.c_int64 * 3)()
        st = L.moe_debug_schedule(self.plan, None, 0, n, self._stream())
        if st != MOE_OK:
            raise MoEError(st, "moe_debug_schedule")
        tiles = np.full((n[1], 4), -1, dtype=np.int32)
        st = L.moe_debug_schedule(self.plan, tiles.ctypes.data, n[1], n, self._stream())
        if st != MOE_OK:
            raise MoEError(st, "moe_debug_schedule")
        return tiles, int(n[0]), int(n[2])

    def router_bound(self, T: int) -> float:
        """cH of the default router's logit error bound for T tokens."""
        return moe_router_bound(self.plan, T)
