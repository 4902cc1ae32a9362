"""Seeded synthetic inputs for the MoE layer, shared by the CUDA path and the oracle.

This module holds no mixture-of-experts arithmetic: it only draws random
tensors and names the five workload shapes.  Two implementations of one
counter-based generator live here and give bit-identical values:

* ``normal_bf16_host`` - the C implementation in ``synth.c`` (fast, host),
  used by the oracle side;
* ``normal_bf16_torch`` - the same float64 operation sequence in torch, used
  to create tensors directly in device memory (and testable on the CPU).

Definition of element ``i`` of tensor ``tid`` under ``seed``::

    word  = fmix64(fmix64(seed*G + tid) + (i+1)*G)       (SplitMix64 finaliser)
    u1    = ((word >> 40) + 0.5) * 2**-24                 in (0, 1)
    u2    = ((word >> 16) & 0xFFFFFF) * 2**-24            in [0, 1)
    n     = sqrt(-2 ln u1) * cos(2 pi u2)                 (Box-Muller)
    value = bf16_rne(f32_rne(n * std))

``ln`` and ``cos`` are float64 polynomials (atanh series, Taylor series)
evaluated with +, -, *, / only, so every platform rounds them identically.
Tensor ids: x = 1, W_router = 2, W1 = 3, W2 = 4.

The workloads follow the mixture-of-experts layer of the X-Stage paper's
MegaMoE background (router -> top-k -> Dispatch -> Linear-1 -> SwiGLU ->
Linear-2 -> Combine): x ~ N(0,1), W_router ~ N(0,1/H), W1 ~ N(0,1/H),
W2 ~ N(0,1/I), bf16, seed 0.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")

G_GOLDEN = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

TID_X, TID_WR, TID_W1, TID_W2 = 1, 2, 3, 4

# float64 constants shared by both implementations.
LN_COEF = [1.0 / (2 * k + 1) for k in range(12)]          # atanh(s)/s = sum s^2k/(2k+1)
COS_COEF = [(-1.0) ** n / float(math.factorial(2 * n)) for n in range(13)]
LN2 = 0.6931471805599453
SQRT_HALF = 0.7071067811865476
TWO_PI = 6.283185307179586
INV24 = 1.0 / 16777216.0


# ----------------------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Workload:
    """One synthetic MoE-layer workload: T tokens, hidden H, intermediate I per
    expert, E experts, top-k routing, optional Zipf(s) expert prior on the
    router logits."""
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    zipf_s: float = 0.0
    seed: int = 0
    description: str = field(default="", compare=False)

    @property
    def R(self) -> int:
        return self.T * self.k

    def useful_flops(self) -> float:
        """2*H*2I (Linear-1) + 2*I*H (Linear-2) per routed row, 2*H*E per token (router)."""
        return 6.0 * self.H * self.I * self.R + 2.0 * self.H * self.E * self.T


WORKLOADS = {
    "tiny": Workload("tiny", 256, 512, 256, 8, 2,
                     description="Tiny MoE layer T=256 H=512 I=256 E=8 top-2"),
    "fine": Workload("fine", 8192, 2048, 768, 128, 8,
                     description="Fine-grained MoE T=8192 H=2048 I=768 E=128 top-8, near-uniform routing"),
    "skew": Workload("skew", 16384, 2048, 768, 128, 8, zipf_s=1.2,
                     description="Skewed routing T=16384 H=2048 I=768 E=128 top-8, Zipf(1.2) prior"),
    "large": Workload("large", 4096, 7168, 2048, 256, 8,
                      description="Large MoE layer T=4096 H=7168 I=2048 E=256 top-8"),
    "smallT": Workload("smallT", 128, 7168, 2048, 256, 8,
                       description="Small-T weight-streaming T=128 H=7168 I=2048 E=256 top-8"),
}


def zipf_bias(E: int, s: float) -> np.ndarray:
    """Router-logit bias 2*ln(p_e) with p_e = (e+1)^-s / sum_e' (e'+1)^-s, as fp32.
    Zero vector when s == 0."""
    if s == 0.0:
        return np.zeros(E, dtype=np.float32)
    w = np.array([(e + 1.0) ** (-s) for e in range(E)], dtype=np.float64)
    p = w / w.sum()
    return (2.0 * np.log(p)).astype(np.float32)


def std_of(fan_in: int) -> float:
    return 1.0 / math.sqrt(fan_in)


# ----------------------------------------------------------------------------- scalar reference
def _fmix64_int(z: int) -> int:
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def word_int(seed: int, tid: int, i: int) -> int:
    """The 64-bit counter word as a Python int (definition above)."""
    key = _fmix64_int((seed * G_GOLDEN + tid) & MASK64)
    return _fmix64_int((key + (i + 1) * G_GOLDEN) & MASK64)


# ----------------------------------------------------------------------------- host (C)
_lib = None


def build_host(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, OpenMP, no FMA contraction)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", src, "-o", _LIB_PATH + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build_host()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.synth_normal_bf16.argtypes = [
            ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
            ctypes.POINTER(ctypes.c_double), ctypes.c_int, ctypes.POINTER(ctypes.c_double),
            ctypes.c_int, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p]
        lib.synth_normal_bf16.restype = None
        lib.synth_word.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_word.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def _dbl(a):
    arr = (ctypes.c_double * len(a))(*a)
    return arr


def normal_bf16_host(n: int, std: float, tid: int, seed: int = 0, start: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of elements start .. start+n-1 of tensor ``tid``."""
    lib = _load()
    out = np.empty(n, dtype=np.uint16)
    if n:
        lib.synth_normal_bf16(seed, tid, start, n, float(std), _dbl(LN_COEF), len(LN_COEF),
                              _dbl(COS_COEF), len(COS_COEF), _dbl([LN2, SQRT_HALF, TWO_PI]),
                              out.ctypes.data)
    return out


# ----------------------------------------------------------------------------- torch (any device)
def _signed(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


def _lsr(z, s: int):
    import torch
    return torch.bitwise_and(z >> s, (1 << (64 - s)) - 1)


def _fmix64_t(z):
    z = (z ^ _lsr(z, 30)) * _signed(M1)
    z = (z ^ _lsr(z, 27)) * _signed(M2)
    return z ^ _lsr(z, 31)


def _ln_t(u):
    import torch
    bits = u.view(torch.int64)
    e = (_lsr(bits, 52) & 0x7FF) - 1022
    mbits = (bits & _signed(0x800FFFFFFFFFFFFF)) | (1022 << 52)
    m = mbits.view(torch.float64)
    small = m < SQRT_HALF
    m = torch.where(small, m * 2.0, m)
    e = torch.where(small, e - 1, e)
    s = (m - 1.0) / (m + 1.0)
    z = s * s
    p = torch.full_like(z, LN_COEF[-1])
    for c in reversed(LN_COEF[:-1]):
        p = p * z + c
    return 2.0 * s * p + e.to(torch.float64) * LN2


def _cos2pi_t(v):
    import torch
    w = torch.where(v > 0.5, 1.0 - v, v)
    flip = w > 0.25
    w = torch.where(flip, 0.5 - w, w)
    sign = torch.where(flip, -1.0, 1.0).to(torch.float64)
    th = w * TWO_PI
    t2 = th * th
    p = torch.full_like(t2, COS_COEF[-1])
    for c in reversed(COS_COEF[:-1]):
        p = p * t2 + c
    return sign * p


def normal_bf16_torch(n: int, std: float, tid: int, seed: int = 0, start: int = 0,
                      device="cpu", chunk: int = 1 << 24):
    """torch.bfloat16 tensor [n] on ``device`` with the same values as normal_bf16_host."""
    import torch
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    key = _fmix64_int((seed * G_GOLDEN + tid) & MASK64)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        i = torch.arange(start + c0 + 1, start + c1 + 1, dtype=torch.int64, device=device)
        z = i * _signed(G_GOLDEN) + _signed(key)
        w = _fmix64_t(z)
        u1 = (_lsr(w, 40).to(torch.float64) + 0.5) * INV24
        u2 = (_lsr(w, 16) & 0xFFFFFF).to(torch.float64) * INV24
        r = torch.sqrt(-2.0 * _ln_t(u1))
        v = r * _cos2pi_t(u2)
        out[c0:c1] = (v * std).to(torch.float32).to(torch.bfloat16)
    return out


# ----------------------------------------------------------------------------- full layer inputs
def expert_slice_host(wl: Workload, which: str, e: int) -> np.ndarray:
    """Host bf16 bits of one expert's weight matrix: W1[e] as [H, 2I] or W2[e] as [I, H]."""
    if which == "W1":
        n = wl.H * 2 * wl.I
        return normal_bf16_host(n, std_of(wl.H), TID_W1, wl.seed, start=e * n).reshape(wl.H, 2 * wl.I)
    if which == "W2":
        n = wl.I * wl.H
        return normal_bf16_host(n, std_of(wl.I), TID_W2, wl.seed, start=e * n).reshape(wl.I, wl.H)
    raise ValueError(which)


def host_inputs(wl: Workload, weights: bool = True) -> dict:
    """All layer inputs as host numpy arrays of bf16 bit patterns (uint16) + fp32 bias."""
    d = {
        "x": normal_bf16_host(wl.T * wl.H, 1.0, TID_X, wl.seed).reshape(wl.T, wl.H),
        "Wr": normal_bf16_host(wl.H * wl.E, std_of(wl.H), TID_WR, wl.seed).reshape(wl.H, wl.E),
        "bias": zipf_bias(wl.E, wl.zipf_s),
    }
    if weights:
        d["W1"] = normal_bf16_host(wl.E * wl.H * 2 * wl.I, std_of(wl.H), TID_W1, wl.seed).reshape(
            wl.E, wl.H, 2 * wl.I)
        d["W2"] = normal_bf16_host(wl.E * wl.I * wl.H, std_of(wl.I), TID_W2, wl.seed).reshape(
            wl.E, wl.I, wl.H)
    return d


def device_inputs(wl: Workload, device="cuda") -> dict:
    """All layer inputs as torch tensors created on ``device`` (bf16 + fp32 bias)."""
    import torch
    return {
        "x": normal_bf16_torch(wl.T * wl.H, 1.0, TID_X, wl.seed, device=device).view(wl.T, wl.H),
        "Wr": normal_bf16_torch(wl.H * wl.E, std_of(wl.H), TID_WR, wl.seed, device=device).view(wl.H, wl.E),
        "bias": torch.from_numpy(zipf_bias(wl.E, wl.zipf_s)).to(device),
        "W1": normal_bf16_torch(wl.E * wl.H * 2 * wl.I, std_of(wl.H), TID_W1, wl.seed,
                                device=device).view(wl.E, wl.H, 2 * wl.I),
        "W2": normal_bf16_torch(wl.E * wl.I * wl.H, std_of(wl.I), TID_W2, wl.seed,
                                device=device).view(wl.E, wl.I, wl.H),
    }
