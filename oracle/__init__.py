"""CPU oracle for the MoE layer - TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product (the CUDA library and its
Python binding) never imports it, and it never imports the product.

The arithmetic lives in ``moe_oracle.c`` (plain C loops, see its header for
the step-by-step definition, which follows the MoE layer of the X-Stage
paper's MegaMoE background paragraph).  This file only marshals numpy
arrays.  bf16 tensors are passed as ``uint16`` bit patterns.

Parity status: every function is pinned by ``tests/test_oracle_pins.py``
(library routines, closed forms, brute-force dense evaluation, exact integer
cases, hand-built rounding-boundary cases, brute-force enumeration of the
intermediate's rounding alternatives); none is "parity unpinned".

Besides the layer's result, ``forward(..., bounds=True)`` reports what the
comparison with another implementation needs: y before its final rounding
(``y32``) and the interval [``ylo``, ``yhi``] that y can take when the
intermediates that lie within the stated accumulation-error bound of a bf16
rounding boundary (``moe_oracle.c``, "Rounding flags") round to their other
neighbour.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

ACT_SWIGLU = 0
ACT_BILINEAR = 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c -> liboracle.so (gcc, OpenMP over tokens, no FP contraction)."""
    src = os.path.join(_HERE, "moe_oracle.c")
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(src):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", src, "-o", _LIB + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.oracle_f32_to_bf16_array.argtypes = [i64, vp, vp]
        L.oracle_router_logits.argtypes = [i64, i32, i32, vp, vp, vp, vp]
        L.oracle_topk.argtypes = [i64, i32, i32, vp, vp, vp]
        L.oracle_dispatch.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp]
        L.oracle_expert_ffn.argtypes = [i32, i32, vp, vp, vp, i32, vp, vp, vp]
        L.oracle_forward_tokens.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i64, vp,
                                            vp, vp, vp]
        L.oracle_forward_tokens.restype = ctypes.c_int
        L.oracle_expert_h_range.argtypes = [i32, i32, vp, vp, i32, vp, vp, vp, vp]
        L.oracle_expert_rows.argtypes = [i32, i32, i32, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.oracle_combine.argtypes = [i32, i32, i64, vp, vp, vp, vp, vp, vp, vp, vp]
        for f in ("oracle_f32_to_bf16_array", "oracle_router_logits", "oracle_topk",
                  "oracle_dispatch", "oracle_expert_ffn", "oracle_expert_h_range", "oracle_expert_rows",
                  "oracle_combine"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ------------------------------------------------------------------------ bf16 helpers
def f32_to_bf16(a) -> np.ndarray:
    a, p = _c(a, np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_f32_to_bf16_array(a.size, p, out.ctypes.data)
    return out


def bf16_to_f32(bits) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------------ steps
def router_logits(x, Wr, bias=None) -> np.ndarray:
    """fp32 [T,E] logits in the canonical order (x: [T,H] bf16 bits, Wr: [H,E] bf16 bits)."""
    x, px = _c(x, np.uint16)
    Wr, pw = _c(Wr, np.uint16)
    T, H = x.shape
    E = Wr.shape[1]
    assert Wr.shape[0] == H and H % 32 == 0
    pb = None
    if bias is not None:
        bias, pb = _c(bias, np.float32)
    out = np.empty((T, E), dtype=np.float32)
    _load().oracle_router_logits(T, H, E, px, pw, pb, out.ctypes.data)
    return out


def topk(logits, k: int):
    """ids int32 [T,k] (descending logit, ties -> lower id), weights fp32 [T,k]."""
    logits, pl = _c(logits, np.float32)
    T, E = logits.shape
    assert 1 <= k <= min(E, 64) and E <= 1024
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _load().oracle_topk(T, E, k, pl, ids.ctypes.data, w.ctypes.data)
    return ids, w


def dispatch(ids, E: int):
    """counts [E], offsets [E+1], row_pair [T*k], row_of [T*k] (all int32)."""
    ids, pi = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    row_pair = np.empty(T * k, np.int32)
    row_of = np.empty(T * k, np.int32)
    _load().oracle_dispatch(T, E, k, pi, counts.ctypes.data, offsets.ctypes.data,
                            row_pair.ctypes.data, row_of.ctypes.data)
    return counts, offsets, row_pair, row_of


def expert_ffn(x_row, W1e, W2e, act: int = ACT_SWIGLU):
    """One expert on one token: a (bf16 bits [I]) and o (fp32 [H])."""
    x_row, px = _c(x_row, np.uint16)
    W1e, p1 = _c(W1e, np.uint16)
    W2e, p2 = _c(W2e, np.uint16)
    H, I2 = W1e.shape
    I = I2 // 2
    assert W2e.shape == (I, H) and x_row.shape == (H,)
    a = np.empty(I, np.uint16)
    o = np.empty(H, np.float32)
    scratch = np.empty(2 * I, np.float32)
    _load().oracle_expert_ffn(H, I, px, p1, p2, act, a.ctypes.data, o.ctypes.data,
                              scratch.ctypes.data)
    return a, o


def forward_tokens(x, ids, w, tokens, W1_of, W2_of, E: int, act: int = ACT_SWIGLU,
                   want_intermediates: bool = False):
    """y (bf16 bits [ns,H]) for the sampled tokens; W1_of(e) -> [H,2I], W2_of(e) -> [I,H]
    give the (host, bf16 bits) weights of expert e.  Optionally a [ns,k,I], o [ns,k,H]."""
    x, px = _c(x, np.uint16)
    ids, pi = _c(ids, np.int32)
    w, pw = _c(w, np.float32)
    tokens, pt = _c(tokens, np.int64)
    T, H = x.shape
    k = ids.shape[1]
    need = sorted({int(e) for t in tokens for e in ids[t]})
    keep = {}
    P1 = (ctypes.c_void_p * E)()
    P2 = (ctypes.c_void_p * E)()
    I = None
    for e in need:
        a1 = np.ascontiguousarray(W1_of(e), dtype=np.uint16)
        a2 = np.ascontiguousarray(W2_of(e), dtype=np.uint16)
        I = a2.shape[0]
        keep[e] = (a1, a2)
        P1[e] = a1.ctypes.data
        P2[e] = a2.ctypes.data
    ns = len(tokens)
    if I is None:
        I = 0
    y = np.empty((ns, H), np.uint16)
    a_out = np.empty((ns, k, I), np.uint16) if want_intermediates else None
    o_out = np.empty((ns, k, H), np.float32) if want_intermediates else None
    rc = _load().oracle_forward_tokens(
        H, I, E, k, act, px, P1, P2, pi, pw, ns, pt, y.ctypes.data,
        a_out.ctypes.data if a_out is not None else None,
        o_out.ctypes.data if o_out is not None else None)
    if rc != 0:
        raise RuntimeError(f"oracle_forward_tokens failed ({rc})")
    if want_intermediates:
        return y, a_out, o_out
    return y


def expert_h_range(x_row, W1e, act: int = ACT_SWIGLU):
    """The bf16 values the intermediate of one token through one expert can take under the
    stated accumulation-error bound: a_lo, a_hi (bf16 bits [I]), plus the exact g|u [2I]
    and their radius [2I] (both float64)."""
    x_row, px = _c(x_row, np.uint16)
    W1e, p1 = _c(W1e, np.uint16)
    H, I2 = W1e.shape
    I = I2 // 2
    lo = np.empty(I, np.uint16)
    hi = np.empty(I, np.uint16)
    g = np.empty(2 * I, np.float64)
    rad = np.empty(2 * I, np.float64)
    _load().oracle_expert_h_range(H, I, px, p1, act, lo.ctypes.data, hi.ctypes.data, g.ctypes.data,
                                  rad.ctypes.data)
    return lo, hi, g, rad


def _forward_by_expert(x, ids, w, tokens, W1_of, W2_of, act, bounds, want_intermediates,
                       experts_per_batch: int = 16, timing=None):
    """y of the sampled tokens, driven expert by expert: the weights of each expert the
    sample touches are requested once, a batch of experts at a time (host memory stays
    bounded), and every (token, slot) row of those experts is evaluated by
    oracle_expert_rows; then oracle_combine sums the slots.  Same arithmetic as
    forward_tokens."""
    x, px = _c(x, np.uint16)
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    ns, k = len(tokens), ids.shape[1]
    H = x.shape[1]
    sel = ids[tokens]                                      # [ns, k]
    experts = sorted({int(e) for e in sel.ravel()})
    L = _load()
    o = a = dlo = dhi = nflag = None
    I = None
    for b0 in range(0, len(experts), experts_per_batch):
        batch = experts[b0:b0 + experts_per_batch]
        mats = {e: (np.ascontiguousarray(W1_of(e), dtype=np.uint16), np.ascontiguousarray(W2_of(e), dtype=np.uint16))
                for e in batch}
        if I is None:
            I = mats[batch[0]][1].shape[0]
            o = np.empty((ns, k, H), np.float32)
            a = np.empty((ns, k, I), np.uint16)
            if bounds:
                dlo = np.empty((ns, k, H), np.float64)
                dhi = np.empty((ns, k, H), np.float64)
                nflag = np.zeros((ns, k), np.int32)
                a_lo = np.empty((ns, k, I), np.uint16)
                a_hi = np.empty((ns, k, I), np.uint16)
        rows = [(s, j) for s in range(ns) for j in range(k) if int(sel[s, j]) in mats]
        n = len(rows)
        toks = np.array([tokens[s] for s, _ in rows], np.int64)
        P1 = (ctypes.c_void_p * n)(*[mats[int(sel[s, j])][0].ctypes.data for s, j in rows])
        P2 = (ctypes.c_void_p * n)(*[mats[int(sel[s, j])][1].ctypes.data for s, j in rows])
        a_b = np.empty((n, I), np.uint16)
        o_b = np.empty((n, H), np.float32)
        dl_b = np.empty((n, H), np.float64) if bounds else None
        dh_b = np.empty((n, H), np.float64) if bounds else None
        nf_b = np.zeros(n, np.int32) if bounds else None
        lo_b = np.empty((n, I), np.uint16) if bounds else None
        hi_b = np.empty((n, I), np.uint16) if bounds else None
        tc = time.perf_counter()
        L.oracle_expert_rows(H, I, act, px, n, toks.ctypes.data, P1, P2, a_b.ctypes.data, o_b.ctypes.data,
                             dl_b.ctypes.data if bounds else None, dh_b.ctypes.data if bounds else None,
                             nf_b.ctypes.data if bounds else None, lo_b.ctypes.data if bounds else None,
                             hi_b.ctypes.data if bounds else None)
        if timing is not None:
            timing["compute_s"] = timing.get("compute_s", 0.0) + time.perf_counter() - tc
        ss = np.array([r[0] for r in rows], np.int64)
        jj = np.array([r[1] for r in rows], np.int64)
        o[ss, jj] = o_b
        a[ss, jj] = a_b
        if bounds:
            dlo[ss, jj] = dl_b
            dhi[ss, jj] = dh_b
            nflag[ss, jj] = nf_b
            a_lo[ss, jj] = lo_b
            a_hi[ss, jj] = hi_b
        del mats
    if I is None:   # no tokens sampled
        I = 0
        o = np.empty((0, k, H), np.float32)
        a = np.empty((0, k, 0), np.uint16)
    ws = np.ascontiguousarray(w[tokens], dtype=np.float32)
    y = np.empty((ns, H), np.uint16)
    out = {}
    tc = time.perf_counter()
    if bounds:
        y32 = np.empty((ns, H), np.float32)
        ylo = np.empty((ns, H), np.float64)
        yhi = np.empty((ns, H), np.float64)
        L.oracle_combine(H, k, ns, ws.ctypes.data, o.ctypes.data, dlo.ctypes.data, dhi.ctypes.data, y.ctypes.data,
                         y32.ctypes.data, ylo.ctypes.data, yhi.ctypes.data)
        out.update(y32=y32, ylo=ylo, yhi=yhi, nflag=nflag, a_lo=a_lo, a_hi=a_hi)
    else:
        L.oracle_combine(H, k, ns, ws.ctypes.data, o.ctypes.data, None, None, y.ctypes.data, None, None, None)
    if timing is not None:
        timing["compute_s"] = timing.get("compute_s", 0.0) + time.perf_counter() - tc
    out["y"] = y
    if want_intermediates:
        out["a"], out["o"] = a, o
    return out


def forward(x, Wr, bias, W1, W2, k: int, act: int = ACT_SWIGLU, tokens=None,
            logits=None, want_intermediates: bool = False, bounds: bool = False,
            experts_per_batch: int = 16, timing=None) -> dict:
    """The whole layer on host arrays.  ``W1``/``W2`` are [E,H,2I]/[E,I,H] arrays or
    callables e -> per-expert matrix (each called once per expert the sample touches,
    ``experts_per_batch`` experts held at a time).  ``logits`` given: used instead of x*Wr.
    ``tokens``: which tokens get y (default all).  ``bounds``: also y32, ylo, yhi, nflag
    (see the module docstring).  ``timing`` (a dict): receives compute_s, the seconds spent in
    the oracle's own arithmetic (fetching the expert weights is not counted)."""
    tc = time.perf_counter()
    if logits is None:
        logits = router_logits(x, Wr, bias)
    E = logits.shape[1]
    ids, w = topk(logits, k)
    counts, offsets, row_pair, row_of = dispatch(ids, E)
    if timing is not None:
        timing["compute_s"] = timing.get("compute_s", 0.0) + time.perf_counter() - tc
    T = x.shape[0]
    if tokens is None:
        tokens = np.arange(T, dtype=np.int64)
    W1_of = W1 if callable(W1) else (lambda e: W1[e])
    W2_of = W2 if callable(W2) else (lambda e: W2[e])
    res = _forward_by_expert(x, ids, w, tokens, W1_of, W2_of, act, bounds, want_intermediates,
                             experts_per_batch, timing)
    out = dict(logits=logits, ids=ids, w=w, counts=counts, offsets=offsets,
               row_pair=row_pair, row_of=row_of, tokens=np.asarray(tokens, np.int64))
    out.update(res)
    return out
