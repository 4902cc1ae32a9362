"""Shared helpers of the GPU tests: inputs (seeded, from synth), the oracle's
expectations, and the output tolerance.

Tolerance on y (bf16), the stated bounds max |y - y_ref| <= 2e-2 * RMS(y_ref) and
|y - y_ref| <= 3e-2 * |y_ref| where |y_ref| > 0.1 * RMS(y_ref), read for bf16
outputs of a bf16-intermediate computation:

* absolute: every element within 2e-2 * RMS + ulp(y_ref).  Both sides round
  their fp32 result to bf16 independently, so nearly equal fp32 values can land
  on adjacent bf16 neighbours; above 2.56 * RMS one bf16 spacing already exceeds
  2e-2 * RMS.
* relative: every element above 0.1 * RMS within 3e-2, except at most
  ceil(1e-5 * n) of them, each within 6e-2.  The intermediate h is rounded to
  bf16 on both sides from fp32 values accumulated in different orders (tensor
  cores vs sequential); ~5e-4 of h elements round to a neighbouring bf16 value,
  and one such flip of a large |h| moves an output by ~0.5% of RMS, which is
  >3e-2 relative on the rare output near 0.1 * RMS that the top-k sum cancels.
* explained outliers (check_y_explained): where the GPU's h is available, elements
  beyond that allowance pass only if h explains them - every GPU h element within
  2e-2 * RMS(h) + ulp of the oracle's (the absolute rule of y, applied to h: near
  g = 0 the accumulation order alone moves silu(g) * u by many ulps, harmlessly),
  at most H * 2^-18 of them different at all (the share of fp32 sums close enough
  to a bf16 rounding boundary for the summation order to matter grows with the
  reduction length H: measured 5e-4 at H = 512 and 2.1e-3 at H = 2048, caps 2e-3
  and 7.8e-3), and y within the same tolerance of the oracle's Linear-2 and
  Combine applied to the GPU's h.
  With k = 1 nothing dilutes a flip: one flipped h element of a token moves its
  whole output row (measured: 7 of 127,037 elements at 3-4.5% relative, all in
  the row of the one token with a flipped element).

Routing (ids, counts, offsets, row_pair, row_of) must be bit-exact; router
weights within 1e-6 relative (the GPU's exp is not the host's).  Logits: with
MOE_FLAG_EXACT_LOGITS every entry is bit-exact; by default the entries of the
selected experts are bit-exact and every other entry is either exact or within
the library's stated bound of the canonical value (check_logits)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def f64(b: np.ndarray) -> np.ndarray:
    return oracle.bf16_to_f32(b).astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def check_y(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, what: str = "y"):
    yg, yr = f64(y_gpu_bits), f64(y_ref_bits)
    assert yg.shape == yr.shape
    rms = float(np.sqrt(np.mean(yr ** 2)))
    d = np.abs(yg - yr)
    assert np.all(np.isfinite(yg)), f"{what}: non-finite outputs"
    excess = d - (2e-2 * rms + bf16_ulp(yr))
    assert excess.max() <= 0, (f"{what}: |dy| {d.max():.3e} exceeds 2e-2 * rms ({2e-2 * rms:.3e}) "
                               f"+ ulp(y_ref) by {excess.max():.3e}")
    big = np.abs(yr) > 0.1 * rms
    rel = d[big] / np.abs(yr[big])
    n_over = int((rel > 3e-2).sum())
    allowed = int(np.ceil(1e-5 * rel.size))
    assert n_over <= allowed, f"{what}: {n_over} elements above 3e-2 relative (allowed {allowed} of {rel.size})"
    assert rel.size == 0 or rel.max() <= 6e-2, f"{what}: max rel err {rel.max():.3e} > 6e-2"
    return dict(max_abs=float(d.max()), rms=rms, max_rel=float(rel.max()) if rel.size else 0.0,
                n_rel_over=n_over)


def check_y_explained(y_gpu_bits: np.ndarray, ref: dict, h_gpu_bits: np.ndarray, W2_bits: np.ndarray,
                      what: str = "y"):
    """check_y against the oracle; outliers beyond its relative allowance are accepted only
    when the GPU's bf16 intermediate h explains them (see the module docstring).
    ref: the oracle's result with intermediates; h_gpu_bits: [T*k, I] in compact row order;
    W2_bits: [E, I, H]."""
    try:
        check_y(y_gpu_bits, ref["y"], what)
        return
    except AssertionError as first:
        failure = first
    T, k, I = ref["a"].shape
    row_of = ref["row_of"].reshape(T, k)
    hg = f64(h_gpu_bits)[row_of]                        # [T, k, I]
    ha = f64(ref["a"])
    dh = np.abs(hg - ha)
    rms_h = float(np.sqrt(np.mean(ha ** 2)))
    assert np.all(dh <= 2e-2 * rms_h + bf16_ulp(ha)), \
        f"{what}: h differs from the oracle's beyond 2e-2 * RMS(h) + ulp ({failure})"
    frac = float((dh != 0).mean())
    H = W2_bits.shape[2]
    cap = H * 2.0 ** -18          # grows with Linear-1's reduction length H (see the module docstring)
    assert frac <= cap, f"{what}: {frac:.2e} of h elements differ from the oracle's, above {cap:.2e} ({failure})"
    E, _, H = W2_bits.shape
    y_alt = np.zeros((T, H), dtype=np.float64)
    for e in np.unique(ref["ids"]):
        W2e = f64(W2_bits[e])                           # [I, H]
        for j in range(k):
            sel = np.nonzero(ref["ids"][:, j] == e)[0]
            if sel.size:
                y_alt[sel] += ref["w"][sel, j].astype(np.float64)[:, None] * (hg[sel, j, :] @ W2e)
    y_alt_bits = oracle.f32_to_bf16(y_alt.astype(np.float32))
    check_y(y_gpu_bits, y_alt_bits, what + " (from the GPU's h)")


def routing_equal(gpu: dict, ref: dict, T: int):
    ids = gpu["ids"].cpu().numpy()
    assert np.array_equal(ids, ref["ids"]), "ids differ"
    assert np.array_equal(gpu["counts"].cpu().numpy(), ref["counts"]), "counts differ"
    assert np.array_equal(gpu["offsets"].cpu().numpy(), ref["offsets"]), "offsets differ"
    assert np.array_equal(gpu["row_pair"].cpu().numpy(), ref["row_pair"]), "row_pair differs"
    assert np.array_equal(gpu["row_of"].cpu().numpy(), ref["row_of"]), "row_of differs"
    w = gpu["w"].cpu().numpy()
    assert np.allclose(w, ref["w"], rtol=1e-6, atol=1e-30, equal_nan=True), "router weights differ"


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    if n >= T:
        return np.arange(T, dtype=np.int64)
    rng = np.random.default_rng(seed)
    s = rng.choice(T, size=n, replace=False)
    s[0], s[-1] = 0, T - 1
    return np.sort(s).astype(np.int64)


def oracle_for(wl: synth.Workload, x_bits: np.ndarray, Wr_bits: np.ndarray, bias, tokens, act=0,
               full_weights=None, want_intermediates=False):
    """Oracle on a workload: routing for all tokens, y for ``tokens``.  Expert weights
    come from the host generator (per expert slice) unless ``full_weights`` is given."""
    if full_weights is not None:
        W1, W2 = full_weights
    else:
        W1 = lambda e: synth.expert_slice_host(wl, "W1", e)   # noqa: E731
        W2 = lambda e: synth.expert_slice_host(wl, "W2", e)   # noqa: E731
    return oracle.forward(x_bits, Wr_bits, bias, W1, W2, wl.k, act=act, tokens=tokens,
                          want_intermediates=want_intermediates)


def logit_bound(x_bits: np.ndarray, Wr_bits: np.ndarray, bias, est: np.ndarray, cH: float) -> np.ndarray:
    """The library's stated bound on |estimate - canonical logit| per (t, e), in float64:
    cH ||x_t|| ||Wr[:,e]|| + 2^-20 (|v| + |b|), v = estimate - bias (cH from moe_router_bound)."""
    x = f64(x_bits)
    Wr = f64(Wr_bits)
    nx = np.sqrt((x * x).sum(axis=1))
    nw = np.sqrt((Wr * Wr).sum(axis=0))
    b = np.zeros(Wr.shape[1]) if bias is None else np.abs(np.asarray(bias, np.float64))
    return cH * np.outer(nx, nw) + 2.0 ** -20 * (np.abs(est.astype(np.float64)) + 2 * b[None, :])


def check_logits(lg_gpu: np.ndarray, ref: dict, x_bits: np.ndarray, Wr_bits: np.ndarray, cH: float, bias=None,
                 rows=None) -> dict:
    """Default router: every selected expert's logit bit-exact, every other entry exact or
    within logit_bound; the observed estimate error must stay under a quarter of the bound
    (the bound carries a wide margin over the tensor-core accumulation error)."""
    ref_l = ref["logits"]
    ids = ref["ids"]
    if rows is not None:
        lg_gpu, ref_l, ids, x_bits = lg_gpu[rows], ref_l[rows], ids[rows], x_bits[rows]
    sel = np.take_along_axis(lg_gpu, ids, axis=1)
    assert np.array_equal(sel.view(np.uint32), np.take_along_axis(ref_l, ids, axis=1).view(np.uint32)), \
        "selected logits not bit-exact"
    exact = lg_gpu.view(np.uint32) == ref_l.view(np.uint32)
    d = np.abs(lg_gpu.astype(np.float64) - ref_l.astype(np.float64))
    bound = logit_bound(x_bits, Wr_bits, bias, lg_gpu, cH)
    ratio = np.where(exact, 0.0, d / bound)
    assert np.all(np.isfinite(lg_gpu[~exact])), "non-finite estimate"
    assert ratio.max() <= 0.25, f"estimate error {ratio.max():.3f} of the stated bound"
    return dict(exact_frac=float(exact.mean()), max_ratio=float(ratio.max()))
