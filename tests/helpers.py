"""Shared helpers of the GPU tests: inputs (seeded, from synth), the oracle's
expectations, and the output tolerance.

Tolerance on y (bf16): the stated bounds max |y - y_ref| <= 2e-2 * RMS(y_ref) and
|y - y_ref| <= 3e-2 * |y_ref| where |y_ref| > 0.1 * RMS(y_ref), read as follows.
Every expectation comes from the oracle and the inputs alone; no GPU intermediate
decides whether y passes.

* Before rounding.  Both sides round their fp32 sum to bf16 once, so the bounds are
  applied to the values before that rounding: the GPU's y stands for any value that
  rounds to it (within half a bf16 spacing of it), and the oracle's for its fp32 sum
  y32.  Without this reading two fp32 sums a hair apart that straddle a bf16
  rounding boundary would fail the absolute bound wherever one bf16 spacing exceeds
  2e-2 * RMS (|y| above 2.56 RMS).
* Rounding of the intermediate.  h = bf16(silu(g) * u) is rounded from fp32
  accumulations whose order the page leaves open.  The oracle flags every element
  that lies within its stated accumulation-error bound of a bf16 rounding boundary
  and carries the flagged elements' other roundings through its Linear-2 and
  Combine as an interval [ylo, yhi] of y around y32 (oracle.forward(bounds=True)).
  The distance from the GPU's y to that interval is what the bounds limit.  Where
  nothing is flagged the interval is the single value y32.

So, per element, d = max(0, dist(y_gpu, [ylo, yhi]) - spacing(y_gpu) / 2), and
d <= 2e-2 * RMS(y_ref) everywhere, d <= 3e-2 * |y_ref| where |y_ref| > 0.1 * RMS.
check_h_in_range checks the other side of the flags: every element of the GPU's own
h must lie in the oracle's range [a_lo, a_hi] (equal to the oracle's h where nothing
is flagged).

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
    """Spacing of bf16 numbers at |v| (8 significant bits; 2^-133 at zero and below
    the normal range)."""
    _, e = np.frexp(np.abs(v))
    return np.where(v == 0, 2.0 ** -133, np.ldexp(1.0, np.maximum(e - 8, -133)))


def _sub(a, rows):
    return a if rows is None else a[rows]


def check_y(y_gpu_bits: np.ndarray, ref: dict, what: str = "y", rows=None) -> dict:
    """y of the GPU against the oracle's result ``ref`` (oracle.forward(..., bounds=True)),
    optionally on the rows ``rows`` of both (see the module docstring for the rule)."""
    yr_bits = _sub(ref["y"], rows)
    yg = f64(y_gpu_bits)
    yr = f64(yr_bits)
    lo = _sub(ref["ylo"], rows).astype(np.float64)
    hi = _sub(ref["yhi"], rows).astype(np.float64)
    y32 = _sub(ref["y32"], rows).astype(np.float64)
    assert yg.shape == yr.shape == lo.shape, f"{what}: shapes {yg.shape} vs {yr.shape}"
    assert np.all(np.isfinite(yg)), f"{what}: non-finite outputs"
    assert np.all(lo <= y32) and np.all(y32 <= hi), "oracle interval does not hold its own y32"
    rms = float(np.sqrt(np.mean(yr ** 2)))
    dist = np.maximum(lo - yg, 0.0) + np.maximum(yg - hi, 0.0)
    d = np.maximum(dist - 0.5 * bf16_ulp(yg), 0.0)
    worst = int(np.argmax(d))
    assert d.max() <= 2e-2 * rms, (f"{what}: |dy| {d.max():.3e} above 2e-2 * RMS ({2e-2 * rms:.3e}) at flat "
                                   f"index {worst}: gpu {yg.flat[worst]:.6g}, oracle {yr.flat[worst]:.6g} "
                                   f"[{lo.flat[worst]:.6g}, {hi.flat[worst]:.6g}]")
    big = np.abs(yr) > 0.1 * rms
    rel = d[big] / np.abs(yr[big])
    if rel.size:
        i = int(np.argmax(rel))
        assert rel.max() <= 3e-2, (f"{what}: relative error {rel.max():.3e} above 3e-2: gpu "
                                   f"{yg[big][i]:.6g}, oracle {yr[big][i]:.6g} [{lo[big][i]:.6g}, {hi[big][i]:.6g}]")
    # diagnostics: the same comparison without either reading
    strict = np.abs(yg - yr)
    srel = strict[big] / np.abs(yr[big]) if rel.size else np.zeros(0)
    return dict(max_abs=float(strict.max()), rms=rms, max_rel=float(srel.max()) if srel.size else 0.0,
                n_strict_abs_over=int((strict > 2e-2 * rms).sum()), n_strict_rel_over=int((srel > 3e-2).sum()),
                n_elems=int(yg.size), n_interval=int((hi > lo).sum()))


def check_h_in_range(h_gpu_bits: np.ndarray, ref: dict, what: str = "h") -> dict:
    """Every element of the GPU's intermediate (compact row order [T*k, I], as
    moe_debug_intermediates returns it) within the oracle's range [a_lo, a_hi] of its
    (token, slot); ``ref`` from oracle.forward(tokens=all, bounds=True,
    want_intermediates=True).  Returns how many elements differ from the oracle's h."""
    T, k, I = ref["a"].shape
    assert T * k == h_gpu_bits.shape[0], "ref must cover every token"
    hg = f64(h_gpu_bits)[ref["row_of"].reshape(T, k)]        # [T, k, I]
    lo, hi, a = f64(ref["a_lo"]), f64(ref["a_hi"]), f64(ref["a"])
    fin = np.isfinite(a)
    out = fin & ((hg < lo) | (hg > hi))
    if out.any():
        t, j, n = np.argwhere(out)[0]
        raise AssertionError(f"{what}: {int(out.sum())} elements outside the oracle's range, e.g. (t={t}, j={j}, "
                             f"n={n}): gpu {hg[t, j, n]:.6g}, range [{lo[t, j, n]:.6g}, {hi[t, j, n]:.6g}]")
    return dict(n_diff=int((fin & (hg != a)).sum()), n_flagged=int((fin & (hi > lo)).sum()), n=int(fin.sum()))


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
               full_weights=None, want_intermediates=False, weights_of=None):
    """Oracle on a workload: routing for all tokens, y (with its interval) for ``tokens``.
    Expert weights come from ``full_weights`` (host arrays), from ``weights_of(which, e)``,
    or else from the host generator (per expert slice)."""
    if full_weights is not None:
        W1, W2 = full_weights
    else:
        get = weights_of or (lambda which, e: synth.expert_slice_host(wl, which, e))
        W1 = lambda e: get("W1", e)   # noqa: E731
        W2 = lambda e: get("W2", e)   # noqa: E731
    return oracle.forward(x_bits, Wr_bits, bias, W1, W2, wl.k, act=act, tokens=tokens,
                          want_intermediates=want_intermediates, bounds=True)


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
                 rows=None, max_ratio: float = 0.25) -> dict:
    """Default router: every selected expert's logit bit-exact, every other entry exact or
    within logit_bound; the observed estimate error must stay under max_ratio of the bound
    (by default a quarter: the bound carries a wide margin over the tensor-core accumulation
    error on ordinary inputs)."""
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
    assert ratio.max() <= max_ratio, f"estimate error {ratio.max():.3f} of the stated bound"
    return dict(exact_frac=float(exact.mean()), max_ratio=float(ratio.max()))
