"""Pins for the CPU oracle: each test checks it against something other than itself.

The layer is the MoE layer of the X-Stage paper's MegaMoE background paragraph
(router top-k, Dispatch, Linear-1, SwiGLU, Linear-2, Combine with router
weights).  Pins used here:

* library routines: torch's bf16 rounding, numpy's stable argsort / lexsort,
  scipy's softmax, numpy int64 matrix products;
* closed forms: exactly representable sums, identity experts in the linear
  regime of SiLU, k = 1, k = E, all-equal logits;
* hand-derived values that distinguish the canonical router summation order
  from every other plausible order;
* a brute-force dense evaluation (every token through every expert, masked).
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def bf16_bits(a):
    """float array -> bf16 bit patterns via torch (library rounding)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return oracle.bf16_to_f32(b).astype(np.float64)


# --------------------------------------------------------------------------- bf16
def test_bf16_rounding_matches_torch():
    vals = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32),
        (RNG.standard_normal(2000) * 1e30).astype(np.float32),
        (RNG.standard_normal(2000) * 1e-38).astype(np.float32),      # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38], np.float32),
        # exact halfway cases: bf16 value + half an ulp
        (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        (np.arange(1, 200, dtype=np.uint32) << 16 | 0x7FFF).view(np.float32),
    ])
    assert np.array_equal(oracle.f32_to_bf16(vals), bf16_bits(vals))
    nan = oracle.f32_to_bf16(np.array([np.nan, -np.nan], np.float32))
    assert np.all(np.isnan(oracle.bf16_to_f32(nan)))


# --------------------------------------------------------------------------- router logits
def test_router_logits_exact_on_integers():
    T, H, E = 7, 96, 5
    x = RNG.integers(-3, 4, size=(T, H))
    Wr = RNG.integers(-3, 4, size=(H, E))
    exact = x.astype(np.int64) @ Wr.astype(np.int64)          # every sum < 2^24: fp32-exact
    got = oracle.router_logits(bf16_bits(x), bf16_bits(Wr))
    assert np.array_equal(got, exact.astype(np.float32))
    bias = RNG.integers(-5, 6, size=E).astype(np.float32)
    got_b = oracle.router_logits(bf16_bits(x), bf16_bits(Wr), bias)
    assert np.array_equal(got_b, (exact + bias).astype(np.float32))


def _one_token_logit(terms):
    """Build x, Wr (H=64, E=1) whose products x[h]*Wr[h] equal ``terms`` (powers of 2)."""
    H = 64
    x = np.zeros((1, H), np.float32)
    w = np.zeros((H, 1), np.float32)
    for h, v in terms.items():
        x[0, h] = np.float32(2.0 ** 12) if abs(v) >= 2 ** 12 else np.float32(1.0)
        w[h, 0] = v / x[0, h]
    return oracle.router_logits(bf16_bits(x), bf16_bits(w))[0, 0]


def test_router_logits_canonical_order_lane_strided():
    # h=0 and h=32 fall in the same residue class (partial 0), h=16 in partial 16.
    # Lane-strided: p0 = 2^24 - 2^24 = 0, p16 = 1, tree -> 1.
    # A plain sequential sum gives (2^24 + 1) rounds to 2^24, then 0.
    assert _one_token_logit({0: 2.0 ** 24, 16: 1.0, 32: -(2.0 ** 24)}) == 1.0


def test_router_logits_canonical_order_tree():
    # p0 = 2^24, p1 = 1, p16 = -2^24.  Tree level 1 pairs (0,16) -> 0 and (1,17) -> 1,
    # total 1.  Summing the 32 partials left to right gives 2^24 + 1 -> 2^24, then 0.
    assert _one_token_logit({0: 2.0 ** 24, 1: 1.0, 16: -(2.0 ** 24)}) == 1.0
    # p0 = 2^24, p8 = 1, p16 = -2^24: level 1 gives p0 = 0, p8 = 1; total 1.
    # Pairing adjacent partials first, (0,1),(2,3).., gives ((2^24 + 0) + ... + 1) ordering
    # that loses the 1 when it meets 2^24 before -2^24 does.
    assert _one_token_logit({0: 2.0 ** 24, 8: 1.0, 16: -(2.0 ** 24)}) == 1.0


def test_router_logits_error_bound_random():
    T, H, E = 16, 512, 16
    x = bf16_bits(RNG.standard_normal((T, H)))
    Wr = bf16_bits(RNG.standard_normal((H, E)) / np.sqrt(H))
    got = oracle.router_logits(x, Wr).astype(np.float64)
    xf, wf = bits_to_f64(x), bits_to_f64(Wr)
    exact = xf @ wf
    mag = np.abs(xf) @ np.abs(wf)
    depth = H // 32 + 5                      # roundings a term passes through
    assert np.all(np.abs(got - exact) <= depth * 2.0 ** -24 * mag * 1.01)


# --------------------------------------------------------------------------- top-k
def _lexsort_topk(logits, k):
    T, E = logits.shape
    out = np.empty((T, k), np.int32)
    for t in range(T):
        key = np.where(np.isnan(logits[t]), -np.inf, logits[t]).astype(np.float64)
        nanrank = np.isnan(logits[t]).astype(np.int64)       # NaN after every number
        order = np.lexsort((np.arange(E), -key, nanrank))
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("E,k", [(8, 2), (16, 4), (128, 8), (256, 8)])
def test_topk_matches_lexsort_with_ties(E, k):
    T = 300
    logits = RNG.integers(-4, 5, size=(T, E)).astype(np.float32) * np.float32(0.5)
    ids, w = oracle.topk(logits, k)
    assert np.array_equal(ids, _lexsort_topk(logits, k))
    sel = np.take_along_axis(logits, ids, 1).astype(np.float64)
    ref = np.exp(sel - sel[:, :1])
    ref /= ref.sum(1, keepdims=True)
    assert np.allclose(w, ref, rtol=1e-6, atol=0)


def test_topk_special_cases():
    from scipy.special import softmax
    T, E = 64, 16
    logits = RNG.standard_normal((T, E)).astype(np.float32)
    ids, w = oracle.topk(logits, 1)
    assert np.all(w == 1.0) and np.array_equal(ids[:, 0], np.argmax(logits, 1))
    ids, w = oracle.topk(logits, E)                      # k = E: renormalised = full softmax
    full = softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(full, ids, 1), rtol=1e-6)
    eq = np.full((4, E), 0.25, np.float32)               # all equal -> 0..k-1, w = 1/k
    ids, w = oracle.topk(eq, 5)
    assert np.array_equal(ids, np.tile(np.arange(5), (4, 1)))
    assert np.allclose(w, 0.2, rtol=2 ** -23, atol=0)
    odd = np.array([[np.nan, -np.inf, 1.0, np.nan, -0.0, 0.0]], np.float32)
    ids, _ = oracle.topk(odd, 6)                         # -0 == +0 -> lower id; NaN last
    assert ids.tolist() == [[2, 4, 5, 1, 0, 3]]


def test_topk_invariants_random():
    T, E, k = 500, 128, 8
    logits = RNG.standard_normal((T, E)).astype(np.float32)
    ids, w = oracle.topk(logits, k)
    for t in range(T):
        assert len(set(ids[t])) == k
        sel = logits[t, ids[t]]
        rest = np.delete(logits[t], ids[t])
        assert sel.min() >= rest.max()
        assert np.all(np.diff(sel) <= 0)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 4 * 2.0 ** -23)


# --------------------------------------------------------------------------- Dispatch
def test_dispatch_matches_stable_argsort():
    T, E, k = 1000, 32, 4
    logits = RNG.standard_normal((T, E)).astype(np.float32)
    ids, _ = oracle.topk(logits, k)
    counts, offsets, row_pair, row_of = oracle.dispatch(ids, E)
    flat = ids.ravel()
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(row_pair, np.argsort(flat, kind="stable"))
    assert np.array_equal(row_of[row_pair], np.arange(T * k))
    tok = row_pair // k
    assert np.array_equal(np.bincount(tok, minlength=T), np.full(T, k))
    for e in range(E):
        seg = tok[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)                  # ascending token within an expert


# --------------------------------------------------------------------------- expert FFN + Combine
def _tiny_layer(T, H, I, E, k, dist="normal"):
    if dist == "normal":
        x = bf16_bits(RNG.standard_normal((T, H)))
        Wr = bf16_bits(RNG.standard_normal((H, E)) / np.sqrt(H))
        W1 = bf16_bits(RNG.standard_normal((E, H, 2 * I)) / np.sqrt(H))
        W2 = bf16_bits(RNG.standard_normal((E, I, H)) / np.sqrt(I))
    else:  # sparse integers in {-1, 0, 1}
        def tern(shape, p):
            return (RNG.random(shape) < p) * RNG.choice([-1.0, 1.0], size=shape)
        x = bf16_bits(tern((T, H), 0.5))
        Wr = bf16_bits(RNG.standard_normal((H, E)) / np.sqrt(H))
        W1 = bf16_bits(tern((E, H, 2 * I), 0.25))
        W2 = bf16_bits(tern((E, I, H), 0.25))
    return x, Wr, W1, W2


def test_bilinear_integer_exact():
    """Integer inputs: every dot product is exact; a = bf16(g*u) is a library rounding."""
    T, H, I, E, k = 24, 64, 32, 4, 2
    x, Wr, W1, W2 = _tiny_layer(T, H, I, E, k, dist="int")
    res = oracle.forward(x, Wr, None, W1, W2, k, act=oracle.ACT_BILINEAR, want_intermediates=True)
    xi = bits_to_f64(x).astype(np.int64)
    W1i = bits_to_f64(W1).astype(np.int64)
    W2i = bits_to_f64(W2).astype(np.int64)
    for t in range(T):
        for j in range(k):
            e = res["ids"][t, j]
            gu = xi[t] @ W1i[e]                                  # [2I] exact
            g, u = gu[:I], gu[I:]
            assert np.all(np.abs(g * u) < 2 ** 24)
            a = bf16_bits((g * u).astype(np.float32))
            assert np.array_equal(bits_to_f64(res["a"][t, j]), bits_to_f64(a))  # -0 == +0
            af = bits_to_f64(a)
            assert np.all(np.abs(af) @ np.abs(W2i[e]) < 2 ** 24)  # every partial sum exact
            o = af @ W2i[e]
            assert np.array_equal(res["o"][t, j], o.astype(np.float32))


def test_dense_masked_bruteforce():
    """Every token through every expert in fp64, masked by the routing weights."""
    T, H, I, E, k = 40, 64, 32, 6, 3
    x, Wr, W1, W2 = _tiny_layer(T, H, I, E, k)
    res = oracle.forward(x, Wr, None, W1, W2, k)
    xf, W1f, W2f = bits_to_f64(x), bits_to_f64(W1), bits_to_f64(W2)
    gu = np.einsum("th,ehn->ten", xf, W1f)                       # [T,E,2I]
    g, u = gu[..., :I], gu[..., I:]
    a = g / (1.0 + np.exp(-g)) * u
    a = bits_to_f64(bf16_bits(a))                                # the intermediate is bf16
    o = np.einsum("tei,eih->teh", a, W2f)                        # [T,E,H]
    mask = np.zeros((T, E))
    for t in range(T):
        mask[t, res["ids"][t]] = res["w"][t]
    y_ref = np.einsum("te,teh->th", mask, o)
    y = bits_to_f64(res["y"])
    rms = np.sqrt(np.mean(y_ref ** 2))
    # y is rounded to bf16 (half an ulp <= 2^-8 |y|); the intermediate's bf16 rounding may
    # differ by one ulp between fp32 and fp64 accumulation.  A wrong token<->row mapping,
    # a dropped slot or a wrong weight is off by O(rms), far outside this bound.
    assert np.all(np.abs(y - y_ref) <= 2.0 ** -8 * np.abs(y_ref) + 5e-3 * rms)


@pytest.mark.parametrize("scaled", [False, True])
def test_identity_experts_closed_form(scaled):
    """W1 gate = 4*Id, up = c_e*Id, W2 = Id, x in [2,4]: y = 4 x^2 sum_j w_j c_{e_j}
    up to SiLU's linear-regime deviation (< e^-8) and bf16 roundings."""
    T, H, E, k = 32, 64, 4, 2
    I = H
    x = bf16_bits(2.0 + 2.0 * RNG.random((T, H)))
    Wr = bf16_bits(RNG.standard_normal((H, E)) / np.sqrt(H))
    c = np.arange(1, E + 1, dtype=np.float64) if scaled else np.ones(E)
    W1 = np.zeros((E, H, 2 * I), np.float32)
    W2 = np.zeros((E, I, H), np.float32)
    for e in range(E):
        W1[e, :, :I] = 4.0 * np.eye(H)
        W1[e, :, I:] = c[e] * np.eye(H)
        W2[e] = np.eye(H)
    res = oracle.forward(x, Wr, None, bf16_bits(W1), bf16_bits(W2), k)
    xf = bits_to_f64(x)
    cw = (res["w"] * c[res["ids"]]).sum(1)
    expect = 4.0 * xf ** 2 * cw[:, None]
    y = bits_to_f64(res["y"])
    assert np.all(np.abs(y / expect - 1.0) <= 3 * 2.0 ** -8)


def test_oracle_matches_its_regression_record():
    """The oracle on the seeded tiny workload equals the record tests/golden/make_golden.py
    wrote (a change detector for the oracle and the generator, not a pin: see the README
    there).  A deliberate change to the oracle's arithmetic is rerecorded with that script."""
    import importlib.util
    import json
    import os
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(here, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    with open(os.path.join(here, "oracle_tiny.json")) as f:
        want = json.load(f)
    assert mg.record() == want


# --------------------------------------------------------------------------- rounding flags of h
def _one_expert(x_vals, gate, up, H=32):
    """One token through one expert with I = 1: x[:len(x_vals)] = x_vals (rest 0), the gate
    and up columns given (rest 0).  Returns x row, W1e [H, 2] (bf16 bits)."""
    x = np.zeros(H, np.float32)
    x[:len(x_vals)] = x_vals
    W1 = np.zeros((H, 2), np.float32)
    W1[:len(gate), 0] = gate
    W1[:len(up), 1] = up
    xb, wb = bf16_bits(x), bf16_bits(W1)
    assert np.array_equal(bits_to_f64(xb), x) and np.array_equal(bits_to_f64(wb), W1)   # exact in bf16
    return xb, wb


@pytest.mark.parametrize("delta,flagged", [(0.0, True), (2.0 ** -23, True), (-(2.0 ** -23), True),
                                           (2.0 ** -16, False), (-(2.0 ** -16), False)])
def test_h_range_on_a_rounding_boundary(delta, flagged):
    """Bilinear g * u with u = 1 and g = 1 + 2^-8 + delta.  delta = 0 is exactly halfway between
    the bf16 values 1 and 1 + 2^-7 (round-to-even gives 1): any other accumulation order may
    give either, so both are in the range.  2^-23 away is inside the stated radius (about
    2^-22 here), 2^-16 away is far outside it: only the nearest value remains."""
    terms = [1.0, 2.0 ** -8] + ([abs(delta)] if delta else [])
    gate = [1.0, 1.0] + ([np.sign(delta)] if delta else [])
    xb, wb = _one_expert(terms, gate, [1.0])
    lo, hi, g, rad = oracle.expert_h_range(xb, wb, act=oracle.ACT_BILINEAR)
    a, _ = oracle.expert_ffn(xb, wb, np.zeros((1, 32), np.uint16), act=oracle.ACT_BILINEAR)
    assert g[0] == 1.0 + 2.0 ** -8 + delta and g[1] == 1.0              # exact sums
    assert 2.0 ** -23 < rad[0] < 2.0 ** -20
    one, up1 = 0x3F80, 0x3F81                                            # bf16 1.0 and 1 + 2^-7
    nearest = one if delta <= 0 else up1
    assert a[0] == nearest
    if flagged:
        assert (lo[0], hi[0]) == (one, up1)
    else:
        assert lo[0] == hi[0] == nearest


def test_h_range_brackets_every_evaluation_within_the_radius():
    """SwiGLU on random inputs: for every element, silu(g') * u' evaluated in float64 at g', u'
    anywhere in the stated radius (endpoints and random interior points) rounds to a bf16 value
    inside [a_lo, a_hi], and the range always holds the oracle's own a."""
    H, I = 512, 64
    rng = np.random.default_rng(77)
    x = bf16_bits(rng.standard_normal(H).astype(np.float32))
    W1 = bf16_bits((rng.standard_normal((H, 2 * I)) / np.sqrt(H)).astype(np.float32))
    W2 = np.zeros((I, H), np.uint16)
    lo, hi, g, rad = oracle.expert_h_range(x, W1)
    a, _ = oracle.expert_ffn(x, W1, W2)
    flo, fhi, fa = bits_to_f64(lo), bits_to_f64(hi), bits_to_f64(a)
    assert np.all(flo <= fa) and np.all(fa <= fhi)
    gg, uu = g[:I], g[I:]
    rg, ru = rad[:I], rad[I:]
    for t in np.concatenate([[-1.0, 1.0], rng.uniform(-1, 1, 30)]):
        for s in (-1.0, 1.0, rng.uniform(-1, 1)):
            gv = gg + t * rg
            uv = uu + s * ru
            v = gv / (1.0 + np.exp(-gv)) * uv
            b = bits_to_f64(bf16_bits(v.astype(np.float32)))
            assert np.all((flo <= b) & (b <= fhi))


def test_h_range_exact_sums_and_silu_minimum():
    """The range's g, u are the exact sums (checked with rational arithmetic) and the constant
    minimum of silu the range uses is silu's minimum (scipy)."""
    from fractions import Fraction
    from scipy.optimize import minimize_scalar
    H, I = 64, 3
    rng = np.random.default_rng(5)
    x = bf16_bits(rng.standard_normal(H).astype(np.float32) * 3)
    W1 = bf16_bits(rng.standard_normal((H, 2 * I)).astype(np.float32) * 1e-3)
    _, _, g, _ = oracle.expert_h_range(x, W1)
    xf, wf = bits_to_f64(x), bits_to_f64(W1)
    for n in range(2 * I):
        exact = sum(Fraction(float(xf[h])) * Fraction(float(wf[h, n])) for h in range(H))
        assert abs(Fraction(float(g[n])) - exact) <= Fraction(2.0 ** -52) * abs(exact) + Fraction(2.0 ** -80)
    m = minimize_scalar(lambda z: z / (1 + np.exp(-z)), bracket=(-3, -1, 0), tol=1e-14)
    src = open(oracle.__file__.replace("__init__.py", "moe_oracle.c")).read()
    const = float(src.split("#define O_SILU_XMIN (")[1].split(")")[0])
    assert abs(const - m.x) < 1e-7


def test_y_interval_equals_enumeration_of_flips():
    """The oracle's [ylo, yhi] against brute force: every combination of the flagged intermediates'
    extreme roundings (plus the oracle's own) carried through Linear-2 and Combine in float64;
    the interval's ends must be the smallest and largest results."""
    H, I, E, k = 512, 48, 4, 2
    rng = np.random.default_rng(9)
    x = bf16_bits(rng.standard_normal((40, H)).astype(np.float32))
    W1 = bf16_bits((rng.standard_normal((E, H, 2 * I)) / np.sqrt(H)).astype(np.float32))
    W2 = bf16_bits((rng.standard_normal((E, I, H)) / np.sqrt(I)).astype(np.float32))
    Wr = bf16_bits((rng.standard_normal((H, E)) / np.sqrt(H)).astype(np.float32))
    ref = oracle.forward(x, Wr, None, W1, W2, k, bounds=True, want_intermediates=True)
    f = ref["nflag"].sum(axis=1)
    cand = [t for t in range(40) if 2 <= f[t] <= 9]
    assert cand, "no token with a handful of flagged elements"
    for t in cand[:3]:
        slots = []
        for j in range(k):
            e = ref["ids"][t, j]
            a = bits_to_f64(ref["a"][t, j])
            lo, hi = bits_to_f64(ref["a_lo"][t, j]), bits_to_f64(ref["a_hi"][t, j])
            fl = np.nonzero((lo != a) | (hi != a))[0]
            slots += [(j, e, n, lo[n] - a[n], hi[n] - a[n]) for n in fl]
        dmin = np.full(H, np.inf)
        dmax = np.full(H, -np.inf)
        for mask in range(3 ** len(slots)):
            d = np.zeros(H)
            mm = mask
            for (j, e, n, dl, dh) in slots:
                c = (0.0, dl, dh)[mm % 3]
                mm //= 3
                d += float(ref["w"][t, j]) * c * bits_to_f64(W2[e, n])
            dmin, dmax = np.minimum(dmin, d), np.maximum(dmax, d)
        y32 = ref["y32"][t].astype(np.float64)
        assert np.allclose(ref["ylo"][t] - y32, dmin, rtol=1e-12, atol=1e-15)
        assert np.allclose(ref["yhi"][t] - y32, dmax, rtol=1e-12, atol=1e-15)
        assert np.array_equal(oracle.f32_to_bf16(ref["y32"][t]), ref["y"][t])


def test_expert_driven_forward_equals_token_driven():
    """oracle.forward (expert by expert, batched) against oracle_forward_tokens (token by token):
    the same arithmetic, so y, h and o bit for bit."""
    H, I, E, k, T = 256, 128, 9, 3, 50
    rng = np.random.default_rng(10)
    x = bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    W1 = bf16_bits((rng.standard_normal((E, H, 2 * I)) / np.sqrt(H)).astype(np.float32))
    W2 = bf16_bits((rng.standard_normal((E, I, H)) / np.sqrt(I)).astype(np.float32))
    Wr = bf16_bits((rng.standard_normal((H, E)) / np.sqrt(H)).astype(np.float32))
    ref = oracle.forward(x, Wr, None, W1, W2, k, want_intermediates=True, bounds=True, experts_per_batch=2)
    y, a, o = oracle.forward_tokens(x, ref["ids"], ref["w"], np.arange(T), lambda e: W1[e], lambda e: W2[e], E,
                                    want_intermediates=True)
    assert np.array_equal(ref["y"], y) and np.array_equal(ref["a"], a) and np.array_equal(ref["o"], o)
