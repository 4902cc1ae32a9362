"""The y acceptance rule of the GPU tests (helpers.check_y), pinned on the CPU against the
oracle's own results: it accepts the oracle's y, rejects an output beyond the absolute or
the relative bound, uses the flip interval only as far as it reaches, and reads each side's
final bf16 rounding as at most half a bf16 spacing of the GPU's value."""
import numpy as np
import pytest

import helpers
import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.fixture(scope="module")
def ref():
    synth.build_host()
    oracle.build()
    wl = synth.Workload("tol", 48, 512, 128, 6, 2)
    h = synth.host_inputs(wl)
    return helpers.oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]),
                              want_intermediates=True)


def _f(b):
    return helpers.f64(b)


def _bits(v):
    return oracle.f32_to_bf16(np.asarray(v, np.float32))


def _rms(ref):
    return float(np.sqrt(np.mean(_f(ref["y"]) ** 2)))


def test_accepts_the_oracle_itself(ref):
    st = helpers.check_y(ref["y"], ref)
    assert st["n_strict_abs_over"] == 0 and st["n_strict_rel_over"] == 0


def test_rejects_absolute_error(ref):
    """The largest element moved by the bound plus one and a half bf16 spacings."""
    y = _f(ref["y"]).copy()
    i = np.unravel_index(np.argmax(np.abs(y)), y.shape)
    y[i] += 2e-2 * _rms(ref) + 1.5 * helpers.bf16_ulp(np.array([y[i]]))[0]
    with pytest.raises(AssertionError, match="above 2e-2"):
        helpers.check_y(_bits(y), ref)


def test_rejects_relative_error_within_the_absolute_bound(ref):
    """An element near 0.2 RMS off by 6% of itself: 1.2% of RMS, inside the absolute bound,
    outside the relative one (its interval is a single value)."""
    y = _f(ref["y"]).copy()
    rms = _rms(ref)
    cand = np.argwhere((np.abs(y) > 0.15 * rms) & (np.abs(y) < 0.25 * rms) & (ref["yhi"] == ref["ylo"]))
    assert len(cand)
    i = tuple(cand[0])
    y[i] *= 1.06
    with pytest.raises(AssertionError, match="relative error"):
        helpers.check_y(_bits(y), ref)


def test_interval_is_used_only_as_far_as_it_reaches(ref):
    """Widen one element's interval by hand: a GPU value at the far end passes; the same value
    against the unwidened interval fails, and so does a value beyond the widened end plus the
    tolerance."""
    rms = _rms(ref)
    y = _f(ref["y"])
    i = tuple(np.argwhere(np.abs(y) > 0.5 * rms)[0])
    wide = {kk: (v.copy() if isinstance(v, np.ndarray) else v) for kk, v in ref.items()}
    span = 0.2 * abs(y[i])
    wide["yhi"][i] += span
    ok = y.copy()
    ok[i] = float(wide["yhi"][i])
    helpers.check_y(_bits(ok), wide)
    with pytest.raises(AssertionError):
        helpers.check_y(_bits(ok), ref)
    bad = y.copy()
    bad[i] = float(wide["yhi"][i]) + 0.05 * abs(y[i]) + 2e-2 * rms
    with pytest.raises(AssertionError):
        helpers.check_y(_bits(bad), wide)


def test_final_rounding_allowance_is_half_a_spacing(ref):
    """A large element whose oracle sum y32 lies next to a bf16 rounding boundary: the GPU's
    y on the other side of that boundary (one spacing away, more than 2e-2 * RMS) passes,
    two spacings away fails."""
    rms = _rms(ref)
    wide = {kk: (v.copy() if isinstance(v, np.ndarray) else v) for kk, v in ref.items()}
    y = _f(ref["y"])
    i = tuple(np.argwhere(np.abs(y) > 0)[0])
    v = 8.0 * rms * np.sign(y[i])                            # made large: one spacing above 2e-2 * RMS
    sp = float(helpers.bf16_ulp(np.array([v]))[0])
    assert sp > 2e-2 * rms
    base = np.float32(_f(_bits([v]))[0])
    mid = np.float32(base + np.float32(sp / 2) * np.float32(np.sign(v)) * np.float32(0.999))   # just below the boundary
    wide["y32"][i] = mid
    wide["ylo"][i] = wide["yhi"][i] = float(mid)
    wide["y"][i] = _bits([mid])[0]
    out = _f(wide["y"]).copy()
    out[i] = float(base) + sp * np.sign(v)                    # the neighbour across the boundary
    helpers.check_y(_bits(out), wide)
    out[i] = float(base) + 2 * sp * np.sign(v)
    with pytest.raises(AssertionError, match="above 2e-2"):
        helpers.check_y(_bits(out), wide)


def test_h_range_check(ref):
    """check_h_in_range accepts the oracle's own h, and an h moved to the far end of a flagged
    element's range; it rejects an element moved one bf16 step beyond its range."""
    T, k, I = ref["a"].shape
    row_of = ref["row_of"].reshape(T, k)
    hc = np.zeros((T * k, I), np.uint16)
    for t in range(T):
        for j in range(k):
            hc[row_of[t, j]] = ref["a"][t, j]
    st = helpers.check_h_in_range(hc, ref)
    assert st["n_diff"] == 0 and st["n_flagged"] > 0
    t, j, n = np.argwhere(ref["a_hi"] != ref["a"])[0]
    h2 = hc.copy()
    h2[row_of[t, j], n] = ref["a_hi"][t, j, n]
    assert helpers.check_h_in_range(h2, ref)["n_diff"] == 1
    t, j, n = np.argwhere(ref["a_hi"] == ref["a"])[0]
    h3 = hc.copy()
    a = float(_f(ref["a"][t, j])[n])
    h3[row_of[t, j], n] = _bits([a + helpers.bf16_ulp(np.array([a]))[0] * 1.01])[0]
    with pytest.raises(AssertionError, match="outside the oracle's range"):
        helpers.check_h_in_range(h3, ref)
