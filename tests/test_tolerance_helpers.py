"""The y acceptance rule of the GPU tests, pinned on the CPU: the explained-outlier path of
helpers.check_y_explained must accept the oracle's own result and reject an intermediate
that is far off or differs in too many elements, or an output error the intermediate does
not explain."""
import numpy as np
import pytest

import helpers
import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.fixture(scope="module")
def case():
    synth.build_host()
    oracle.build()
    wl = synth.Workload("tol", 48, 256, 128, 6, 2)
    h = synth.host_inputs(wl)
    ref = helpers.oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]),
                             want_intermediates=True)
    T, k, I = ref["a"].shape
    row_of = ref["row_of"].reshape(T, k)
    hc = np.zeros((T * k, I), np.uint16)
    for t in range(T):
        for j in range(k):
            hc[row_of[t, j]] = ref["a"][t, j]
    return ref, hc, h["W2"]


def _forced(monkeypatch):
    """Make the first (direct) comparison fail so that the explained path runs."""
    real = helpers.check_y
    calls = []

    def fake(a, b, what="y"):
        calls.append(what)
        if len(calls) == 1:
            raise AssertionError("forced")
        return real(a, b, what)
    monkeypatch.setattr(helpers, "check_y", fake)
    return calls


def test_accepts_the_oracle_itself(case, monkeypatch):
    ref, hc, W2 = case
    helpers.check_y_explained(ref["y"], ref, hc, W2)          # direct path
    calls = _forced(monkeypatch)
    helpers.check_y_explained(ref["y"], ref, hc, W2)          # explained path
    assert len(calls) == 2


def test_rejects_h_far_off(case, monkeypatch):
    ref, hc, W2 = case
    h = helpers.f64(hc)
    rms = float(np.sqrt(np.mean(h ** 2)))
    r, i = np.unravel_index(np.argmax(np.abs(h)), h.shape)
    h[r, i] += rms                                            # far beyond 2e-2 * RMS(h) + one ulp
    _forced(monkeypatch)
    with pytest.raises(AssertionError, match="beyond 2e-2"):
        helpers.check_y_explained(ref["y"], ref, oracle.f32_to_bf16(h.astype(np.float32)), W2)


def test_rejects_many_h_flips(case, monkeypatch):
    ref, hc, W2 = case
    bad = hc.copy().ravel()
    nz = np.nonzero(helpers.f64(bad) != 0)[0]
    bad[nz[:: 50]] += 1                                       # one bf16 ulp on 2% of the elements
    _forced(monkeypatch)
    with pytest.raises(AssertionError, match="of h elements differ"):
        helpers.check_y_explained(ref["y"], ref, bad.reshape(hc.shape), W2)


def test_rejects_output_error_not_explained_by_h(case, monkeypatch):
    ref, hc, W2 = case
    y = helpers.f64(ref["y"])
    rms = float(np.sqrt(np.mean(y ** 2)))
    t, m = np.unravel_index(np.argmax(np.abs(y)), y.shape)
    y[t, m] += 0.1 * rms                                      # a wrong output, h untouched
    y_bad = oracle.f32_to_bf16(y.astype(np.float32))
    _forced(monkeypatch)
    with pytest.raises(AssertionError):
        helpers.check_y_explained(y_bad, ref, hc, W2)
