"""The seeded generator: C and torch implementations agree bit for bit, and both
match the scalar definition (SplitMix64 words, Box-Muller with libm log/cos)."""
import math

import numpy as np
import torch

import synth


def test_host_and_torch_bit_identical():
    for tid, std, start in [(1, 1.0, 0), (3, 0.02, 123456789), (4, 1 / 27.7, 7 * 10 ** 9)]:
        a = synth.normal_bf16_host(50000, std, tid, 0, start=start)
        b = synth.normal_bf16_torch(50000, std, tid, 0, start=start)
        assert np.array_equal(a, b.view(torch.int16).numpy().view(np.uint16))


def test_matches_scalar_definition():
    a = synth.normal_bf16_host(2000, 0.5, 2, seed=5)
    vals = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float().numpy()
    lib = synth._load()
    mism = 0
    for i in range(2000):
        w = synth.word_int(5, 2, i)
        assert w == lib.synth_word(5, 2, i)
        u1 = ((w >> 40) + 0.5) * 2.0 ** -24
        u2 = ((w >> 16) & 0xFFFFFF) * 2.0 ** -24
        n = math.sqrt(-2 * math.log(u1)) * math.cos(2 * math.pi * u2) * 0.5
        ref = torch.tensor([float(np.float32(n))]).to(torch.bfloat16).item()
        mism += ref != vals[i]
    assert mism == 0


def test_polynomials_accurate():
    u = np.linspace(1e-7, 1 - 1e-9, 10001)
    got = synth._ln_t(torch.from_numpy(u)).numpy()
    assert np.max(np.abs(got - np.log(u))) < 1e-14
    v = np.linspace(0, 1 - 2 ** -24, 10001)
    got = synth._cos2pi_t(torch.from_numpy(v)).numpy()
    assert np.max(np.abs(got - np.cos(2 * np.pi * v))) < 1e-14


def test_moments_and_zipf():
    a = synth.normal_bf16_host(1 << 20, 1.0, 1)
    v = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert abs(v.mean()) < 5e-3 and abs(v.std() - 1.0) < 5e-3
    b = synth.zipf_bias(128, 1.2)
    assert np.all(np.diff(b) < 0)
    p = np.exp(b.astype(np.float64) / 2)
    assert abs(p.sum() - 1) < 1e-5
    assert abs(b[0] - b[1] - 2.4 * math.log(2)) < 1e-5
