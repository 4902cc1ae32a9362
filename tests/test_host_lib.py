"""Host-side checks of the C-ABI library (no GPU): exported symbols, argument
validation, and the expert-wave tile schedule the device builds."""
import ctypes
import os
import re

import numpy as np
import pytest

import mixture_experts_layer_top_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.load()


def test_exports_match_header(lib):
    hdr = open(os.path.join(ROOT, "include", "moe_gb300.h")).read()
    names = re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", hdr, flags=re.M)
    assert len(names) >= 10
    assert set(names) == set(moe.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_config_struct_layout():
    assert ctypes.sizeof(moe.moe_config_t) == 56
    assert moe.moe_config_t.timeout_ns.offset == 40 and moe.moe_config_t.router_bias.offset == 48


@pytest.mark.parametrize("kw,status", [
    (dict(H=100), moe.MOE_ERR_UNSUPPORTED), (dict(I=96), moe.MOE_ERR_UNSUPPORTED),
    (dict(H=32), moe.MOE_ERR_UNSUPPORTED), (dict(I=160), moe.MOE_ERR_UNSUPPORTED),
    (dict(E=300), moe.MOE_ERR_UNSUPPORTED), (dict(top_k=9), moe.MOE_ERR_UNSUPPORTED),
    (dict(top_k=0), moe.MOE_ERR_INVALID_ARG), (dict(T_max=0), moe.MOE_ERR_INVALID_ARG),
    (dict(schedule=4), moe.MOE_ERR_INVALID_ARG), (dict(E=4, top_k=5), moe.MOE_ERR_UNSUPPORTED),
    (dict(flags=moe.MOE_FLAG_GEMM_STREAMING | moe.MOE_FLAG_GEMM_COMPUTE), moe.MOE_ERR_INVALID_ARG),
])
def test_config_validation(lib, kw, status):
    base = dict(T_max=256, H=512, I=256, E=8, top_k=2)
    base.update(kw)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_workspace_bytes(moe.MoEConfig(**base).c())
    assert ei.value.status == status


@pytest.mark.parametrize("H,I", [(64, 64), (320, 192), (448, 64), (2048 + 64, 768 + 64)])
def test_config_accepts_multiples_of_64(lib, H, I):
    """H and I need only be multiples of 64 (one 64-column TMA box): the last Linear-1 tile of an
    expert may hold 64 intermediate columns, the last Linear-2 tile 64, 128 or 192 outputs."""
    b = moe.moe_workspace_bytes(moe.MoEConfig(256, H, I, 8, 2).c())
    assert b >= 256 * 2 * (2 * H + 2 * I + 4 * H)


def test_workspace_bytes_padded_layout(lib):
    """x, h and P live in a padded row space: every 256-row unit of an expert owns its rows,
    so the workspace holds at least R and at most R + 256*E rows of (2H + 2I + 4H) bytes."""
    T, H, I, E, k = 8192, 2048, 768, 128, 8
    b = moe.moe_workspace_bytes(moe.MoEConfig(T, H, I, E, k).c())
    per_row = 2 * H + 2 * I + 4 * H
    R = T * k
    assert R * per_row <= b
    assert b <= (R + 256 * E + 256) * (per_row + 8) + R * 24 + T * H * 4 + (16 << 20)
    small = moe.moe_workspace_bytes(moe.MoEConfig(1024, H, I, E, k).c())
    assert small < b


def test_plan_without_device_fails_cleanly(lib):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except Exception:
        pass
    h = ctypes.c_void_p(0)
    st = lib.moe_plan(ctypes.byref(moe.MoEConfig(256, 512, 256, 8, 2).c()), 0, ctypes.byref(h))
    assert st != moe.MOE_OK and not h.value


def _check_schedule(counts, H, I, sms, mode, wave_experts=0, lead=1):
    tiles, n1 = moe.moe_schedule_host(counts, H, I, sms, mode, wave_experts, lead)
    nL1, nL2 = -(-I // 128), -(-H // 256)          # the last tile of each may be partial
    mt = (np.asarray(counts) + 255) // 256          # units: pairs of 128-row m-tiles (one 2-CTA cluster)
    mtb = np.concatenate([[0], np.cumsum(mt)])
    total_mt = int(mtb[-1])
    assert len(tiles) == total_mt * (nL1 + nL2)
    assert n1 == total_mt * nL1
    # every tile exactly once
    keys = set()
    for ph_n, e, m, g in tiles.tolist():
        ph, nb, rows = ph_n & 1, (ph_n >> 1) & 0x7FFF, ph_n >> 16
        assert 0 <= m < mt[e] and g == mtb[e] + m
        assert nb < (nL1 if ph == 0 else nL2)
        assert rows == min(256, counts[e] - 256 * m) and rows >= 1
        keys.add((ph, nb, e, m))
    assert len(keys) == len(tiles)
    # topological: every Linear-2 tile after all Linear-1 tiles of its m-tile
    last_l1 = {}
    for i, (ph_n, e, m, g) in enumerate(tiles.tolist()):
        if ph_n & 1 == 0:
            last_l1[g] = i
    seen = {}
    for i, (ph_n, e, m, g) in enumerate(tiles.tolist()):
        if ph_n & 1 == 0:
            seen[g] = seen.get(g, 0) + 1
        else:
            assert seen.get(g, 0) == nL1 and last_l1[g] < i
    return tiles, n1


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("dist", ["uniform", "zipf", "zeros", "one"])
def test_schedule_permutation_and_order(lib, mode, dist):
    rng = np.random.default_rng(7)
    E = 64
    if dist == "uniform":
        counts = rng.multinomial(E * 300, np.ones(E) / E)
    elif dist == "zipf":
        p = (np.arange(1, E + 1) ** -1.2)
        counts = rng.multinomial(20000, p / p.sum())
    elif dist == "zeros":
        counts = np.zeros(E, np.int64)
        counts[[3, 17, 40]] = [5, 1000, 129]
    else:
        counts = np.zeros(E, np.int64)
        counts[E - 1] = 4096
    _check_schedule(counts, 512, 256, 20, mode, 0, 2 if mode == 1 else 1)


@pytest.mark.parametrize("H,I", [(64, 64), (320, 192), (704, 320)])
def test_schedule_partial_column_blocks(lib, H, I):
    """Shapes whose I is not a multiple of 128 or H of 256 get ceil(I/128) Linear-1 and
    ceil(H/256) Linear-2 tiles per unit (the last one partial)."""
    counts = np.random.default_rng(3).multinomial(3000, np.ones(12) / 12)
    for mode in (0, 1, 2):
        tiles, n1 = _check_schedule(counts, H, I, 12, mode)
        nb1 = {(t[0] >> 1) & 0x7FFF for t in tiles[:n1].tolist() if t[0] & 1 == 0}
        nb2 = {(t[0] >> 1) & 0x7FFF for t in tiles.tolist() if t[0] & 1 == 1}
        assert nb1 == set(range(-(-I // 128))) and nb2 == set(range(-(-H // 256)))


def test_schedule_phased_is_l1_then_l2(lib):
    counts = np.random.default_rng(1).multinomial(5000, np.ones(16) / 16)
    tiles, n1 = _check_schedule(counts, 512, 256, 10, 2)
    assert np.all(tiles[:n1, 0] & 1 == 0) and np.all(tiles[n1:, 0] & 1 == 1)


def test_schedule_wave_serial_vs_interleaved(lib):
    counts = np.full(32, 512)        # 2 units per expert, nL1 = 2 -> 4 L1 tiles per expert
    sms = 16                         # 16 workers: waves of 4 experts
    t0, _ = _check_schedule(counts, 512, 256, sms, 0)
    t1, _ = _check_schedule(counts, 512, 256, sms, 1, 0, 1)
    ph0, ph1 = t0[:, 0] & 1, t1[:, 0] & 1
    # wave-serial: runs of 16 L1 then 16 L2 tiles (nL2 = 2), wave by wave
    assert ph0[:16].sum() == 0 and ph0[16:32].sum() == 16 and ph0[32:48].sum() == 0
    # interleaved (lead 1): after the first wave's L1, L2(w) alternates with L1(w+1)
    assert ph1[:16].sum() == 0
    assert ph1[16:48].tolist() == [1, 0] * 16
    # same multiset of tiles
    assert sorted(map(tuple, t0.tolist())) == sorted(map(tuple, t1.tolist()))


def test_merge_positions_proportional(lib):
    # unequal lists: a = 3 L2 tiles vs b = 9 L1 tiles per wave
    counts = np.full(8, 256 * 3)     # 3 units/expert
    tiles, _ = _check_schedule(counts, 256, 384, 9, 1, 1, 1)   # 1 expert per wave, nL1=3, nL2=1
    ph = (tiles[:, 0] & 1).tolist()
    seg = ph[9:9 + 12]               # merged segment: 3 L2 + 9 L1
    assert sum(seg) == 3
    pos = [i for i, v in enumerate(seg) if v == 1]
    assert pos == [1, 5, 9]          # L2 tiles at ~1/6, 1/2, 5/6 of the segment


def test_flag_constants_match_header():
    """The binding's MOE_FLAG_* / MOE_SCHED_* constants are the header's values."""
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                            "moe_gb300.h")).read()
    found = 0
    for name, shift, plain in re.findall(r"#define (MOE_(?:FLAG|SCHED)_[A-Z_]+) +(?:\(1u << (\d+)\)|(\d+))", src):
        v = (1 << int(shift)) if shift else int(plain)
        assert getattr(moe, name) == v, name
        found += 1
    assert found >= 12
