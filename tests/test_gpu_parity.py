"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every input comes from the seeded generator; device tensors are drawn on the
GPU by the torch implementation, which is bit-identical to the host one the
oracle uses (checked by test_device_generator_matches_host)."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_top_gb300 as moe
import oracle
import synth
from helpers import (bits, check_h_in_range, check_logits, check_y, f64, from_bits, oracle_for, routing_equal,
                     sample_tokens)

EXACT = moe.MOE_FLAG_EXACT_LOGITS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe.build()
    oracle.build()
    synth.build_host()
    torch.cuda.init()


def _layer(wl, schedule=0, flags=0, T_max=None, timeout_ns=0, wave_experts=0, lead=1, bias=None):
    cfg = moe.MoEConfig(T_max or wl.T, wl.H, wl.I, wl.E, wl.k, schedule=schedule, flags=flags,
                        timeout_ns=timeout_ns, wave_experts=wave_experts, lead_waves=lead)
    return moe.MoELayer(cfg, 0, router_bias=bias)


def _router_plan(T, H, E, exact=False):
    """(router launches, every logit canonical) of a forward under the library's router rule:
    the canonical task kernel (+ top-k unless E <= 8) while 32-token x 8-expert tasks fit one per
    SM, else the tensor-core estimate + transpose + certified selection (or the 32 x 32
    canonical kernel + top-k under EXACT)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if -(-T // 32) * -(-E // 8) <= sms:
        return (1 if E <= 8 else 2), True
    return (2, True) if exact else (3, False)


def _bias(wl):
    return synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None


# --------------------------------------------------------------------------- generator
def test_device_generator_matches_host():
    for tid, std, start in [(1, 1.0, 0), (3, 0.02, 5 * 10 ** 9 + 17)]:
        a = synth.normal_bf16_host(1 << 20, std, tid, 0, start=start)
        d = synth.normal_bf16_torch(1 << 20, std, tid, 0, start=start, device="cuda")
        assert np.array_equal(a, bits(d))


# --------------------------------------------------------------------------- tiny config
@pytest.mark.parametrize("schedule,flags", [(0, 0), (1, 0), (2, 0), (0, EXACT), (2, EXACT)])
def test_tiny_full_parity(schedule, flags):
    """Whole layer on the 256-token config, every schedule.  The default router is the canonical
    task kernel here, with the top-k in the same launch (as with MOE_FLAG_EXACT_LOGITS): logits
    bit-exact either way."""
    wl = synth.WORKLOADS["tiny"]
    h = synth.host_inputs(wl)
    ref = oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]))
    d = {k: from_bits(v) for k, v in h.items() if k != "bias"}
    layer = _layer(wl, schedule, flags=flags)
    y, logits = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    assert np.array_equal(logits.cpu().numpy(), ref["logits"]), "logits not bit-exact"
    routing_equal(layer.routing(wl.T), ref, wl.T)
    check_y(bits(y), ref)
    assert layer.launch_count() == _router_plan(wl.T, wl.H, wl.E, bool(flags & EXACT))[0] + (5 if schedule == 2 else 4)


def test_bilinear_integer_exact():
    """Integer-valued inputs and the bilinear GLU: every accumulation is exact, so
    h, P and y must match the oracle bit for bit (tiling, TMA boxes, descriptors).
    The caller's logits give each token k tied top logits, so every router weight is
    exactly 1/k and the check does not depend on the rounding of the softmax."""
    T, H, I, E, k = 300, 512, 256, 8, 2
    rng = np.random.default_rng(11)

    def tern(shape, p):
        return ((rng.random(shape) < p) * rng.choice([-1.0, 1.0], size=shape)).astype(np.float32)

    x = oracle.f32_to_bf16(tern((T, H), 0.5))
    Wr = oracle.f32_to_bf16((rng.standard_normal((H, E)) / np.sqrt(H)).astype(np.float32))
    W1 = oracle.f32_to_bf16(tern((E, H, 2 * I), 0.2))
    W2 = oracle.f32_to_bf16(tern((E, I, H), 0.2))
    logits = np.zeros((T, E), np.float32)
    for t in range(T):
        logits[t, rng.choice(E, size=k, replace=False)] = 1.0
    ref = oracle.forward(x, Wr, None, W1, W2, k, act=oracle.ACT_BILINEAR, logits=logits,
                         want_intermediates=True)
    assert np.all(ref["w"] == np.float32(1.0 / k))
    layer = moe.MoELayer(moe.MoEConfig(T, H, I, E, k, flags=moe.MOE_FLAG_ACT_BILINEAR), 0)
    y, _ = layer.forward(from_bits(x), None, from_bits(W1), from_bits(W2),
                         logits=torch.from_numpy(logits).cuda(), check=True)
    r = layer.routing(T)
    routing_equal(r, ref, T)
    hh, P = layer.intermediates(T)
    row_of = ref["row_of"].reshape(T, k)
    h_gpu = f64(bits(hh))
    P_gpu = P.cpu().numpy()
    a_ref = f64(ref["a"])
    P_ref = ref["w"][:, :, None].astype(np.float32) * ref["o"]       # fp32 product, as the epilogue
    for t in range(T):
        for j in range(k):
            assert np.array_equal(h_gpu[row_of[t, j]], a_ref[t, j]), f"h row (t={t}, j={j})"
            assert np.array_equal(P_gpu[t * k + j], P_ref[t, j]), f"P row (t={t}, j={j})"
    assert np.array_equal(f64(bits(y)), f64(ref["y"])), "y not bit-exact on integer inputs"


@pytest.mark.parametrize("exp2", [20, -30])
def test_expert_outputs_far_outside_fp16_range(exp2):
    """P is stored as fp16 times a power-of-two scale per (row, 128 columns): W2 scaled by
    2^20 (|P| far above 65504) or 2^-30 (|P| far below fp16's normal range) must give the
    oracle's y within the usual tolerance, with no overflow to inf and no flush to zero."""
    wl = synth.Workload("range", 512, 512, 256, 8, 2)
    h = synth.host_inputs(wl)
    W2 = oracle.f32_to_bf16(oracle.bf16_to_f32(h["W2"]) * np.float32(2.0 ** exp2))   # exact
    ref = oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], W2))
    layer = _layer(wl)
    d = {k: from_bits(v) for k, v in h.items() if k != "bias"}
    y, _ = layer.forward(d["x"], d["Wr"], d["W1"], from_bits(W2), check=True)
    yr = f64(ref["y"])
    assert np.abs(yr).max() > (1e6 if exp2 > 0 else 0) and np.abs(yr).max() < (np.inf if exp2 > 0 else 1e-6)
    check_y(bits(y), ref)


@pytest.mark.parametrize("name", ["skew", "smallT"])
def test_device_schedule_equals_host_schedule(name):
    """The Dispatch kernel builds the tile list in parallel; it must equal the serial host
    builder's (whose permutation and dependency order the host tests check) for every mode."""
    wl = synth.WORKLOADS[name]
    bias = _bias(wl)
    d = synth.device_inputs(wl)
    for sched, we, lead in [(0, 0, 1), (1, 0, 1), (1, 0, 3), (2, 0, 1), (0, 5, 1), (1, 7, 2), (3, 0, 1)]:
        layer = _layer(wl, sched, wave_experts=we, lead=lead, bias=bias)
        layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
        tiles, n1, workers = layer.schedule()
        counts = layer.routing(wl.T)["counts"].cpu().numpy()
        if sched == moe.MOE_SCHED_AUTO:   # resolves to wave-serial with one wave of all experts
            sched, we = moe.MOE_SCHED_WAVE_SERIAL, wl.E
        ref, n1_ref = moe.moe_schedule_host(counts, wl.H, wl.I, workers, sched, we, lead)
        assert n1 == n1_ref and np.array_equal(tiles, ref), f"schedule {sched}/{we}/{lead} differs"
        layer.close()
    del d
    torch.cuda.empty_cache()


def test_schedules_bitwise_identical():
    """Every tile schedule and both shared-memory splits of the grouped GEMM give the same bits
    (the default streaming split and the forced compute split)."""
    wl = synth.Workload("mid", 2048, 1024, 512, 32, 4)
    d = synth.device_inputs(wl)
    outs = []
    S = moe.MOE_FLAG_GEMM_COMPUTE
    for sched, we, lead, fl in [(0, 0, 1, 0), (1, 0, 1, 0), (1, 0, 3, 0), (2, 0, 1, 0), (0, 3, 1, 0),
                                (1, 2, 2, 0), (3, 0, 1, 0), (1, 0, 1, S), (2, 0, 1, S), (0, 3, 1, S)]:
        layer = _layer(wl, sched, wave_experts=we, lead=lead, flags=fl)
        y, _ = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
        y2, _ = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "repeat not bitwise identical"
        outs.append(bits(y))
        layer.close()
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "schedules differ"
    h = synth.host_inputs(wl, weights=False)
    tok = sample_tokens(wl.T, 48)
    ref = oracle_for(wl, h["x"], h["Wr"], None, tok)
    check_y(outs[0][tok], ref)


# --------------------------------------------------------------------------- full-size workloads
def _cover_tokens(ids: np.ndarray, n: int, min_experts: int) -> np.ndarray:
    """n tokens chosen greedily (by the oracle's routing) so that their experts cover as many
    distinct experts as possible - at least min_experts - plus the first and last token."""
    T = ids.shape[0]
    chosen, seen = [0, T - 1], set(ids[0]) | set(ids[T - 1])
    order = np.random.default_rng(3).permutation(T)
    while len(chosen) < n:
        best, gain = None, -1
        for t in order[:4096]:
            if t in chosen:
                continue
            g = len(set(ids[t]) - seen)
            if g > gain:
                best, gain = int(t), g
        chosen.append(best)
        seen |= set(ids[best])
    assert len(seen) >= min_experts, f"only {len(seen)} experts covered"
    return np.sort(np.array(chosen, np.int64))


def _device_weights(d):
    """Host copies of the expert slices of the device tensors the synth generator drew (the
    generator's device and host implementations are bit-identical)."""
    return lambda which, e: d[which][e].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name,nsample,schedule,flags", [
    ("fine", 48, 0, 0), ("fine", 16, 1, EXACT), ("skew", 32, 0, 0), ("large", 64, 0, 0), ("smallT", 128, 0, 0),
    ("smallT", 128, 1, EXACT)])
def test_workload_parity(name, nsample, schedule, flags):
    """Full-size workloads: routing of every token against the oracle (ids, counts, order
    bit-exact), logits (bit-exact, or selected-exact and bounded), y on sampled tokens: every
    token of the 128-token workload, and on the large layer 64 tokens chosen to reach at least
    200 of its 256 experts."""
    wl = synth.WORKLOADS[name]
    bias = _bias(wl)
    d = synth.device_inputs(wl)
    layer = _layer(wl, schedule, bias=bias, flags=flags)
    y, logits = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    h = synth.host_inputs(wl, weights=False)
    lg_ref = oracle.router_logits(h["x"], h["Wr"], bias)
    if name == "large":
        tok = _cover_tokens(oracle.topk(lg_ref, wl.k)[0], nsample, 200)
        assert np.array_equal(synth.expert_slice_host(wl, "W2", 17), _device_weights(d)("W2", 17))
    else:
        tok = sample_tokens(wl.T, nsample)
    ref = oracle.forward(h["x"], h["Wr"], bias, lambda e: _device_weights(d)("W1", e),
                         lambda e: _device_weights(d)("W2", e), wl.k, tokens=tok, logits=lg_ref, bounds=True)
    if flags & EXACT:
        assert np.array_equal(logits.cpu().numpy(), ref["logits"]), "logits not bit-exact"
    else:
        st = check_logits(logits.cpu().numpy(), ref, h["x"], h["Wr"], layer.router_bound(wl.T), bias)
        print(f"{name}: canonical entries {st['exact_frac']:.3f}, estimate error <= "
              f"{st['max_ratio']:.2e} of the bound")
    routing_equal(layer.routing(wl.T), ref, wl.T)
    if name == "skew":
        assert (ref["counts"] == 0).any(), "skewed workload should leave experts idle"
    n_exp = len({int(e) for e in ref["ids"][tok].ravel()})
    st = check_y(bits(y)[tok], ref, what=name)
    print(f"{name}: y on {len(tok)} tokens ({n_exp} experts): {st}")
    del d
    layer.close()
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------- edge cases
@pytest.mark.parametrize("T,flags", [(1, 0), (127, 0), (129, 0), (1000, 0),
                                     (129, moe.MOE_FLAG_GEMM_COMPUTE), (1000, moe.MOE_FLAG_GEMM_COMPUTE)])
def test_ragged_token_counts(T, flags):
    """Ragged token counts against the full oracle (default split, and the compute split forced)."""
    wl = synth.Workload("edge", T, 512, 256, 16, 4)
    h = synth.host_inputs(wl)
    ref = oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]))
    layer = _layer(wl, 0, T_max=1024, flags=flags)
    d = {k: from_bits(v) for k, v in h.items() if k != "bias"}
    y, logits = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    check_logits(logits.cpu().numpy(), ref, h["x"], h["Wr"], layer.router_bound(T))
    routing_equal(layer.routing(T), ref, T)
    check_y(bits(y), ref)


@pytest.mark.parametrize("schedule", [moe.MOE_SCHED_AUTO, moe.MOE_SCHED_INTERLEAVED, moe.MOE_SCHED_PHASED])
def test_plan_reused_across_batches(schedule):
    """One plan, six forwards with different token counts and different inputs (weights
    included), two of them through the host-buffer entry point: each against the full
    oracle, so that nothing a forward leaves in the workspace (counts, chunk histograms,
    readiness counters, padded rows, the staging buffers, the router's split estimates) reaches
    the next one.  With 64 experts the router changes between forwards: the tensor-core one for
    1000 and 640 tokens, the canonical task kernel for the others."""
    layer = None
    plans = [(1000, 11, False), (37, 12, False), (513, 13, False), (200, 14, True), (1000, 15, False), (640, 16, True)]
    assert [_router_plan(T, 512, 64)[1] for T, _, _ in plans] == [False, True, True, True, False, False]
    for T, seed, host in plans:
        wl = synth.Workload("reuse", T, 512, 256, 64, 4, seed=seed)
        if layer is None:
            layer = _layer(wl, schedule, T_max=1024)
        h = synth.host_inputs(wl)
        ref = oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]), want_intermediates=True)
        d = {kk: from_bits(v) for kk, v in h.items() if kk != "bias"}
        if host:
            y = torch.empty((T, wl.H), dtype=torch.bfloat16).pin_memory()
            logits = torch.empty((T, wl.E), dtype=torch.float32, device="cuda")
            layer.forward_host(d["x"].cpu().pin_memory(), d["Wr"], d["W1"], d["W2"], logits, y, check=True)
        else:
            y, logits = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
        check_logits(logits.cpu().numpy(), ref, h["x"], h["Wr"], layer.router_bound(T))
        routing_equal(layer.routing(T), ref, T)
        h_gpu, _ = layer.intermediates(T, want_P=False)
        check_y(bits(y), ref)
        check_h_in_range(bits(h_gpu), ref)
    layer.close()


@pytest.mark.parametrize("T,H,I,E,k", [(100, 256, 128, 6, 2), (64, 256, 128, 1, 1), (50, 512, 128, 40, 8),
                                       (300, 256, 384, 3, 3), (33, 768, 256, 200, 8),
                                       (77, 64, 64, 5, 2), (200, 320, 192, 12, 3), (129, 384, 320, 40, 4),
                                       (300, 448, 128, 9, 4), (60, 2112, 832, 16, 8),
                                       (5000, 256, 64, 5, 2), (9000, 1024, 64, 1, 1), (6000, 512, 64, 6, 3),
                                       (1200, 2048, 128, 6, 3),
                                       (2048, 16384, 64, 64, 2), (100, 64, 8192, 8, 2)])
@pytest.mark.parametrize("flags", [0, EXACT])
def test_odd_shapes_full_oracle(T, H, I, E, k, flags):
    """Expert counts that are not multiples of 8 / 16 / 32 (tensor-core router N padding,
    transpose tiles, selection keys), one expert, k = E, the smallest H and I the layout allows
    (64), and H = 64, 128, 192 (mod 256) with I = 64 (mod 128) - partial last Linear-1 and
    Linear-2 tiles and P scale blocks, router rows not a multiple of 256 h, a long hidden size
    (H = 16384) and a wide intermediate (I = 8192): routing and y against the full oracle,
    default and all-canonical routers.  Which router runs follows the library's rule
    (`_router_plan`): the canonical kernels' logits equal the oracle's, the tensor-core
    router's estimates lie within the bound (shapes with more 32 x 8 tasks than SMs, among them
    ones with at most 8 experts)."""
    wl = synth.Workload("odd", T, H, I, E, k)
    h = synth.host_inputs(wl)
    ref = oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]))
    layer = _layer(wl, flags=flags)
    d = {kk: from_bits(v) for kk, v in h.items() if kk != "bias"}
    y, logits = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    n_router, canonical = _router_plan(T, H, E, bool(flags & EXACT))
    assert layer.launch_count() == n_router + 4      # router launches + Dispatch, gather, GEMM, Combine
    if canonical:
        assert np.array_equal(logits.cpu().numpy(), ref["logits"])
    else:
        st = check_logits(logits.cpu().numpy(), ref, h["x"], h["Wr"], layer.router_bound(T))
        if E > k:
            assert st["exact_frac"] < 1.0, "tensor-core estimates expected"
    routing_equal(layer.routing(T), ref, T)
    check_y(bits(y), ref)


def _random_cases(n: int, seed: int = 20261202):
    """Seeded layer shapes within the library's limits: H and I multiples of 64, E up
    to 256, k up to min(8, E), T up to 300 with a larger T_max, any schedule, the default or
    all-canonical router, the compute ring split or the single launch, a Zipf router bias on
    some."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        E = int(rng.choice([int(rng.integers(1, 65)), int(rng.integers(65, 257))]))
        out.append(dict(T=int(rng.integers(1, 301)), H=int(rng.choice([64, 256, 320, 512, 704, 768, 1024, 2048])),
                        I=int(rng.choice([64, 128, 192, 256, 384, 448, 512])), E=E, k=int(rng.integers(1, min(8, E) + 1)),
                        sched=int(rng.integers(0, 4)), extra=int(rng.integers(0, 200)),
                        flags=[0, EXACT, moe.MOE_FLAG_GEMM_COMPUTE, moe.MOE_FLAG_SINGLE_LAUNCH][int(rng.integers(0, 4))],
                        zipf=float(rng.choice([0.0, 1.2])), host=bool(rng.integers(0, 3) == 0)))
    return out


def _random_cases_many_tokens(n: int, seed: int = 20261203):
    """Seeded shapes with 300 to 2000 tokens and small H and I (multiples of 64 up to 512 / 256),
    so that the tensor-core router, experts of several 256-row units and multi-wave schedules
    meet ragged shapes while the full oracle stays cheap."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        E = int(rng.choice([int(rng.integers(2, 33)), int(rng.integers(33, 257))]))
        out.append(dict(T=int(rng.integers(300, 2001)), H=64 * int(rng.integers(1, 9)), I=64 * int(rng.integers(1, 5)),
                        E=E, k=int(rng.integers(1, min(8, E) + 1)), sched=int(rng.integers(0, 4)),
                        extra=int(rng.integers(0, 300)),
                        flags=[0, 0, EXACT, moe.MOE_FLAG_GEMM_COMPUTE, moe.MOE_FLAG_SINGLE_LAUNCH][int(rng.integers(0, 5))],
                        zipf=float(rng.choice([0.0, 1.2])), host=bool(rng.integers(0, 3) == 0)))
    return out


@pytest.mark.parametrize("c", _random_cases(48) + _random_cases_many_tokens(64),
                         ids=lambda c: "T{T}-H{H}-I{I}-E{E}-k{k}-s{sched}-f{flags}-z{zipf}-h{host:d}".format(**c))
def test_random_shapes_full_oracle(c):
    """Routing (bit-exact) and y (stated tolerance) against the full oracle on seeded random
    shapes, schedules and kernel variants, with the plan sized above the batch; a third of
    the cases through the host-buffer entry point (page-locked x and y), half of those as
    pipelined host forwards (MOE_FLAG_HOST_PIPELINE: y copied out on the plan's own stream)."""
    wl = synth.Workload("rand", c["T"], c["H"], c["I"], c["E"], c["k"], zipf_s=c["zipf"])
    h = synth.host_inputs(wl)
    bias = _bias(wl)
    ref = oracle_for(wl, h["x"], h["Wr"], bias, None, full_weights=(h["W1"], h["W2"]), want_intermediates=True)
    pipe = moe.MOE_FLAG_HOST_PIPELINE if c["host"] and c["extra"] % 2 else 0
    layer = _layer(wl, c["sched"], flags=c["flags"] | pipe, T_max=c["T"] + c["extra"], bias=bias)
    d = {kk: from_bits(v) for kk, v in h.items() if kk != "bias"}
    if c["host"]:
        x_host = d["x"].cpu().pin_memory()
        y = torch.empty((c["T"], c["H"]), dtype=torch.bfloat16).pin_memory()
        logits = torch.empty((c["T"], c["E"]), dtype=torch.float32, device="cuda")
        layer.forward_host(x_host, d["Wr"], d["W1"], d["W2"], logits, y, check=True)
    else:
        y, logits = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    if c["flags"] & (EXACT | moe.MOE_FLAG_SINGLE_LAUNCH):     # the single launch's logits are all canonical
        assert np.array_equal(logits.cpu().numpy(), ref["logits"])
    else:
        check_logits(logits.cpu().numpy(), ref, h["x"], h["Wr"], layer.router_bound(c["T"]), bias)
    routing_equal(layer.routing(c["T"]), ref, c["T"])
    st = check_y(bits(y), ref)
    h_gpu, _ = layer.intermediates(c["T"], want_P=False)
    hs = check_h_in_range(bits(h_gpu), ref)
    print(f"y: {st}; h: {hs}")
    layer.close()


def test_phased_plans_overlap_on_two_streams():
    """Two plans with the phased schedule, forwards enqueued on two streams without ordering
    (the overlap the header allows): each result bitwise equal to the plan's solo forward."""
    wls = [synth.Workload("ovA", 2048, 1024, 512, 32, 4), synth.Workload("ovB", 1500, 768, 384, 20, 6)]
    ins = [synth.device_inputs(wl) for wl in wls]
    layers = [_layer(wl, moe.MOE_SCHED_PHASED) for wl in wls]
    solo = []
    for layer, d in zip(layers, ins):
        y, _ = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
        solo.append(y.view(torch.int16).clone())
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = [[], []]
    for _ in range(3):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                y, _ = layers[i].forward(ins[i]["x"], ins[i]["Wr"], ins[i]["W1"], ins[i]["W2"])
                outs[i].append(y)
    torch.cuda.synchronize()
    for i in range(2):
        with torch.cuda.stream(streams[i]):
            layers[i].check()
        for y in outs[i]:
            assert torch.equal(y.view(torch.int16), solo[i]), f"plan {i} differs when overlapped"
        layers[i].close()


def test_inconsistent_routing_reported_and_contained():
    """A test-only flag makes Dispatch see the first (token, slot) pair with an out-of-range
    expert id: moe_get_status reports MOE_ERR_DEVICE_CHECK, that pair is dropped without any
    access outside the workspace, every other token's y is bitwise the clean forward's, and
    the context stays usable (a clean forward afterwards matches the oracle)."""
    wl = synth.WORKLOADS["tiny"]
    h = synth.host_inputs(wl)
    d = {kk: from_bits(v) for kk, v in h.items() if kk != "bias"}
    good = _layer(wl)
    y_good, _ = good.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    bad = _layer(wl, flags=moe.MOE_FLAG_TEST_BAD_ID)
    y_bad, _ = bad.forward(d["x"], d["Wr"], d["W1"], d["W2"])
    assert moe.moe_get_status(bad.plan, bad._stream()) == moe.MOE_ERR_DEVICE_CHECK
    assert moe.moe_get_status(bad.plan, bad._stream()) == moe.MOE_OK          # the word is cleared
    assert torch.equal(y_bad[1:].view(torch.int16), y_good[1:].view(torch.int16))
    assert torch.isfinite(y_bad[0].float()).all()
    h_bad, P_bad = bad.intermediates(wl.T)                                      # debug copies stay in bounds
    torch.cuda.synchronize()
    bad.close()
    y2, _ = good.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    ref = oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]))
    check_y(bits(y2), ref)
    good.close()


def test_zero_tokens_is_noop():
    wl = synth.WORKLOADS["tiny"]
    layer = _layer(wl)
    x = torch.zeros((0, wl.H), dtype=torch.bfloat16, device="cuda")
    st = moe.moe_forward(layer.plan, 0, 16, 16, 16, 16, 16, 16, 0)   # nothing dereferenced at T = 0
    assert st == moe.MOE_OK and layer.launch_count() == 0
    del x


@pytest.mark.parametrize("mode,T,flags", [("pinned", 1000, 0), ("pinned_view", 1000, 0), ("pinned_offset8", 1000, 0),
                                          ("pageable", 1000, 0), ("pinned", 100, 0), ("pinned", 1000, EXACT),
                                          ("pageable", 100, EXACT)])
def test_host_buffers_match_device_forward(mode, T, flags):
    """The host-buffer entry point against the device one on the same inputs: y, the logits
    and the routing bit for bit.  Page-locked buffers at 16-byte-aligned addresses (a whole
    buffer, a view starting 3 rows in) are copied by the copy engines in up to 4 ranges of whole
    128-token chunks, each routed as it lands, with the split plan of the whole batch - and
    Combine writes y in place; a page-locked view 8 bytes off alignment and pageable buffers
    are staged whole.  The canonical routers (all-canonical, and the task kernel the 100-token
    batch takes) copy x whole."""
    wl = synth.Workload("host", T, 1024, 256, 64, 4)
    h = synth.host_inputs(wl)
    d = {k: from_bits(v) for k, v in h.items() if k != "bias"}
    layer = _layer(wl, flags=flags)
    y_dev, lg_dev = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    n_dev = layer.launch_count()
    r_dev = {k: v.cpu() for k, v in layer.routing(T).items()}
    n = wl.T * wl.H
    pin = mode != "pageable"
    xb = torch.empty(n + 3 * wl.H, dtype=torch.bfloat16, pin_memory=pin)
    yb = torch.full((n + 3 * wl.H,), float("nan"), dtype=torch.bfloat16, pin_memory=pin)
    off = {"pinned": 0, "pinned_view": 3 * wl.H, "pinned_offset8": 4, "pageable": 0}[mode]
    x_host = xb[off:off + n].view(wl.T, wl.H)
    y_host = yb[off:off + n].view(wl.T, wl.H)
    x_host.copy_(d["x"].cpu())
    logits = torch.empty_like(lg_dev)
    layer.forward_host(x_host, d["Wr"], d["W1"], d["W2"], logits, y_host, check=True)
    assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
    assert torch.equal(logits, lg_dev)
    for k_, v in layer.routing(T).items():
        assert torch.equal(v.cpu(), r_dev[k_]), k_
    direct = mode in ("pinned", "pinned_view")
    ranges = min(4, -(-T // 128))
    canonical = _router_plan(T, wl.H, wl.E, bool(flags & EXACT))[1]
    # the copies are the copy engines' (no launch); the tensor-core router runs once per range
    extra = 2 * (ranges - 1) if direct and not canonical else 0
    assert layer.launch_count() == n_dev + extra
    assert torch.isnan(yb[:off]).all() and torch.isnan(yb[off + n:]).all()   # nothing outside y_host


def test_router_certified_selection_on_ties_and_infinities():
    """Default router on adversarial inputs.  Integer-valued x and Wr make many canonical
    logits tie exactly (the bound then keeps every tied expert a candidate and the exact
    values break ties to the lower id); an infinite Wr entry makes one expert's logits
    non-finite, so every token falls back to canonical logits for all experts."""
    T, H, I, E, k = 1000, 512, 256, 64, 8
    assert not _router_plan(T, H, E)[1]               # the tensor-core router runs
    rng = np.random.default_rng(5)
    x = oracle.f32_to_bf16(rng.integers(-1, 2, size=(T, H)).astype(np.float32))
    Wr = oracle.f32_to_bf16((rng.integers(-2, 3, size=(H, E)) * 0.0625).astype(np.float32))
    wl = synth.Workload("ties", T, H, I, E, k)
    h = synth.host_inputs(wl)
    W1, W2 = from_bits(h["W1"]), from_bits(h["W2"])
    ref = oracle_for(wl, x, Wr, None, None, full_weights=(h["W1"], h["W2"]))
    layer = _layer(wl)
    y, logits = layer.forward(from_bits(x), from_bits(Wr), W1, W2, check=True)
    st = check_logits(logits.cpu().numpy(), ref, x, Wr, layer.router_bound(T))
    routing_equal(layer.routing(T), ref, T)
    check_y(bits(y), ref)
    assert st["exact_frac"] > 0.1     # ties force many candidates
    Wr_inf = Wr.copy()
    Wr_inf[3, 5] = 0x7F80              # bf16 +inf
    ref = oracle.forward(x, Wr_inf, None, h["W1"], h["W2"], k, tokens=np.arange(4, dtype=np.int64))
    y, logits = layer.forward(from_bits(x), from_bits(Wr_inf), W1, W2, check=True)
    lg, rl = logits.cpu().numpy(), ref["logits"]
    nan = np.isnan(rl)
    assert nan.any() and np.array_equal(np.isnan(lg), nan), "NaN logits differ"   # 0 * inf
    assert np.array_equal(lg[~nan].view(np.uint32), rl[~nan].view(np.uint32)), "fallback logits not canonical"
    routing_equal(layer.routing(T), ref, T)


def _stress_router_inputs(T, H, E, k, mode, seed=21):
    """Inputs built against the tensor-core router's error model; experts 0..23 are contenders
    with one shared small positive column, experts 24.. have a strongly negative column (the
    bound excludes them, so their estimates are written out).
    mode "align": the first 16 h of every token hold +64 and W_router +1 there, the last 16 h
    the same x with W_router -1, so every exact logit loses those 1024-sized terms, but the
    accumulation chain that takes the first K block carries a partial sum of 1024 while it adds
    the many small products in between (whose low bits an aligning adder drops).
    mode "ladder": contender pair p adds, at one h, p times one fp32 unit of the logit (x there
    picks 0, 1 or 2 units per token), so the k-th and (k+1)-th logits tie or differ by 1-2
    units."""
    rng = np.random.default_rng(seed)
    x = (2.0 ** -3 * (1.0 + rng.integers(0, 128, size=(T, H)) / 128.0)).astype(np.float32)
    Wr = np.empty((H, E), np.float32)
    base = 2.0 ** -6 * (1.0 + rng.integers(0, 128, size=H) / 128.0)
    Wr[:, :24] = base[:, None]
    Wr[:, 24:] = -4.0 * 2.0 ** -6 * (1.0 + rng.integers(0, 128, size=(H, E - 24)) / 128.0)
    if mode == "align":
        x[:, :16] = 64.0
        x[:, H - 16:] = 64.0
        Wr[:16] = 1.0
        Wr[H - 16:] = -1.0
    else:
        hz = 20
        x[:, hz] = rng.choice([0.0, 2.0 ** -3, 2.0 ** -2], size=T)
        Wr[hz, :24] = (np.arange(24) // 2) * 2.0 ** -18
    xb, wb = oracle.f32_to_bf16(x), oracle.f32_to_bf16(Wr)
    assert np.array_equal(oracle.bf16_to_f32(xb), x) and np.array_equal(oracle.bf16_to_f32(wb), Wr)
    return xb, wb


@pytest.mark.parametrize("mode", ["align", "ladder"])
def test_router_certificate_under_stress(mode):
    """Default router on inputs built to push the tensor-core estimate error toward its bound
    ("align") or to put the k-th place on exact ties and 1-2 unit gaps ("ladder"): routing
    bit-exact, selected logits canonical, every written estimate within the bound; the
    largest observed error/bound ratio is printed."""
    T, H, I, E, k = 1024, 1024, 256, 64, 8        # 256 router tasks: the tensor-core router runs
    assert not _router_plan(T, H, E)[1]
    xb, wb = _stress_router_inputs(T, H, E, k, mode)
    wl = synth.Workload("rstress", T, H, I, E, k)
    hw = synth.host_inputs(wl)
    ref = oracle_for(wl, xb, wb, None, None, full_weights=(hw["W1"], hw["W2"]))
    lg = ref["logits"]
    srt = np.sort(lg, axis=1)[:, ::-1]
    gap_ulp = (srt[:, k - 1] - srt[:, k]) / np.spacing(np.abs(srt[:, k - 1]))
    if mode == "ladder":
        assert set(np.unique(gap_ulp)) >= {0.0, 1.0, 2.0}, "ties and 1-2 unit gaps at the k-th place expected"
    layer = _layer(wl)
    y, logits = layer.forward(from_bits(xb), from_bits(wb), from_bits(hw["W1"]), from_bits(hw["W2"]), check=True)
    routing_equal(layer.routing(T), ref, T)
    st = check_logits(logits.cpu().numpy(), ref, xb, wb, layer.router_bound(T), max_ratio=1.0)
    print(f"router stress ({mode}): k-th gaps (ulp) {np.unique(gap_ulp, return_counts=True)}; estimates written for "
          f"{1 - st['exact_frac']:.2f} of the logits; largest error/bound {st['max_ratio']:.3e}")
    assert st["exact_frac"] < 0.9, "the losers' estimates should be written out"
    check_y(bits(y), ref)


def test_logits_as_input_and_one_hot_expert():
    """W_router = NULL: the caller's logits route; all tokens to one expert (all
    rows in one expert, every other expert empty)."""
    wl = synth.Workload("onehot", 700, 512, 256, 8, 1)
    h = synth.host_inputs(wl)
    logits = np.full((wl.T, wl.E), -5.0, np.float32)
    logits[:, 6] = 3.0
    ref = oracle.forward(h["x"], h["Wr"], None, h["W1"], h["W2"], wl.k, logits=logits, bounds=True)
    assert ref["counts"][6] == wl.T and ref["counts"].sum() == wl.T
    layer = _layer(wl)
    d = {k: from_bits(v) for k, v in h.items() if k != "bias"}
    lg = torch.from_numpy(logits).cuda()
    y, _ = layer.forward(d["x"], None, d["W1"], d["W2"], logits=lg, check=True)
    routing_equal(layer.routing(wl.T), ref, wl.T)
    check_y(bits(y), ref)


def test_router_weights_wide_logits():
    """Softmax weights over the k selected logits within 1e-6 relative of the oracle's
    fp64 evaluation when the logits spread widely (exp arguments down to about -150),
    tie in blocks (integer-valued rows), and some rows hold only 3 finite logits."""
    wl = synth.Workload("widelogits", 2048, 512, 256, 64, 8)
    h = synth.host_inputs(wl)
    rng = np.random.default_rng(7)
    logits = (rng.standard_normal((wl.T, wl.E)) * 25.0).astype(np.float32)
    logits[::5] = np.round(logits[::5] / 10.0)                       # many exact ties
    few = np.arange(3, wl.T, 11)
    logits[few, 3:] = -np.inf                                        # only 3 finite logits
    ref = oracle.forward(h["x"], h["Wr"], None, h["W1"], h["W2"], wl.k, logits=logits, bounds=True)
    layer = _layer(wl)
    d = {k: from_bits(v) for k, v in h.items() if k != "bias"}
    y, _ = layer.forward(d["x"], None, d["W1"], d["W2"], logits=torch.from_numpy(logits).cuda(), check=True)
    routing_equal(layer.routing(wl.T), ref, wl.T)
    check_y(bits(y), ref)


def test_nan_token_stays_local():
    wl = synth.Workload("nan", 256, 512, 256, 8, 2)
    h = synth.host_inputs(wl)
    x = h["x"].copy()
    x[5, 17] = 0x7FC0           # bf16 quiet NaN
    ref = oracle_for(wl, x, h["Wr"], None, None, full_weights=(h["W1"], h["W2"]))
    layer = _layer(wl)
    d = {k: from_bits(v) for k, v in h.items() if k != "bias"}
    y, logits = layer.forward(from_bits(x), d["Wr"], d["W1"], d["W2"], check=True)
    yg = f64(bits(y))
    assert np.all(np.isnan(yg[5])) and np.all(np.isnan(f64(ref["y"])[5]))
    others = np.arange(wl.T) != 5
    assert np.all(np.isfinite(yg[others]))
    assert np.array_equal(layer.routing(wl.T)["ids"].cpu().numpy(), ref["ids"])
    check_y(bits(y)[others], ref, rows=others)


def test_timeout_reports_status_and_context_survives():
    """Host-made fault: Linear-2 tiles wait for a readiness count that nothing
    reaches; the bounded wait expires (20 ms), the kernel exits cleanly and the
    status word says MOE_ERR_TIMEOUT.  The next forward on a fresh plan works."""
    wl = synth.WORKLOADS["tiny"]
    d = synth.device_inputs(wl)
    bad = _layer(wl, 0, flags=moe.MOE_FLAG_TEST_STALL, timeout_ns=20_000_000)
    bad.forward(d["x"], d["Wr"], d["W1"], d["W2"])
    assert moe.moe_get_status(bad.plan, bad._stream()) == moe.MOE_ERR_TIMEOUT
    assert moe.moe_get_status(bad.plan, bad._stream()) == moe.MOE_OK      # cleared after reading
    bad.close()
    good = _layer(wl, 0)
    y, _ = good.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    h = synth.host_inputs(wl)
    ref = oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]))
    check_y(bits(y), ref)


def test_invalid_arguments_rejected_before_launch():
    wl = synth.WORKLOADS["tiny"]
    layer = _layer(wl)
    d = synth.device_inputs(wl)
    lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    p = [d["x"].data_ptr(), lg.data_ptr(), d["Wr"].data_ptr(), d["W1"].data_ptr(), d["W2"].data_ptr(),
         y.data_ptr()]
    s = layer._stream()
    assert moe.moe_forward(layer.plan, wl.T + 1, *p, s) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_forward(layer.plan, -1, *p, s) == moe.MOE_ERR_INVALID_ARG
    bad = list(p)
    bad[0] += 2                                                  # misaligned x
    assert moe.moe_forward(layer.plan, wl.T, *bad, s) == moe.MOE_ERR_INVALID_ARG
    bad = list(p)
    bad[3] = None
    assert moe.moe_forward(layer.plan, wl.T, *bad, s) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_get_status(layer.plan, s) == moe.MOE_OK


# --------------------------------------------------------------------------- single launch
SINGLE = moe.MOE_FLAG_SINGLE_LAUNCH


@pytest.mark.parametrize("shape,schedule", [((256, 512, 256, 8, 2), 3), ((1000, 512, 256, 16, 4), 0),
                                            ((1000, 512, 256, 16, 4), 1), ((300, 768, 384, 6, 3), 2),
                                            ((33, 768, 256, 200, 8), 3), ((1, 256, 128, 1, 1), 3),
                                            ((200, 320, 192, 12, 3), 3), ((77, 64, 64, 5, 2), 0)])
def test_single_launch_bitwise_equals_multi_launch_and_oracle(shape, schedule):
    """MOE_FLAG_SINGLE_LAUNCH (the whole layer in one kernel) against the multi-launch path with
    all-canonical logits: logits, routing and y bit for bit, on several shapes (E not a multiple of
    8, one expert, one token, H and I not multiples of 256 and 128) and schedules; y against the
    full oracle; one launch."""
    T, H, I, E, k = shape
    wl = synth.Workload("single", T, H, I, E, k)
    h = synth.host_inputs(wl)
    d = {kk: from_bits(v) for kk, v in h.items() if kk != "bias"}
    multi = _layer(wl, schedule, flags=EXACT)
    y_m, lg_m = multi.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    r_m = {kk: v.cpu() for kk, v in multi.routing(T).items()}
    one = _layer(wl, schedule, flags=SINGLE)
    for _ in range(2):                                  # the plan's second forward starts from the first's state
        y_s, lg_s = one.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
        assert one.launch_count() == 1
        assert torch.equal(lg_s, lg_m), "logits differ"
        for kk, v in one.routing(T).items():
            assert torch.equal(v.cpu(), r_m[kk]), kk
        assert torch.equal(y_s.view(torch.int16), y_m.view(torch.int16)), "y differs from the multi-launch path"
    ref = oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]))
    assert np.array_equal(lg_s.cpu().numpy(), ref["logits"])
    routing_equal(one.routing(T), ref, T)
    check_y(bits(y_s), ref)
    multi.close()
    one.close()


def test_single_launch_workloads_and_inputs():
    """The single launch on the 128-token workload (full oracle on every token), with the
    caller's logits as input, and through the host-buffer entry point."""
    wl = synth.WORKLOADS["smallT"]
    d = synth.device_inputs(wl)
    one = _layer(wl, flags=SINGLE)
    y, lg = one.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    multi = _layer(wl, flags=EXACT)
    y_m, lg_m = multi.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    assert torch.equal(lg, lg_m) and torch.equal(y.view(torch.int16), y_m.view(torch.int16))
    h = synth.host_inputs(wl, weights=False)
    ref = oracle.forward(h["x"], h["Wr"], None, lambda e: _device_weights(d)("W1", e),
                         lambda e: _device_weights(d)("W2", e), wl.k, bounds=True)
    assert np.array_equal(lg.cpu().numpy(), ref["logits"])
    routing_equal(one.routing(wl.T), ref, wl.T)
    check_y(bits(y), ref)
    y2, _ = one.forward(d["x"], None, d["W1"], d["W2"], logits=lg.clone(), check=True)     # logits as input
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    x_host = d["x"].cpu().pin_memory()
    y_host = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    lg3 = torch.empty_like(lg)
    one.forward_host(x_host, d["Wr"], d["W1"], d["W2"], lg3, y_host, check=True)
    assert torch.equal(y_host.view(torch.int16), y.cpu().view(torch.int16)) and torch.equal(lg3, lg)
    one.close()
    multi.close()
    del d
    torch.cuda.empty_cache()


def test_single_launch_reports_timeout_and_bad_id():
    """Host-made faults in the single launch: a Linear-2 readiness wait that never completes
    (bounded, MOE_ERR_TIMEOUT) and an out-of-range expert id seen by Dispatch
    (MOE_ERR_DEVICE_CHECK); the context stays usable and a clean forward matches the oracle."""
    wl = synth.WORKLOADS["tiny"]
    h = synth.host_inputs(wl)
    d = {kk: from_bits(v) for kk, v in h.items() if kk != "bias"}
    bad = _layer(wl, flags=SINGLE | moe.MOE_FLAG_TEST_STALL, timeout_ns=20_000_000)
    bad.forward(d["x"], d["Wr"], d["W1"], d["W2"])
    assert moe.moe_get_status(bad.plan, bad._stream()) == moe.MOE_ERR_TIMEOUT
    bad.close()
    bad = _layer(wl, flags=SINGLE | moe.MOE_FLAG_TEST_BAD_ID)
    bad.forward(d["x"], d["Wr"], d["W1"], d["W2"])
    assert moe.moe_get_status(bad.plan, bad._stream()) == moe.MOE_ERR_DEVICE_CHECK
    bad.close()
    good = _layer(wl, flags=SINGLE)
    y, _ = good.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    ref = oracle_for(wl, h["x"], h["Wr"], None, None, full_weights=(h["W1"], h["W2"]))
    check_y(bits(y), ref)
    good.close()


def test_single_launch_phase_stamps_and_trace_layout():
    """MOE_FLAG_TRACE: the trace has one row per CTA of the larger grid plus one row of phase
    stamps; after a single-launch forward the stamps are non-decreasing and span less than the
    forward's event time, after a multi-launch forward the stamp row is zero."""
    wl = synth.WORKLOADS["tiny"]
    d = synth.device_inputs(wl)
    for flags, single in [(SINGLE | moe.MOE_FLAG_TRACE, True), (moe.MOE_FLAG_TRACE, False)]:
        layer = _layer(wl, flags=flags)
        for _ in range(2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
            b.record()
            b.synchronize()
        tr = moe.moe_trace_read(layer.plan)
        assert tr.shape[1] == 8 and tr.shape[0] >= 2
        stamps = tr[-1].astype(np.int64)
        if single:
            assert np.all(stamps[:7] > 0) and np.all(np.diff(stamps[:7]) >= 0), stamps
            assert (stamps[6] - stamps[0]) / 1e6 < a.elapsed_time(b)       # ns vs ms
            assert tr[:-1, 5].max() > 0                                      # the GEMM phase's CTA lifetimes
        else:
            assert np.all(stamps == 0)
            assert tr[:-1, 5].max() > 0
        layer.close()


@pytest.mark.parametrize("schedule,flags", [(moe.MOE_SCHED_AUTO, 0), (moe.MOE_SCHED_INTERLEAVED, 0),
                                            (moe.MOE_SCHED_PHASED, 0), (moe.MOE_SCHED_AUTO, SINGLE)])
def test_tile_trace_records_every_tile(schedule, flags):
    """moe_trace_tiles: one record per tile of the tile list and CTA rank, for every launch form:
    SM ids inside the GPU, the two CTAs of a tile on two SMs, each cluster's tiles on one SM
    pair in ticket order, start <= accumulator ready <= end, and every Linear-2 tile's
    accumulator complete no earlier than the last Linear-1 tile of its unit finished (the
    readiness dependency); without MOE_FLAG_TRACE the call is refused."""
    wl = synth.Workload("trace", 1500, 1024, 384, 24, 4)
    d = synth.device_inputs(wl)
    layer = _layer(wl, schedule, flags=flags | moe.MOE_FLAG_TRACE)
    for _ in range(2):                                   # the second forward's records start from zero
        layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    tiles, n1, workers = layer.schedule()
    tr = moe.moe_trace_tiles(layer.plan).astype(np.int64)
    assert tr.shape == (len(tiles), 2, 4)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sm, start, acc, end = tr[..., 0], tr[..., 1], tr[..., 2], tr[..., 3]
    assert np.all(start > 0) and np.all(sm < sms) and np.all(sm[:, 0] != sm[:, 1])
    assert np.all(start <= acc) and np.all(acc <= end)
    # both CTAs' loads feed the pair MMA: each accumulator is complete after both producers started
    assert np.all(acc.min(axis=1) >= start.max(axis=1))
    phased = schedule == moe.MOE_SCHED_PHASED
    idx = np.arange(len(tiles))
    first = np.where(phased & (idx >= n1), n1, 0)        # the phased schedule's second launch starts at n1
    group = (first > 0) * 10**6 + (idx - first) % workers     # (launch, cluster) of each tile
    for gk in np.unique(group):
        sel = idx[group == gk]
        for r in range(2):
            assert len(set(sm[sel, r].tolist())) == 1, "a persistent CTA stays on its SM"
            assert np.all(np.diff(start[sel, r]) >= 0) and np.all(np.diff(end[sel, r]) >= 0)
    l1_end = {}
    for i, (ph_n, e, m, g) in enumerate(tiles.tolist()):
        if ph_n & 1 == 0:
            l1_end[g] = max(l1_end.get(g, 0), int(end[i].max()))
    for i, (ph_n, e, m, g) in enumerate(tiles.tolist()):
        if ph_n & 1 == 1:
            assert acc[i].min() >= l1_end[g], (i, g)
    layer.close()
    plain = _layer(wl, schedule, flags=flags)
    plain.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    with pytest.raises(moe.MoEError):
        moe.moe_trace_tiles(plain.plan)
    plain.close()


@pytest.mark.parametrize("schedule,flags", [(moe.MOE_SCHED_AUTO, 0), (moe.MOE_SCHED_INTERLEAVED, 0),
                                            (moe.MOE_SCHED_PHASED, 0), (moe.MOE_SCHED_AUTO, EXACT),
                                            (moe.MOE_SCHED_AUTO, SINGLE)])
def test_forward_captured_in_cuda_graph(schedule, flags):
    """moe_forward is stream-ordered and never synchronises, so a forward can be captured in a
    CUDA graph: replays on new inputs copied into the captured buffers give logits, routing and y
    bitwise equal to eager forwards of the same inputs, and the device status stays clean."""
    wl = synth.Workload("graph", 700, 512, 256, 16, 4)
    layer = _layer(wl, schedule, flags=flags)
    w = synth.device_inputs(wl)
    xs = [synth.device_inputs(synth.Workload("graph", 700, 512, 256, 16, 4, seed=s))["x"] for s in (1, 2, 3)]
    x = torch.empty_like(xs[0])
    logits = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    x.copy_(xs[0])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                       # warm-up outside the capture
        layer.forward(x, w["Wr"], w["W1"], w["W2"], logits=logits, y=y)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, w["Wr"], w["W1"], w["W2"], logits=logits, y=y)
    for xi in xs:
        x.copy_(xi)
        g.replay()
        torch.cuda.synchronize()
        layer.check()
        got = (y.view(torch.int16).clone(), logits.clone(), {kk: v.cpu() for kk, v in layer.routing(wl.T).items()})
        y_e, lg_e = layer.forward(xi, w["Wr"], w["W1"], w["W2"], check=True)
        assert torch.equal(got[0], y_e.view(torch.int16)), "y of the replay differs from the eager forward"
        assert torch.equal(got[1], lg_e), "logits differ"
        for kk, v in layer.routing(wl.T).items():
            assert torch.equal(got[2][kk], v.cpu()), kk
    del g
    layer.close()


@pytest.mark.parametrize("schedule,flags", [(moe.MOE_SCHED_AUTO, 0), (moe.MOE_SCHED_INTERLEAVED, 0),
                                            (moe.MOE_SCHED_AUTO, SINGLE)])
def test_plan_reuse_long_random_sequence(schedule, flags):
    """Forty forwards of one plan with seeded random token counts (1 to 2048: every router the
    rule picks, experts of one to several units, some through the host-buffer entry point), each
    bitwise equal - logits, routing, y - to a fresh plan's forward of the same inputs: nothing a
    forward leaves in the workspace changes a later one."""
    H, I, E, k, T_max = 512, 256, 64, 4, 2048
    rng = np.random.default_rng(77)
    wl_max = synth.Workload("seq", T_max, H, I, E, k)
    w = synth.device_inputs(wl_max)
    xs = synth.device_inputs(synth.Workload("seq", T_max, H, I, E, k, seed=5))["x"]
    layer = _layer(wl_max, schedule, flags=flags)
    for step in range(40):
        T = int(rng.choice([int(rng.integers(1, 65)), int(rng.integers(65, 700)), int(rng.integers(700, T_max + 1))]))
        off = int(rng.integers(0, T_max - T + 1))
        x = xs[off:off + T].contiguous()
        host = bool(rng.integers(0, 4) == 0)
        if host:
            y = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
            lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
            layer.forward_host(x.cpu().pin_memory(), w["Wr"], w["W1"], w["W2"], lg, y, check=True)
        else:
            y, lg = layer.forward(x, w["Wr"], w["W1"], w["W2"], check=True)
        r = {kk: v.cpu() for kk, v in layer.routing(T).items()}
        fresh = _layer(synth.Workload("seq", T, H, I, E, k), schedule, flags=flags)
        y_f, lg_f = fresh.forward(x, w["Wr"], w["W1"], w["W2"], check=True)
        assert torch.equal(lg.cpu(), lg_f.cpu()), f"logits differ at step {step} (T={T})"
        for kk, v in fresh.routing(T).items():
            assert torch.equal(r[kk], v.cpu()), f"{kk} differs at step {step} (T={T})"
        assert torch.equal(y.cpu().view(torch.int16), y_f.cpu().view(torch.int16)), f"y differs at step {step} (T={T})"
        fresh.close()
    layer.close()


@pytest.mark.parametrize("flags", [0, moe.MOE_FLAG_SINGLE_LAUNCH])
def test_host_pipeline_long_random_sequence(flags):
    """Forty forwards of one MOE_FLAG_HOST_PIPELINE plan enqueued back to back with no
    synchronisation: seeded random token counts (1 to 2048, every router the rule picks),
    pipelined host forwards (routing on the plan's copy stream, y copied out beside the next
    forward) mixed with device-buffer forwards, each with its own output and logits buffers.
    After moe_host_wait every y and every logits row bitwise equal to a plain plan's forward of
    the same input."""
    H, I, E, k, T_max = 512, 256, 64, 4, 2048
    rng = np.random.default_rng(78)
    wl_max = synth.Workload("seq", T_max, H, I, E, k)
    w = synth.device_inputs(wl_max)
    xs = synth.device_inputs(synth.Workload("seq", T_max, H, I, E, k, seed=7))["x"]
    steps = []
    for _ in range(40):
        T = int(rng.choice([int(rng.integers(1, 65)), int(rng.integers(65, 700)), int(rng.integers(700, T_max + 1))]))
        off = int(rng.integers(0, T_max - T + 1))
        steps.append((T, off, bool(rng.integers(0, 3) != 0)))
    plain = _layer(wl_max, flags=flags)
    ref = []
    for T, off, _ in steps:
        y_r, lg_r = plain.forward(xs[off:off + T].contiguous(), w["Wr"], w["W1"], w["W2"], check=True)
        ref.append((y_r.cpu(), lg_r.cpu()))
    plain.close()
    layer = _layer(wl_max, flags=flags | moe.MOE_FLAG_HOST_PIPELINE)
    x_host = xs.cpu().pin_memory()       # written on the host before any pipelined forward
    outs = []
    torch.cuda.synchronize()
    for T, off, host in steps:
        lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
        if host:
            y = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
            layer.forward_host(x_host[off:off + T], w["Wr"], w["W1"], w["W2"], lg, y)
        else:
            y, _ = layer.forward(xs[off:off + T].contiguous(), w["Wr"], w["W1"], w["W2"], logits=lg)
        outs.append((y, lg))
    layer.host_wait()
    torch.cuda.current_stream().synchronize()
    for i, ((T, off, host), (y, lg), (y_r, lg_r)) in enumerate(zip(steps, outs, ref)):
        assert torch.equal(lg.cpu(), lg_r), f"logits differ at step {i} (T={T}, host={host})"
        assert torch.equal(y.cpu().view(torch.int16), y_r.view(torch.int16)), f"y differs at step {i} (T={T}, host={host})"
    layer.check()
    layer.close()


def _random_mid_cases(n: int, seed: int = 20261204):
    """Seeded mid-size layers: 1000 to 6000 tokens, H up to 3072 and I up to 1536 (multiples of
    64), up to 256 experts (T*H*E <= 3e9, so that the oracle's logits stay cheap), with every
    schedule and kernel variant and a Zipf router bias on some."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        T, H, I = int(rng.integers(1000, 6001)), 64 * int(rng.integers(8, 49)), 64 * int(rng.integers(4, 25))
        E = int(rng.integers(8, 257))
        k = int(rng.integers(1, min(8, E) + 1))
        if T * H * E > 3e9:
            continue
        out.append(dict(T=T, H=H, I=I, E=E, k=k, zipf=float(rng.choice([0.0, 1.2])), sched=int(rng.integers(0, 4)),
                        flags=[0, 0, EXACT, moe.MOE_FLAG_GEMM_COMPUTE, moe.MOE_FLAG_SINGLE_LAUNCH][int(rng.integers(0, 5))]))
    return out


@pytest.mark.parametrize("c", _random_mid_cases(16),
                         ids=lambda c: "T{T}-H{H}-I{I}-E{E}-k{k}-s{sched}-f{flags}-z{zipf}".format(**c))
def test_random_mid_shapes_sampled(c):
    """Seeded mid-size shapes (experts of several 256-row units, H and I well past one tile):
    logits and routing of every token against the oracle, y on 24 sampled tokens within the
    stated tolerance."""
    wl = synth.Workload("mid", c["T"], c["H"], c["I"], c["E"], c["k"], zipf_s=c["zipf"])
    bias = _bias(wl)
    d = synth.device_inputs(wl)
    layer = _layer(wl, c["sched"], flags=c["flags"], bias=bias)
    y, logits = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    h = synth.host_inputs(wl, weights=False)
    lg_ref = oracle.router_logits(h["x"], h["Wr"], bias)
    tok = sample_tokens(c["T"], 24, seed=c["T"])
    ref = oracle.forward(h["x"], h["Wr"], bias, lambda e: _device_weights(d)("W1", e),
                         lambda e: _device_weights(d)("W2", e), wl.k, tokens=tok, logits=lg_ref, bounds=True)
    if c["flags"] & (EXACT | moe.MOE_FLAG_SINGLE_LAUNCH):     # all logits canonical
        assert np.array_equal(logits.cpu().numpy(), lg_ref)
    else:
        check_logits(logits.cpu().numpy(), ref, h["x"], h["Wr"], layer.router_bound(c["T"]), bias)
    routing_equal(layer.routing(c["T"]), ref, c["T"])
    check_y(bits(y)[tok], ref, what=f"T={c['T']}")
    del d
    layer.close()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,schedule,zipf", [(65536, moe.MOE_SCHED_AUTO, 0.0), (131072, moe.MOE_SCHED_AUTO, 1.2),
                                             (65536, moe.MOE_SCHED_INTERLEAVED, 0.0)])
def test_many_tokens_routing_and_sampled_y(T, schedule, zipf):
    """Batches far above the five workloads (65536 and 131072 tokens: 512 and 1024 chunks of 128
    tokens, half a million and a million routed rows, the skewed one with its hottest expert in
    every token's top-k): routing of every token bit-exact against the oracle, y on 48 sampled
    tokens within the stated tolerance."""
    wl = synth.Workload("many", T, 1024, 256, 64, 8, zipf_s=zipf)
    bias = _bias(wl)
    d = synth.device_inputs(wl)
    layer = _layer(wl, schedule, bias=bias)
    y, logits = layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    h = synth.host_inputs(wl, weights=False)
    lg_ref = oracle.router_logits(h["x"], h["Wr"], bias)
    tok = sample_tokens(T, 48, seed=3)
    ref = oracle.forward(h["x"], h["Wr"], bias, lambda e: _device_weights(d)("W1", e),
                         lambda e: _device_weights(d)("W2", e), wl.k, tokens=tok, logits=lg_ref, bounds=True)
    check_logits(logits.cpu().numpy(), ref, h["x"], h["Wr"], layer.router_bound(T), bias)
    routing_equal(layer.routing(T), ref, T)
    check_y(bits(y)[tok], ref, what=f"T={T}")
    del d
    layer.close()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,pin", [(1000, True), (100, True), (1000, False)])
def test_host_forward_waits_for_stream_ordered_input(T, pin):
    """By default moe_forward_host is stream-ordered like any other operation: an x_host written
    by a device-to-host copy enqueued on the stream just before the call is the input the forward
    sees (tensor-core router in ranges, the canonical task router, pageable staging)."""
    wl = synth.Workload("strict", T, 1024, 256, 64, 4)
    w = synth.device_inputs(wl)
    xb = synth.device_inputs(synth.Workload("strict", T, 1024, 256, 64, 4, seed=9))["x"]
    layer = _layer(wl)
    y_a, _ = layer.forward(w["x"], w["Wr"], w["W1"], w["W2"], check=True)
    y_b, _ = layer.forward(xb, w["Wr"], w["W1"], w["W2"], check=True)
    x_host = torch.empty((T, wl.H), dtype=torch.bfloat16, pin_memory=pin)
    y_host = torch.empty((T, wl.H), dtype=torch.bfloat16, pin_memory=pin)
    lg = torch.empty((T, wl.E), dtype=torch.float32, device="cuda")
    x_host.copy_(w["x"].cpu())
    layer.forward_host(x_host, w["Wr"], w["W1"], w["W2"], lg, y_host)
    x_host.copy_(xb, non_blocking=pin)          # stream-ordered write of the next input
    layer.forward_host(x_host, w["Wr"], w["W1"], w["W2"], lg, y_host, check=True)
    assert torch.equal(y_host.view(torch.int16), y_b.cpu().view(torch.int16)), "the forward read a stale x_host"
    layer.close()


def test_host_pipeline_back_to_back():
    """MOE_FLAG_HOST_PIPELINE: back-to-back host forwards with no synchronisation between them,
    alternating two page-locked inputs written on the host beforehand, each with its own output:
    every y bitwise equal to the device forward of its input."""
    wl = synth.Workload("pipe", 1000, 1024, 256, 64, 4)
    w = synth.device_inputs(wl)
    xs = [w["x"], synth.device_inputs(synth.Workload("pipe", 1000, 1024, 256, 64, 4, seed=4))["x"]]
    ref = _layer(wl)
    y_ref = [ref.forward(x, w["Wr"], w["W1"], w["W2"], check=True)[0].cpu() for x in xs]
    ref.close()
    layer = _layer(wl, flags=moe.MOE_FLAG_HOST_PIPELINE)
    x_host = [x.cpu().pin_memory() for x in xs]
    lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    y_host = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory() for _ in range(6)]
    for i in range(6):
        layer.forward_host(x_host[i % 2], w["Wr"], w["W1"], w["W2"], lg, y_host[i])
    layer.check()
    for i in range(6):
        assert torch.equal(y_host[i].view(torch.int16), y_ref[i % 2].view(torch.int16)), f"forward {i}"
    layer.close()


def test_host_pipeline_mixed_with_device_forwards():
    """A plan with MOE_FLAG_HOST_PIPELINE serving device-buffer and pipelined host-buffer
    forwards in turn: a host forward's routing, which runs on the plan's own stream, must still
    wait for the previous device forward's Dispatch (the last reader of the routing buffers).
    Every y bitwise equal to a plain plan's forward of the same input."""
    wl = synth.Workload("pipe", 1000, 1024, 256, 64, 4)
    w = synth.device_inputs(wl)
    xs = [w["x"], synth.device_inputs(synth.Workload("pipe", 1000, 1024, 256, 64, 4, seed=6))["x"]]
    ref = _layer(wl)
    y_ref = [ref.forward(x, w["Wr"], w["W1"], w["W2"], check=True)[0].cpu() for x in xs]
    ref.close()
    layer = _layer(wl, flags=moe.MOE_FLAG_HOST_PIPELINE)
    x_host = [x.cpu().pin_memory() for x in xs]
    lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    outs = []
    for i, (xi, host) in enumerate([(0, False), (1, True), (1, False), (0, True), (0, False), (1, True)]):
        if host:
            yh = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
            layer.forward_host(x_host[xi], w["Wr"], w["W1"], w["W2"], lg, yh)
            outs.append((xi, yh))
        else:
            outs.append((xi, layer.forward(xs[xi], w["Wr"], w["W1"], w["W2"])[0]))
    layer.host_wait()
    torch.cuda.current_stream().synchronize()
    for i, (xi, y) in enumerate(outs):
        assert torch.equal(y.cpu().view(torch.int16), y_ref[xi].view(torch.int16)), f"forward {i}"
    layer.check()
    layer.close()


@pytest.mark.parametrize("extra", [0, moe.MOE_FLAG_SINGLE_LAUNCH])
def test_host_pipeline_output_copies(extra):
    """MOE_FLAG_HOST_PIPELINE output side: y leaves through the plan's alternating staging buffers
    on its own stream; after moe_host_wait on the caller's stream (no moe_get_status) every
    y_host of a back-to-back run holds its forward's y - with token counts below T_max (the
    tensor-core and the canonical task router), a pageable y_host mixed in (that one
    stream-ordered, through the first staging buffer), multi-launch and single launch."""
    wl = synth.Workload("pipe", 1000, 1024, 256, 64, 4)
    w = synth.device_inputs(wl)
    xs = [w["x"], synth.device_inputs(synth.Workload("pipe", 1000, 1024, 256, 64, 4, seed=5))["x"]]
    ref = _layer(wl)
    runs = [(0, 1000, True), (1, 1000, True), (0, 300, True), (1, 1000, False), (1, 700, True), (0, 1000, True),
            (1, 1000, True)]
    y_ref = {}
    for xi, T, _ in runs:
        if (xi, T) not in y_ref:
            y_ref[(xi, T)] = ref.forward(xs[xi][:T], w["Wr"], w["W1"], w["W2"], check=True)[0].cpu()
    ref.close()
    layer = _layer(wl, flags=moe.MOE_FLAG_HOST_PIPELINE | extra)
    x_host = [x.cpu().pin_memory() for x in xs]
    lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda")
    y_host = []
    for _, T, pin in runs:
        yh = torch.full((T, wl.H), -1, dtype=torch.int16)
        y_host.append((yh.pin_memory() if pin else yh).view(torch.bfloat16))
    for (xi, T, _), yh in zip(runs, y_host):
        layer.forward_host(x_host[xi][:T], w["Wr"], w["W1"], w["W2"], lg[:T], yh)
    layer.host_wait()
    torch.cuda.current_stream().synchronize()
    for i, ((xi, T, _), yh) in enumerate(zip(runs, y_host)):
        assert torch.equal(yh.view(torch.int16), y_ref[(xi, T)].view(torch.int16)), f"forward {i} (T={T})"
    layer.check()
    layer.close()
