"""moe_dispatch_static: the Dispatch sort for callers that cannot allocate device
memory - code running under an allocator that owns the whole device pool or a fixed
memory budget, where a cudaMalloc behind its back fails or breaks the accounting, and
paths that must not take the implicit synchronisation of cudaMalloc/cudaFree.

Its output must equal the Dispatch of moe_forward (the existing entry point) and the
oracle's stable counting sort exactly (integer work), on two calls in a row, the second
starting from the first call's leftover scratch.  Also covered: the scalar tail path
(T*k not a multiple of 4, ids not 16-byte aligned), E = 256 (the scratch limit), no
weights, T = 0, and expert ids outside [0, E), which get row_of = -1 and are left out
of offsets[E].

This file is collected last on purpose, so a failure here stops a -x run only after
every other test has run."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_top_gb300 as moe
import oracle
import synth

pytestmark = pytest.mark.gpu

FILL = -7


def _dispatch_static(ids, w, E, k, T=None):
    """Call the entry point; ids/w are device tensors (any alignment the header allows)."""
    T = ids.numel() // k if T is None else T
    R = T * k
    out = dict(offsets=torch.full((E + 1,), FILL, dtype=torch.int32, device="cuda"),
               row_pair=torch.full((max(R, 1),), FILL, dtype=torch.int32, device="cuda"),
               row_of=torch.full((max(R, 1),), FILL, dtype=torch.int32, device="cuda"),
               row_w=torch.full((max(R, 1),), float(FILL), dtype=torch.float32, device="cuda"))
    st = moe.moe_dispatch_static(T, E, k, ids.data_ptr() if R else None, w.data_ptr() if w is not None else None,
                                 out["offsets"].data_ptr(), out["row_pair"].data_ptr(), out["row_of"].data_ptr(),
                                 out["row_w"].data_ptr() if w is not None else None,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    torch.cuda.synchronize()
    return {kk: v.cpu().numpy() for kk, v in out.items()}


def _against_oracle(got, ids_np, w_np, E, check_w=True):
    """Compare with the oracle's stable counting sort.  Out-of-range ids are given the
    extra expert E for the oracle, whose rows then come after every placed row."""
    T, k = ids_np.shape
    R = T * k
    bad = (ids_np < 0) | (ids_np >= E)
    mapped = np.where(bad, E, ids_np).astype(np.int32)
    counts, offsets, row_pair, row_of = oracle.dispatch(mapped, E + 1)
    placed = int(offsets[E])
    assert np.array_equal(got["offsets"], offsets[:E + 1]), "offsets"
    assert np.array_equal(got["row_pair"][:placed], row_pair[:placed]), "row_pair"
    ro = np.where(bad.reshape(-1), -1, row_of)
    assert np.array_equal(got["row_of"][:R], ro), "row_of"
    if placed < R:   # rows past offsets[E] are not written
        assert np.all(got["row_pair"][placed:R] == FILL)
    if check_w:
        assert np.array_equal(got["row_w"][:placed], w_np.reshape(-1)[row_pair[:placed]]), "row_w"
    return placed


@pytest.mark.parametrize("name", ["fine", "skew"])
def test_dispatch_static_matches_forward_and_oracle(name):
    moe.build()
    oracle.build()
    wl = synth.WORKLOADS[name]
    bias = synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None
    d = synth.device_inputs(wl)
    layer = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, schedule=1), 0, router_bias=bias)
    layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    ref = {kk: v.cpu().numpy() for kk, v in layer.routing(wl.T).items()}
    ids_d = torch.from_numpy(ref["ids"]).cuda()
    w_d = torch.from_numpy(ref["w"]).cuda()
    for _ in range(2):                       # the second call reuses the first call's scratch
        got = _dispatch_static(ids_d, w_d, wl.E, wl.k)
        for key in ("offsets", "row_pair", "row_of"):
            assert np.array_equal(got[key], ref[key]), key            # the existing entry point's Dispatch
        assert _against_oracle(got, ref["ids"], ref["w"], wl.E) == wl.T * wl.k
    assert moe.moe_get_status(layer.plan, layer._stream()) == moe.MOE_OK
    layer.close()


@pytest.mark.parametrize("T,E,k,misalign,with_w", [(1001, 37, 3, False, True), (1001, 37, 3, True, True),
                                                    (4099, 256, 8, True, False), (20000, 256, 5, False, True),
                                                    (1, 1, 1, True, False)])
def test_dispatch_static_shapes(T, E, k, misalign, with_w):
    """Random ids: the tail path (T*k % 4 != 0), ids 4 bytes off 16-byte alignment, the largest E,
    no weights; two calls in a row against the oracle."""
    moe.build()
    rng = np.random.default_rng(T + E + k)
    ids_np = rng.integers(0, E, size=(T, k), dtype=np.int32)
    w_np = rng.random((T, k), dtype=np.float32)
    off = 1 if misalign else 0
    buf = torch.zeros(T * k + 4, dtype=torch.int32, device="cuda")
    ids_d = buf[off:off + T * k]
    ids_d.copy_(torch.from_numpy(ids_np.reshape(-1)))
    assert (ids_d.data_ptr() % 16 != 0) == misalign
    w_d = torch.from_numpy(w_np).cuda() if with_w else None
    for _ in range(2):
        got = _dispatch_static(ids_d, w_d, E, k, T=T)
        assert _against_oracle(got, ids_np, w_np, E, check_w=with_w) == T * k
        if not with_w:
            assert np.all(got["row_w"] == FILL)


def test_dispatch_static_out_of_range_ids():
    """Ids planted outside [0, E) on the host (negative, E, far above E): those pairs get
    row_of = -1, offsets[E] counts only the placed pairs, every other pair is placed as the
    oracle places it; a clean call afterwards is exact again."""
    moe.build()
    T, E, k = 777, 19, 4
    rng = np.random.default_rng(3)
    ids_np = rng.integers(0, E, size=(T, k), dtype=np.int32)
    clean = ids_np.copy()
    ids_np[0, 0], ids_np[5, 3], ids_np[400, 1], ids_np[776, 2] = -1, E, 1 << 20, -(1 << 30)
    w_np = rng.random((T, k), dtype=np.float32)
    got = _dispatch_static(torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda(), E, k)
    placed = _against_oracle(got, ids_np, w_np, E)
    assert placed == T * k - 4 and got["offsets"][E] == placed
    assert np.all(got["row_of"][[0, 5 * k + 3, 400 * k + 1, 776 * k + 2]] == -1)
    got = _dispatch_static(torch.from_numpy(clean).cuda(), torch.from_numpy(w_np).cuda(), E, k)
    assert _against_oracle(got, clean, w_np, E) == T * k


def test_dispatch_static_zero_tokens_and_limits():
    moe.build()
    E = 12
    got = _dispatch_static(torch.zeros(1, dtype=torch.int32, device="cuda"), None, E, 2, T=0)
    assert np.all(got["offsets"] == 0)
    assert np.all(got["row_pair"] == FILL) and np.all(got["row_of"] == FILL)
    ids = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    z = torch.zeros(16, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert moe.moe_dispatch_static(4, 300, 2, ids.data_ptr(), None, z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                   None, s) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_dispatch_static(4, 8, 9, ids.data_ptr(), None, z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                   None, s) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_dispatch_static(4, 8, 2, ids.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                   None, s) == moe.MOE_ERR_INVALID_ARG    # w without row_w
