"""moe_dispatch_static: the Dispatch sort for callers that cannot allocate device
memory (a foreign allocator owning the pool or a fixed budget, paths that must not
take cudaMalloc's implicit synchronisation).  Its
output must equal the Dispatch of moe_forward exactly (integer work), on two calls
in a row, the second starting from the first call's leftover scratch."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_top_gb300 as moe
import synth

pytestmark = pytest.mark.gpu


def _dispatch_static(ids, w, E, k):
    T = ids.shape[0]
    R = T * k
    out = dict(offsets=torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
               row_pair=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
               row_of=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
               row_w=torch.full((R,), -7.0, dtype=torch.float32, device="cuda"))
    st = moe.moe_dispatch_static(T, E, k, ids.data_ptr(), w.data_ptr(), out["offsets"].data_ptr(),
                                 out["row_pair"].data_ptr(), out["row_of"].data_ptr(),
                                 out["row_w"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    return out


@pytest.mark.parametrize("name", ["fine", "skew"])
def test_dispatch_static_matches_forward(name):
    moe.build()
    wl = synth.WORKLOADS[name]
    bias = synth.zipf_bias(wl.E, wl.zipf_s) if wl.zipf_s else None
    d = synth.device_inputs(wl)
    layer = moe.MoELayer(moe.MoEConfig(wl.T, wl.H, wl.I, wl.E, wl.k, schedule=1), 0, router_bias=bias)
    layer.forward(d["x"], d["Wr"], d["W1"], d["W2"], check=True)
    ref = layer.routing(wl.T)
    for _ in range(2):                       # the second call reuses the first call's scratch
        got = _dispatch_static(ref["ids"], ref["w"], wl.E, wl.k)
        torch.cuda.synchronize()
        for key in ("offsets", "row_pair", "row_of"):
            assert torch.equal(got[key], ref[key]), key
        w_rows = ref["w"].reshape(-1)[ref["row_pair"].long()]
        assert torch.equal(got["row_w"], w_rows)
    assert moe.moe_get_status(layer.plan, layer._stream()) == moe.MOE_OK
    layer.close()


def test_dispatch_static_limits():
    moe.build()
    ids = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    z = torch.zeros(16, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert moe.moe_dispatch_static(4, 300, 2, ids.data_ptr(), None, z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                   None, s) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_dispatch_static(4, 8, 9, ids.data_ptr(), None, z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                   None, s) == moe.MOE_ERR_INVALID_ARG
