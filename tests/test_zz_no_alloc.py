"""The batch-1 decode forward that allocates nothing (moe_forward_decode_static).

It exists for callers that cannot provide scratch memory (a plugin handed only input and
output device pointers by a host program that owns every allocation, or a loop that must not
allocate once running): its scratch is a fixed array inside the library.  This file is
collected last so that a run stopping at its first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import quantized_grouped_gemm_gb300 as moe
from moe_workload import configs, gen
from gpu_helpers import DeviceLayer, assert_output_close, assert_routing_equal, routing_to_host, to_dev, y_to_f64

pytestmark = pytest.mark.gpu


NO_ALLOC_CASES = [
    # d=1024, I=256: the one-launch decode kernel
    configs.custom_workload("noalloc_t1_d1024_i256", T=1, d=1024, I=256),
    # d=256, I=1152: (k+1) I / 128 = 81 units do not fit at once, so the three decode kernels
    # run on the static array's layout (about 106 KB of its 128 KB)
    configs.custom_workload("noalloc_t1_d256_i1152", T=1, d=256, I=1152),
]


@pytest.mark.parametrize("wl", NO_ALLOC_CASES, ids=lambda w: w.name)
def test_static_scratch_decode_matches_workspace_forward_two_calls(wl):
    sh = wl.shape
    lay = configs.make_layer(wl)
    shp = moe.shape(1, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    dl = DeviceLayer(shp, lay)
    xs = gen.normal_bf16(wl.seed, 77, (2, sh.d))
    for call in range(2):                       # two calls in a row share the static array
        x = np.ascontiguousarray(xs[call:call + 1])
        xd = to_dev(x)
        rt_ws, rt_st = moe.Routing(1), moe.Routing(1)
        ws = moe.workspace(shp)
        y_ws = torch.empty(1, sh.d, dtype=torch.int16, device="cuda")
        y_st = torch.empty(1, sh.d, dtype=torch.int16, device="cuda")
        moe.moe_forward(shp, xd, dl.w_router, None, dl.packed_routed, dl.packed_shared, rt_ws, ws, y_ws)
        moe.moe_forward_decode_static(shp, xd, dl.w_router, None, dl.packed_routed, dl.packed_shared, rt_st, y_st)
        torch.cuda.synchronize()
        assert moe.moe_read_status(ws)[0] == moe.MOE_OK
        a, b = routing_to_host(rt_st, 1), routing_to_host(rt_ws, 1)
        for key in ("topk_idx", "counts", "offsets", "perm", "pos", "tiles"):
            assert np.array_equal(a[key], b[key]), key
        assert np.abs(a["topk_w"] - b["topk_w"]).max() <= 1e-5
        assert_output_close(y_to_f64(y_st), y_to_f64(y_ws), f"static-scratch call {call}")
        # and both against the oracle: routing bit-exact, output within the layer tolerance
        ref = oracle.route(x, lay.w_router)
        assert_routing_equal(a, ref)
        out = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
        assert_output_close(y_to_f64(y_st), out, f"static-scratch call {call} vs oracle")
