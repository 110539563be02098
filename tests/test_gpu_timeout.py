"""A bounded wait inside the grouped-FFN kernel that runs out: the kernel records a timeout in
the workspace status word and unwinds (no trap, no unbounded wait), the host reads
MOE_ERR_DEVICE_TIMEOUT, and the same process then gets correct results from a re-zeroed
workspace.

The failure is made by a separate copy of the library built for this test only: its waits
give up after 2e7 SM cycles (about 10 ms) instead of about 2 s, and the token-row producer of
CTA 0 never arms the "ready" barrier of its fourth K block, so the MMA threads' wait on it can
never complete.  The product library is built without either change.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import quantized_grouped_gemm_gb300 as moe
from quantized_grouped_gemm_gb300 import _lib, build as build_mod
from moe_workload import configs
from gpu_helpers import (DeviceLayer, assert_output_close, assert_routing_equal, routing_to_host, run_forward,
                         to_dev, y_to_f64)

pytestmark = pytest.mark.gpu

_DIR = os.path.join(os.path.dirname(build_mod.__file__), "_build", "timeout_test")


def _timeout_library():
    path = os.path.join(_DIR, "libmoe_timeout.so")
    build_mod.build(out=path, build_dir=os.path.join(_DIR, "objs"),
                    defines=["MOE_WAIT_LIMIT_CYCLES=20000000ll", "MOE_TEST_DROP_TOKEN_BLOCK=3"])
    L = ctypes.CDLL(path)
    for name, (res, args) in _lib._SIG.items():
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    return L


def test_ffn_wait_timeout_is_reported_and_workspace_recovers():
    L = _timeout_library()
    wl = configs.custom_workload("timeout_t256_d512_i128", T=256, d=512, I=128, seed=51)
    sh = wl.shape
    lay = configs.make_layer(wl)
    x = configs.make_x(wl)
    shp = moe.shape(sh.T, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    dl = DeviceLayer(shp, lay)            # packed by the product library (same packed format)
    xd = to_dev(x)
    rt = moe.Routing(sh.T)
    ws = moe.workspace(shp)
    y = torch.empty(sh.T, sh.d, dtype=torch.int16, device="cuda")
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.moe_forward(ctypes.byref(shp), P(xd), P(dl.w_router), None, P(dl.packed_routed), P(dl.packed_shared),
                       rt.ref(), P(ws), ws.numel(), P(y), None, st)
    assert rc == moe.MOE_OK                      # the launches themselves succeed
    bits = ctypes.c_int(0)
    rc = L.moe_read_status(P(ws), st, ctypes.byref(bits))
    assert rc == moe.MOE_ERR_DEVICE_TIMEOUT and bits.value & moe.MOE_STATUS_TIMEOUT, (rc, bits.value)
    torch.cuda.synchronize()                     # the context is still usable
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK    # read and cleared
    # after a timeout the workspace counters are undefined: zero it, then the product library
    # gives the oracle's routing and outputs on the same buffers
    ws.zero_()
    moe.moe_forward(shp, xd, dl.w_router, None, dl.packed_routed, dl.packed_shared, rt, ws, y)
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK
    ref = oracle.route(x, lay.w_router)
    assert_routing_equal(routing_to_host(rt, sh.T), ref)
    out = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
    assert_output_close(y_to_f64(y), out, "after the timeout, re-zeroed workspace")
