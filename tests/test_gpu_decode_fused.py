"""GPU parity of the one-launch decode kernel (moe_forward with T = 1) against the CPU oracle.

Same bars as the other parity tests: routing bit-exact, routing weights within 1e-5, the layer
output within max |err| <= 2e-2 (|ref| + 1e-2) and relative Frobenius error <= 5e-3.  Each
case also checks how many kernels the call launched (1 for the fused path, 3 for the GEMV
path), so a silent fallback shows up.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_grouped_gemm_gb300 as moe
from moe_workload import configs
from gpu_helpers import (DeviceLayer, assert_output_close, assert_routing_equal, routing_to_host, to_dev,
                         y_to_f64)

pytestmark = pytest.mark.gpu


def _layer(name, d, I, seed=0, layer=0):
    wl = configs.custom_workload(name, T=1, d=d, I=I, seed=seed)
    lay = configs.make_layer(wl, layer=layer)
    shp = moe.shape(1, d, 256, 8, I, I)
    return wl, lay, shp, DeviceLayer(shp, lay)


def _forward(shp, dl, xd, rt, ws, y, opts=None, stream=None):
    n0 = moe.moe_launch_count()
    moe.moe_forward(shp, xd, dl.w_router, dl.bias, dl.packed_routed, dl.packed_shared, rt, ws, y, opts, stream)
    return moe.moe_launch_count() - n0


def _check(x, lay, rt, y, what):
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    assert_routing_equal(routing_to_host(rt, 1), ref)
    out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
    return assert_output_close(y_to_f64(y)[:1], out_ref, what)


# (d, I): one h slice; two; four; six; long rows (ring refills, router rows beyond registers)
SHAPES = [(512, 128), (256, 256), (2048, 512), (1024, 768), (4096, 256), (7168, 256)]


@pytest.mark.parametrize("d,I", SHAPES, ids=lambda v: str(v))
def test_fused_decode_matches_oracle(d, I):
    wl, lay, shp, dl = _layer(f"fz_d{d}_i{I}", d, I)
    x = configs.make_decode_x(wl, 1)
    rt, ws = moe.Routing(1), moe.workspace(shp)
    y = torch.empty(1, d, dtype=torch.int16, device="cuda")
    n = _forward(shp, dl, to_dev(x), rt, ws, y)
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK
    assert n == 1, f"expected the one-launch decode kernel, got {n} launches"
    _check(x, lay, rt, y, f"fused d={d} I={I}")


def test_fused_and_gemv_paths_agree_with_oracle():
    wl, lay, shp, dl = _layer("fz_vs_gemv", 2048, 512, seed=5)
    x = configs.make_decode_x(wl, 1)
    for path, launches in ((moe.DECODE_AUTO, 1), (moe.DECODE_GEMV, 3)):
        rt, ws = moe.Routing(1), moe.workspace(shp)
        y = torch.empty(1, 2048, dtype=torch.int16, device="cuda")
        n = _forward(shp, dl, to_dev(x), rt, ws, y, moe.options(decode_path=path))
        assert moe.moe_read_status(ws)[0] == moe.MOE_OK
        assert n == launches
        _check(x, lay, rt, y, f"decode path {path}")


def test_fused_decode_many_steps_one_workspace():
    """The grid's counters reset themselves: many tokens through one workspace."""
    wl = configs.WORKLOADS["decode_t1_d2048"]
    sh = wl.shape
    lay = configs.make_layer(wl)
    shp = moe.shape(1, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    dl = DeviceLayer(shp, lay)
    xs = configs.make_decode_x(wl, 6)
    rt, ws = moe.Routing(1), moe.workspace(shp)
    ys = []
    for s in range(6):
        y = torch.empty(1, sh.d, dtype=torch.int16, device="cuda")
        assert _forward(shp, dl, to_dev(np.ascontiguousarray(xs[s:s + 1])), rt, ws, y) == 1
        ys.append((y, {k: v.clone() for k, v in vars(rt).items() if isinstance(v, torch.Tensor)}))
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK
    for s, (y, saved) in enumerate(ys):
        r = moe.Routing(1)
        for k, v in saved.items():
            getattr(r, k).copy_(v)
        _check(np.ascontiguousarray(xs[s:s + 1]), lay, r, y, f"step {s}")


def test_fused_decode_chained_layers_in_a_graph():
    """Four launches captured in one CUDA graph: layer 0 then layer 1 reading layer 0's output,
    twice over (two tokens).  The kernels start their weight prologue before the previous
    kernel ends (programmatic dependent launch) and must still read x only after it is
    written.  (Chains stop at two layers: without the normalisation that sits between MoE
    layers in a model, SwiGLU grows the activations about six-fold per layer.)"""
    wl = configs.WORKLOADS["decode_t1_d2048"]
    sh = wl.shape
    shp = moe.shape(1, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    lays = [configs.make_layer(wl, layer=i) for i in range(2)]
    dls = [DeviceLayer(shp, l) for l in lays]
    xs = configs.make_decode_x(wl, 2)
    z = lambda: torch.zeros(1, sh.d, dtype=torch.int16, device="cuda")
    xa, xb = to_dev(np.ascontiguousarray(xs[0:1])), to_dev(np.ascontiguousarray(xs[1:2]))
    ya0, ya1, yb0, yb1 = z(), z(), z(), z()
    plan = [(0, xa, ya0), (1, ya0, ya1), (0, xb, yb0), (1, yb0, yb1)]
    rts = [moe.Routing(1) for _ in plan]
    ws = moe.workspace(shp)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for (li, xin, yout), rt in zip(plan, rts):   # warm up outside the capture
            _forward(shp, dls[li], xin, rt, ws, yout, None, s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            for (li, xin, yout), rt in zip(plan, rts):
                _forward(shp, dls[li], xin, rt, ws, yout, None, s)
        for b in (ya0, ya1, yb0, yb1):
            b.zero_()
        g.replay()
        g.replay()
    s.synchronize()
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK
    for (li, xin, yout), rt in zip(plan, rts):
        _check(xin.cpu().numpy().view(np.uint16), lays[li], rt, yout, f"layer {li}")


def test_fused_decode_fallback_scale_encoding_and_bias():
    """Large scales (the 128 + q encoding) and a logit bias through the fused kernel."""
    wl, lay, shp, _ = _layer("fz_big", 512, 256, seed=9)
    big = np.uint16(0x3D80)
    lay.routed.up.scales[11, 40, 3] = big
    lay.shared.gate.scales[0, 2, 1] = big
    lay.logit_bias = configs.zipf_logit_bias(3, 256, 1.2, 1.0)
    dl = DeviceLayer(shp, lay)
    assert int(dl.packed_routed[:4].view(torch.int32).item()) == 1
    x = configs.make_decode_x(wl, 1)
    rt, ws = moe.Routing(1), moe.workspace(shp)
    y = torch.empty(1, 512, dtype=torch.int16, device="cuda")
    assert _forward(shp, dl, to_dev(x), rt, ws, y) == 1
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK
    _check(x, lay, rt, y, "fallback encoding + bias")


def test_gemv_decode_path_on_request():
    """decode_path = DECODE_GEMV: the three decode kernels run (route, gate/up GEMV, down GEMV)
    and match the oracle on a shape the fused kernel would also take."""
    wl, lay, shp, dl = _layer("fz_i384", 512, 384, seed=2)
    x = configs.make_decode_x(wl, 1)
    for path, launches in ((moe.DECODE_GEMV, 3), (moe.DECODE_AUTO, 1)):
        rt, ws = moe.Routing(1), moe.workspace(shp)
        y = torch.empty(1, 512, dtype=torch.int16, device="cuda")
        assert _forward(shp, dl, to_dev(x), rt, ws, y, moe.options(decode_path=path)) == launches
        assert moe.moe_read_status(ws)[0] == moe.MOE_OK
        _check(x, lay, rt, y, f"I=384 path {path}")


def test_decode_largest_intermediate_falls_back_to_gemv():
    """I = 8192 (the largest supported): the one-launch kernel's grid (9 slots x 64 h slices)
    cannot be resident at once, so moe_forward runs the three decode kernels; routing exact,
    output within tolerance."""
    wl, lay, shp, dl = _layer("fz_d256_i8192", 256, 8192, seed=9)
    x = configs.make_decode_x(wl, 1)
    rt, ws = moe.Routing(1), moe.workspace(shp)
    y = torch.empty(1, 256, dtype=torch.int16, device="cuda")
    n = _forward(shp, dl, to_dev(x), rt, ws, y)
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK
    assert n == 3, f"expected the three decode kernels, got {n} launches"
    _check(x, lay, rt, y, "decode d=256 I=8192")
