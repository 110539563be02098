"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Routing (top-k experts, counts, offsets, perm, pos, block map) must match bit-exactly;
routing weights within 1e-5; the layer output within max |err| <= 2e-2 (|ref| + 1e-2)
elementwise and relative Frobenius error <= 5e-3 against the oracle's fp64 result.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_grouped_gemm_gb300 as moe
from moe_workload import configs, gen
from gpu_helpers import (DeviceLayer, assert_output_close, assert_routing_equal, routing_to_host, run_forward,
                         to_dev, y_to_f64)

pytestmark = pytest.mark.gpu


def _setup(wl, x_rows=None):
    sh = wl.shape
    lay = configs.make_layer(wl)
    x = configs.make_x(wl) if x_rows is None else x_rows
    T = x.shape[0]
    shp = moe.shape(T, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    return shp, lay, x, DeviceLayer(shp, lay)


SMALL = [
    configs.WORKLOADS["tiny_t128_d512"],
    configs.custom_workload("ragged_t200_d512_i256", T=200, d=512, I=256),
    configs.custom_workload("t33_d256_i128", T=33, d=256, I=128),
    configs.custom_workload("t2_d512_i128", T=2, d=512, I=128),
    configs.custom_workload("t1_d512_i128", T=1, d=512, I=128),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("split", [False, True], ids=["forward", "three_calls"])
def test_small_full_parity(wl, split):
    shp, lay, x, dl = _setup(wl)
    rt, ws, y = run_forward(shp, dl, to_dev(x), split_calls=split)
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    assert_routing_equal(routing_to_host(rt, shp.T), ref)
    out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
    assert_output_close(y_to_f64(y)[: shp.T], out_ref, wl.name)


def test_decode_t1_layer_steps():
    wl = configs.WORKLOADS["decode_t1_d2048"]
    sh = wl.shape
    lay = configs.make_layer(wl)
    xs = configs.make_decode_x(wl, 3)
    shp = moe.shape(1, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    dl = DeviceLayer(shp, lay)
    for s in range(3):
        x = np.ascontiguousarray(xs[s:s + 1])
        rt, ws, y = run_forward(shp, dl, to_dev(x))
        ref = oracle.route(x, lay.w_router, lay.logit_bias)
        assert_routing_equal(routing_to_host(rt, 1), ref)
        out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
        assert_output_close(y_to_f64(y)[:1], out_ref, f"decode step {s}")


def test_decode_path_equals_prefill_path_for_one_token():
    wl = configs.custom_workload("t1_d1024_i256", T=1, d=1024, I=256)
    shp, lay, x, dl = _setup(wl)
    _, _, y_dec = run_forward(shp, dl, to_dev(x), opts=moe.options(decode_max_tokens=1))
    _, _, y_pre = run_forward(shp, dl, to_dev(x), opts=moe.options(decode_max_tokens=0))
    ref = oracle.route(x, lay.w_router)
    out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
    assert_output_close(y_to_f64(y_dec)[:1], out_ref, "decode kernels")
    assert_output_close(y_to_f64(y_pre)[:1], out_ref, "prefill kernels")


def test_concentrated_routing_big_groups():
    """A logit bias sends every token to experts 0..7: eight groups of T rows (N tiles of
    256 + remainder), 248 empty experts."""
    wl = configs.custom_workload("conc_t600_d512_i128", T=600, d=512, I=128)
    sh = wl.shape
    lay = configs.make_layer(wl)
    lay.logit_bias = np.where(np.arange(256) < 8, 50.0, 0.0).astype(np.float32)
    x = configs.make_x(wl)
    shp = moe.shape(sh.T, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    dl = DeviceLayer(shp, lay)
    rt, ws, y = run_forward(shp, dl, to_dev(x))
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    assert (ref["counts"][:8] == 600).all() and ref["counts"][8:].sum() == 0
    assert_routing_equal(routing_to_host(rt, shp.T), ref)
    toks = np.arange(0, 600, 37, dtype=np.int32)
    out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared, toks)
    assert_output_close(y_to_f64(y)[toks], out_ref, "concentrated")


def test_tile_rows_option_changes_only_block_map():
    wl = configs.custom_workload("t70_d256_i128", T=70, d=256, I=128)
    shp, lay, x, dl = _setup(wl)
    for bm in (16, 64):
        opts = moe.options(tile_rows=bm)
        rt, ws, y = run_forward(shp, dl, to_dev(x), opts=opts)
        ref = oracle.route(x, lay.w_router, tile_rows=bm)
        assert_routing_equal(routing_to_host(rt, shp.T), ref)


def test_zero_tokens_is_noop():
    shp = moe.shape(0, 512, I=128)
    rt = moe.Routing(0)
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    x = torch.zeros(1, 512, dtype=torch.int16, device="cuda")
    moe.moe_route(shp, x, x, None, rt, ws)          # returns before touching anything


def test_repeat_calls_same_workspace_are_stable():
    wl = configs.custom_workload("t96_d512_i128", T=96, d=512, I=128)
    shp, lay, x, dl = _setup(wl)
    rt = moe.Routing(shp.T)
    ws = moe.workspace(shp)
    xd = to_dev(x)
    outs = []
    for _ in range(3):
        y = torch.empty(shp.T, shp.d, dtype=torch.int16, device="cuda")
        moe.moe_forward(shp, xd, dl.w_router, None, dl.packed_routed, dl.packed_shared, rt, ws, y)
        outs.append(y_to_f64(y))
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK
    ref = oracle.route(x, lay.w_router)
    out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
    for o in outs:
        assert_output_close(o, out_ref, "repeat")


def test_bad_expert_index_sets_status_not_fault():
    """Corrupt routing (an expert id out of range) fed to the FFN: the kernels flag it in the
    status word and skip the access."""
    wl = configs.custom_workload("t1_d512_i128b", T=1, d=512, I=128)
    shp, lay, x, dl = _setup(wl)
    rt = moe.Routing(1)
    ws = moe.workspace(shp)
    xd = to_dev(x)
    moe.moe_route(shp, xd, dl.w_router, None, rt, ws)
    rt.topk_idx[0, 3] = 999
    moe.moe_grouped_ffn(shp, xd, rt, dl.packed_routed, dl.packed_shared, ws)
    rc, bits = moe.moe_read_status(ws)
    assert rc == moe.MOE_ERR_DEVICE_STATUS and bits & moe.MOE_STATUS_BAD_EXPERT
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK      # cleared


def _routing_case(wl, w_router, bias=None):
    sh = wl.shape
    lay = configs.make_layer(wl)
    x = configs.make_x(wl)
    shp = moe.shape(sh.T, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    xd = to_dev(x)
    rt = moe.Routing(sh.T)
    ws = moe.workspace(shp)
    moe.moe_route(shp, xd, to_dev(w_router), None if bias is None else to_dev(bias), rt, ws)
    assert moe.moe_read_status(ws)[0] == moe.MOE_OK
    ref = oracle.route(x, w_router, bias)
    assert_routing_equal(routing_to_host(rt, sh.T), ref)
    return ref


def test_router_all_logits_equal_takes_full_recompute():
    """Every router row identical: all 256 logits tie, more than 32 candidates, so the exact
    logits of all experts are recomputed; ties go to the lower index."""
    wl = configs.custom_workload("tie_t70_d512", T=70, d=512, I=128)
    wr = configs.make_layer(wl).w_router.copy()
    wr[:] = wr[3]
    ref = _routing_case(wl, wr)
    assert (ref["topk_idx"] == np.arange(8)).all()


def test_router_duplicate_rows_exact_ties_at_the_boundary():
    """Pairs of identical router rows give exact ties, some at the 8th/9th place."""
    wl = configs.custom_workload("dup_t300_d1024", T=300, d=1024, I=128)
    wr = configs.make_layer(wl).w_router.copy()
    for a, b in [(1, 200), (17, 18), (40, 255), (100, 101), (7, 250)]:
        wr[b] = wr[a]
    _routing_case(wl, wr)


def test_router_skew_bias_many_tokens_same_experts():
    """The skewed workload's logit bias (a few experts take most rows)."""
    wl = configs.WORKLOADS["skew_t16384_d2048"]
    lay = configs.make_layer(wl)
    sub = configs.custom_workload("skew_sub", T=1000, d=2048, I=512, seed=wl.seed)
    ref = _routing_case(sub, lay.w_router, lay.logit_bias)
    assert ref["counts"].max() > 300


@pytest.mark.parametrize("T", [96, 1])
def test_large_scales_use_the_exact_fallback_encoding(T):
    """A stack with a scale >= 2^-5 cannot store scale * 2^133 in bf16; the packed buffer then
    keeps scales as they are (header word 1) and the kernels dequantise through 128 + q."""
    wl = configs.custom_workload(f"bigscale_t{T}", T=T, d=512, I=128)
    sh = wl.shape
    lay = configs.make_layer(wl)
    big = np.uint16(0x3D80)                      # 0.0625 >= 2^-5
    lay.routed.gate.scales[3, 5, 1] = big
    lay.shared.down.scales[0, 7, 0] = big
    x = configs.make_x(wl)
    shp = moe.shape(T, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    dl = DeviceLayer(shp, lay)
    assert int(dl.packed_routed[:4].view(torch.int32).item()) == 1
    assert int(dl.packed_shared[:4].view(torch.int32).item()) == 1
    rt, ws, y = run_forward(shp, dl, to_dev(x))
    ref = oracle.route(x, lay.w_router)
    out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
    assert_output_close(y_to_f64(y)[:T], out_ref, "fallback encoding")


def test_default_scales_use_the_denormal_encoding():
    wl = configs.custom_workload("smallscale", T=8, d=256, I=128)
    sh = wl.shape
    shp = moe.shape(8, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    dl = DeviceLayer(shp, configs.make_layer(wl))
    assert int(dl.packed_routed[:4].view(torch.int32).item()) == 0


def test_output_paths_and_deterministic_mode():
    """A 1024-token chunk: by default the down projection adds its weighted rows into the fp32
    sum; deterministic = 1 stores the rows (9 x 1024 x 2048 fp32 = 75 MB) and sums them in a
    fixed order.  Both match the oracle (sampled tokens), and the deterministic mode gives
    identical bits on a repeated call."""
    wl = configs.custom_workload("t1024_d2048_i512", T=1024, d=2048, I=512, seed=11)
    shp, lay, x, dl = _setup(wl)
    xd = to_dev(x)
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    toks = np.unique(np.concatenate([[0, shp.T - 1], np.random.default_rng(3).choice(shp.T, 14, replace=False)]))
    toks = toks.astype(np.int32)
    out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared, toks)
    ys = {}
    for det in (0, 1, 1):
        opts = moe.options(deterministic=det)
        rt, ws, y = run_forward(shp, dl, xd, opts=opts)
        assert_routing_equal(routing_to_host(rt, shp.T), ref)
        assert_output_close(y_to_f64(y)[toks], out_ref, f"deterministic={det}")
        ys.setdefault(det, []).append(y.clone())
    assert torch.equal(ys[1][0], ys[1][1]), "deterministic mode: repeated calls differ"


HOST_ROUTING = [
    configs.custom_workload("skew_t333_d512_i128", T=333, d=512, I=128, seed=21, zipf_s=1.2),
    configs.WORKLOADS["prefill_t512_d2048"],
]


@pytest.mark.parametrize("wl", HOST_ROUTING, ids=lambda w: w.name)
def test_host_routing_ablation_matches_device_routing(wl):
    """moe_options.host_routing = 1 (counts copied to the host, scan / block map / GEMM tile
    lists computed there and copied back) reproduces the GPU-resident routing exactly: the
    same routing outputs as the oracle and the same output bits (deterministic mode)."""
    shp, lay, x, dl = _setup(wl)
    xd = to_dev(x)
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    got = {}
    for hr in (0, 1):
        rt, ws, y = run_forward(shp, dl, xd, opts=moe.options(host_routing=hr, deterministic=1))
        r = routing_to_host(rt, shp.T)
        assert_routing_equal(r, ref)
        got[hr] = (r, y.clone())
    for key in ("topk_idx", "topk_w", "counts", "offsets", "perm", "pos", "tiles"):
        assert np.array_equal(got[0][0][key], got[1][0][key]), key
    assert torch.equal(got[0][1], got[1][1]), "host-routing output bits differ from the device path"


UNFUSED = [
    configs.WORKLOADS["tiny_t128_d512"],
    configs.custom_workload("skew_t333_d512_i128", T=333, d=512, I=128, seed=21, zipf_s=1.2),
    configs.WORKLOADS["prefill_t512_d2048"],
]


@pytest.mark.parametrize("wl", UNFUSED, ids=lambda w: w.name)
def test_unfused_dequant_ablation_matches_fused(wl):
    """moe_options.unfused_dequant = 1 (every weight of a projection dequantised to bf16 in the
    workspace by a separate kernel, then streamed by the GEMM) uses the same exact
    dequantisation, so in deterministic mode the output bits equal the fused path's; both
    match the oracle."""
    shp, lay, x, dl = _setup(wl)
    xd = to_dev(x)
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    toks = np.unique(np.concatenate([[0, shp.T - 1], np.random.default_rng(5).choice(shp.T, 10, replace=False)]))
    toks = toks.astype(np.int32)
    out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared, toks)
    ys = {}
    for uf in (0, 1):
        opts = moe.options(unfused_dequant=uf, deterministic=1)
        rt, ws, y = run_forward(shp, dl, xd, opts=opts)
        assert_routing_equal(routing_to_host(rt, shp.T), ref)
        assert_output_close(y_to_f64(y)[toks], out_ref, f"unfused_dequant={uf}")
        ys[uf] = y.clone()
    assert torch.equal(ys[0], ys[1]), "unfused-dequant output bits differ from the fused path"


def _adversarial_router(T, d, seed):
    """bf16 rows whose products span fp32's range: exponents from -75 to +40 (subnormal
    products and subnormal bf16 inputs included), random signs, some exact zeros."""
    rng = np.random.default_rng(seed)
    def rows(n):
        m = rng.uniform(1.0, 2.0, (n, d)) * rng.choice([-1.0, 1.0], (n, d))
        e = rng.integers(-75, 41, (n, d)).astype(np.float64)
        v = m * np.exp2(e)
        v[rng.random((n, d)) < 0.02] = 0.0
        sub = rng.random((n, d)) < 0.01                      # bf16 subnormals (below 2^-126)
        v[sub] = rng.uniform(-1, 1, sub.sum()) * 2.0 ** -127
        return gen.f32_to_bf16_bits(v.astype(np.float32))
    return rows(T), rows(256)


ROUTER_LOGIT_CASES = [
    ("tiny_t128_d512", None),
    ("prefill_t512_d2048", 64),
    ("d768", None),
    ("adversarial_d2048", None),
    ("adversarial_d768", None),
]


@pytest.mark.parametrize("case,rows", ROUTER_LOGIT_CASES, ids=[c[0] for c in ROUTER_LOGIT_CASES])
def test_router_logits_bit_exact(case, rows):
    """moe_router_logits (the device code of the exact recomputation) equals the oracle's fixed
    fp32 order bit for bit, with and without a logit bias, for ordinary router inputs and for
    rows whose products cover subnormal to large magnitudes; d = 768 takes the generic loop."""
    if case.startswith("adversarial"):
        d = int(case.split("_d")[1])
        x, wr = _adversarial_router(96, d, seed=d)
    elif case == "d768":
        wl = configs.custom_workload("t40_d768_i128", T=40, d=768, I=128, seed=17)
        lay = configs.make_layer(wl)
        x, wr = configs.make_x(wl), lay.w_router
    else:
        wl = configs.WORKLOADS[case]
        lay = configs.make_layer(wl)
        x, wr = configs.make_x(wl), lay.w_router
    if rows is not None:
        x = x[:rows]
    T, d = x.shape
    shp = moe.shape(T, d, 256, 8, 128, 128)
    bias = np.random.default_rng(T + d).normal(0.0, 0.5, 256).astype(np.float32)
    for b in (None, bias):
        out = torch.empty(T, 256, dtype=torch.float32, device="cuda")
        moe.moe_router_logits(shp, to_dev(x), to_dev(wr), None if b is None else to_dev(b), out)
        got = out.cpu().numpy()
        ref = oracle.router_logits(x, wr, b)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
            f"{case} bias={b is not None}: {(got.view(np.uint32) != ref.view(np.uint32)).sum()} logits differ"


MAX_SHAPES = [
    configs.custom_workload("max_t65536_d256_i128", T=65536, d=256, I=128, seed=31),
    configs.custom_workload("max_t64_d7168_i128", T=64, d=7168, I=128, seed=32),
    configs.custom_workload("max_t64_d256_i8192", T=64, d=256, I=8192, seed=33),
]


@pytest.mark.parametrize("wl", MAX_SHAPES, ids=lambda w: w.name)
def test_maximum_sizes(wl):
    """Each largest supported dimension (T = 65536, d = 7168, I = 8192) with the others small:
    routing bit-exact, sampled outputs within tolerance, deterministic mode included for the
    row path."""
    shp, lay, x, dl = _setup(wl)
    xd = to_dev(x)
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    T = shp.T
    toks = np.unique(np.concatenate([[0, T - 1], np.random.default_rng(7).choice(T, 14, replace=False)]))
    toks = toks.astype(np.int32)
    out_ref = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared, toks)
    for det in (0, 1):
        rt, ws, y = run_forward(shp, dl, xd, opts=moe.options(deterministic=det))
        assert_routing_equal(routing_to_host(rt, T), ref)
        assert_output_close(y_to_f64(y)[toks], out_ref, f"{wl.name} deterministic={det}")
        del rt, ws, y
        torch.cuda.empty_cache()
