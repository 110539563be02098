"""GPU parity at the benchmark sizes, through the C ABI, against the CPU oracle.

* The 512-token chunk (d=2048, I=512): every token's output.
* The 4096-token chunk: one token from every 32-row block of every expert group (and of the
  shared expert's rows), plus every row of the largest group, so every GEMM tile of both
  projections contributes checked rows.
* The skewed long prefill as the pages run it (section "Limit temporary memory with prompt
  chunking"): four 4096-token chunks back to back on one stream, reusing one workspace and
  one set of routing buffers, with no host synchronisation between chunks; each chunk's
  routing (bit for bit) and sampled outputs are then checked.
* moe_options.gemm_rows (largest token block of the grouped GEMMs, "Match tile size to
  expert load"): every value against the oracle on a skewed chunk, all tokens compared.

Routing must match bit for bit; outputs within max |err| <= 2e-2 (|ref| + 1e-2) elementwise
and relative Frobenius error <= 5e-3 against the oracle's fp64 result.
"""
import numpy as np
import pytest
import torch

import oracle
import quantized_grouped_gemm_gb300 as moe
from moe_workload import configs
from gpu_helpers import (DeviceLayer, assert_output_close, assert_routing_equal, routing_to_host, run_forward,
                         to_dev, y_to_f64)

pytestmark = pytest.mark.gpu


def _layer(wl, T):
    sh = wl.shape
    lay = configs.make_layer(wl)
    shp = moe.shape(T, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    return shp, lay, DeviceLayer(shp, lay)


def block_sample_tokens(ref, T, k=8, block=32, seed=0):
    """One token from every `block`-row piece of every expert group and of the shared expert's
    token rows, plus every token of the largest group (sorted, unique)."""
    rng = np.random.default_rng(seed)
    off, perm = ref["offsets"], ref["perm"]
    toks = []
    for e in range(len(off) - 1):
        for r0 in range(off[e], off[e + 1], block):
            r = r0 + rng.integers(0, min(block, off[e + 1] - r0))
            toks.append(perm[r] // k)
    for t0 in range(0, T, block):
        toks.append(t0 + rng.integers(0, min(block, T - t0)))
    big = int(np.argmax(np.diff(off)))
    toks.extend((perm[off[big]:off[big + 1]] // k).tolist())
    return np.unique(np.asarray(toks, dtype=np.int32))


def test_prefill_t512_every_token():
    wl = configs.WORKLOADS["prefill_t512_d2048"]
    x = configs.make_x(wl)
    shp, lay, dl = _layer(wl, x.shape[0])
    rt, ws, y = run_forward(shp, dl, to_dev(x))
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    assert_routing_equal(routing_to_host(rt, shp.T), ref)
    out = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
    assert_output_close(y_to_f64(y), out, "prefill_t512_d2048, all 512 tokens")


def test_prefill_t4096_every_gemm_block_sampled():
    wl = configs.WORKLOADS["prefill_t4096_d2048"]
    x = configs.make_x(wl)
    T = x.shape[0]
    shp, lay, dl = _layer(wl, T)
    rt, ws, y = run_forward(shp, dl, to_dev(x))
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    assert_routing_equal(routing_to_host(rt, T), ref)
    toks = block_sample_tokens(ref, T, seed=1)
    assert len(toks) > 700
    out = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared, toks)
    assert_output_close(y_to_f64(y)[toks], out, f"prefill_t4096_d2048, {len(toks)} tokens")


def test_skew_four_chunks_back_to_back_one_workspace():
    wl = configs.WORKLOADS["skew_t16384_d2048"]
    x_all = configs.make_x(wl)
    T = wl.chunk
    nch = wl.shape.T // T
    assert nch == 4
    shp, lay, dl = _layer(wl, T)
    xs = [to_dev(np.ascontiguousarray(x_all[c * T:(c + 1) * T])) for c in range(nch)]
    rt = moe.Routing(T)
    ws = moe.workspace(shp)
    y = torch.empty(T, shp.d, dtype=torch.int16, device="cuda")
    keep = []
    torch.cuda.synchronize()
    for c in range(nch):        # one stream, one workspace, one set of routing buffers, no host sync
        moe.moe_forward(shp, xs[c], dl.w_router, dl.bias, dl.packed_routed, dl.packed_shared, rt, ws, y)
        keep.append(dict(topk_idx=rt.topk_idx.clone(), topk_w=rt.topk_w.clone(), counts=rt.counts.clone(),
                         offsets=rt.offsets.clone(), perm=rt.perm.clone(), pos=rt.pos.clone(),
                         tiles=rt.tiles.clone(), num_tiles=rt.num_tiles.clone(), y=y.clone()))
    rc, bits = moe.moe_read_status(ws)
    assert rc == moe.MOE_OK, (rc, bits)
    for c in range(nch):
        x = np.ascontiguousarray(x_all[c * T:(c + 1) * T])
        ref = oracle.route(x, lay.w_router, lay.logit_bias)
        kc = keep[c]
        nt = int(kc["num_tiles"].item())
        got = dict(topk_idx=kc["topk_idx"].cpu().numpy(), topk_w=kc["topk_w"].cpu().numpy(),
                   counts=kc["counts"].cpu().numpy(), offsets=kc["offsets"].cpu().numpy(),
                   perm=kc["perm"].cpu().numpy(), pos=kc["pos"].cpu().numpy(),
                   tiles=kc["tiles"][:nt].cpu().numpy(), num_tiles=nt)
        assert_routing_equal(got, ref)
        assert np.diff(ref["offsets"]).max() > 1000          # the skew: a few experts take most rows
        # the smallest and the largest groups, and a spread of other tokens
        rng = np.random.default_rng(100 + c)
        cnt = np.diff(ref["offsets"])
        small = [e for e in np.argsort(cnt) if cnt[e] > 0][:8]
        toks = [ref["perm"][ref["offsets"][e]] // 8 for e in small]
        big = int(np.argmax(cnt))
        toks += list(ref["perm"][ref["offsets"][big]:ref["offsets"][big + 1]][::97] // 8)
        toks += list(rng.choice(T, 24, replace=False)) + [0, T - 1]
        toks = np.unique(np.asarray(toks, dtype=np.int32))
        out = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared, toks)
        assert_output_close(y_to_f64(kc["y"])[toks], out, f"skew chunk {c} ({len(toks)} tokens)")


GEMM_ROWS_WL = configs.custom_workload("skew_t1500_d512_i128", T=1500, d=512, I=128, seed=41, zipf_s=1.2)


@pytest.mark.parametrize("rows", [16, 32, 64, 128])
def test_gemm_rows_option_parity(rows):
    """Each token-block size of the grouped GEMMs on a skewed chunk (groups from 0 to ~1500
    rows): routing bit for bit, every token's output within tolerance, in both output modes."""
    wl = GEMM_ROWS_WL
    x = configs.make_x(wl)
    shp, lay, dl = _layer(wl, x.shape[0])
    ref = oracle.route(x, lay.w_router, lay.logit_bias)
    out = oracle.moe_tokens(x, ref["topk_idx"], ref["topk_w"], lay.routed, lay.shared)
    for det in (0, 1):
        rt, ws, y = run_forward(shp, dl, to_dev(x), opts=moe.options(gemm_rows=rows, deterministic=det))
        assert_routing_equal(routing_to_host(rt, shp.T), ref)
        assert_output_close(y_to_f64(y), out, f"gemm_rows={rows} deterministic={det}")
