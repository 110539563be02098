"""Helpers for the GPU tests: upload seeded workloads, run the CUDA path, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import quantized_grouped_gemm_gb300 as moe
from moe_workload import configs, gen

# tolerances of the MoE layer output against the oracle's fp64 result
ELEM_RTOL = 2e-2
ELEM_ATOL_SCALE = 1e-2      # max |err| <= 2e-2 * (|ref| + 1e-2)
FROB_RTOL = 5e-3
TOPK_W_ATOL = 1e-5


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def upload_q4(m: configs.Q4, device="cuda"):
    return (to_dev(m.codes, device), to_dev(m.scales, device), to_dev(m.biases, device))


class DeviceLayer:
    """One MoE layer on the device: router weight, optional logit bias, packed weights."""

    def __init__(self, shp, layer: configs.LayerInputs, device="cuda"):
        self.shp = shp
        self.w_router = to_dev(layer.w_router, device)
        self.bias = None if layer.logit_bias is None else to_dev(layer.logit_bias, device)
        r, s = layer.routed, layer.shared
        self.packed_routed = moe.moe_pack_weights(shp, upload_q4(r.gate), upload_q4(r.up), upload_q4(r.down), shp.I)
        self.packed_shared = moe.moe_pack_weights(shp, upload_q4(s.gate), upload_q4(s.up), upload_q4(s.down),
                                                  shp.I_shared)
        torch.cuda.synchronize()


def run_forward(shp, dl: DeviceLayer, x_dev: torch.Tensor, opts=None, split_calls=False):
    rt = moe.Routing(shp.T, shp.k, shp.E, (opts.tile_rows if opts is not None and opts.tile_rows else 32))
    ws = moe.workspace(shp, opts)
    y = torch.empty(max(shp.T, 1), shp.d, dtype=torch.int16, device=x_dev.device)
    if split_calls:
        moe.moe_route(shp, x_dev, dl.w_router, dl.bias, rt, ws, opts)
        moe.moe_grouped_ffn(shp, x_dev, rt, dl.packed_routed, dl.packed_shared, ws, opts)
        moe.moe_combine(shp, rt, ws, y, opts)
    else:
        moe.moe_forward(shp, x_dev, dl.w_router, dl.bias, dl.packed_routed, dl.packed_shared, rt, ws, y, opts)
    rc, bits = moe.moe_read_status(ws)
    assert rc == moe.MOE_OK, (rc, bits)
    return rt, ws, y


def routing_to_host(rt: moe.Routing, T: int):
    nt = int(rt.num_tiles.item())
    return dict(topk_idx=rt.topk_idx[:T].cpu().numpy(), topk_w=rt.topk_w[:T].cpu().numpy(),
                counts=rt.counts.cpu().numpy(), offsets=rt.offsets.cpu().numpy(),
                perm=rt.perm[:8 * T].cpu().numpy(), pos=rt.pos[:T].cpu().numpy(),
                tiles=rt.tiles[:nt].cpu().numpy(), num_tiles=nt)


def assert_routing_equal(got: dict, ref: dict):
    assert np.array_equal(got["topk_idx"], ref["topk_idx"]), "top-k experts differ"
    dw = np.abs(got["topk_w"].astype(np.float64) - ref["topk_w"])
    assert dw.max() <= TOPK_W_ATOL, f"routing weights differ by {dw.max()}"
    assert np.abs(got["topk_w"].astype(np.float64).sum(1) - 1).max() <= 1e-5
    for key in ("counts", "offsets", "perm", "pos"):
        assert np.array_equal(got[key], ref[key]), f"{key} differs"
    assert got["num_tiles"] == ref["num_tiles"]
    assert np.array_equal(got["tiles"], ref["tiles"]), "block map differs"


def y_to_f64(y: torch.Tensor) -> np.ndarray:
    return gen.bf16_bits_to_f32(y.cpu().numpy().view(np.uint16)).astype(np.float64)


def assert_output_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(got - ref)
    bound = ELEM_RTOL * (np.abs(ref) + ELEM_ATOL_SCALE)
    bad = err > bound
    frob = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; worst err "
                           f"{err.max():.3e}; frob {frob:.3e}")
    assert frob <= FROB_RTOL, f"{what}: relative Frobenius error {frob:.3e}"
    return frob
